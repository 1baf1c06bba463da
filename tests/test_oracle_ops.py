"""Pins of the oracle's per-op functions against what the pages and the
mathematics fix: printed worked examples (tests/golden), closed forms,
invariants, library routines on special cases and brute force.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------- contract
def test_residual_dims_check_matches_page_examples():
    g = gold("p1_status_contract.json")
    for case in g["residual_dims_check"]:
        assert O.residual_dims_check(*case["args"]) == case["status"]
    assert O.residual_dims_check(0, 0, 0) == 561
    assert O.residual_dims_check(g["max_dim"] + 1, g["max_dim"] + 1, g["max_dim"] + 1) == 564
    assert O.residual_dims_check(6, 6, 5) == 563


# ----------------------------------------------------------------- bf16
def test_bf16_rounding_matches_torch_including_ties():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(2000).astype(np.float32) * 10
    # exact halfway cases: low 16 bits == 0x8000, both parities of bit 16
    upper = rng.integers(0x0080, 0x7f00, 200).astype(np.uint32)  # finite, normal
    halves = ((upper << 16) | 0x8000).view(np.float32)
    x = np.concatenate([x, halves, -halves,
                        np.array([0.0, -0.0, 1.0, np.inf, -np.inf], np.float32)])
    ours = O.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # NaN stays NaN (payload bits are not meaningful)
    nan_bits = O.f32_to_bf16_bits(np.array([np.nan], np.float32))[0]
    assert (nan_bits & 0x7f80) == 0x7f80 and (nan_bits & 0x007f) != 0
    # widening is exact
    assert np.array_equal(O.bf16_bits_to_f64(ref),
                          torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy())


# ----------------------------------------------------------------- GEMV
def test_gemv_transposed_worked_example():
    g = gold("p1_gemv_worked_example.json")
    y = O.gemv_transposed(g["A"], g["x"], g["rows"], g["cols"])
    assert y.tolist() == g["y"]


@pytest.mark.parametrize("rows,cols", [(300, 300), (128, 1536), (7, 33)])
def test_gemv_transposed_against_numpy(rows, cols):
    # the page checks 300x300 and 128x1536 against the scalar kernel to 1e-9
    rng = np.random.default_rng(rows * 7 + cols)
    A = rng.standard_normal((rows, cols)).astype(np.float32)
    x = rng.standard_normal(rows)
    y = O.gemv_transposed(A.ravel(), x, rows, cols)
    np.testing.assert_allclose(y, A.astype(np.float64).T @ x, rtol=0, atol=1e-9)
    # the untransposed product differs, so a swapped operand would fail
    if rows == cols:
        assert np.abs(y - A.astype(np.float64) @ x).max() > 1e-3


def test_gemv_transposed_bf16_widens_exactly():
    rng = np.random.default_rng(3)
    A = torch.from_numpy(rng.standard_normal((64, 96)).astype(np.float32)).to(torch.bfloat16)
    x = rng.standard_normal(64)
    bits = A.view(torch.int16).numpy().view(np.uint16).ravel()
    y = O.gemv_transposed(bits, x, 64, 96, O.DT_BF16)
    np.testing.assert_allclose(y, A.double().numpy().T @ x, rtol=0, atol=1e-10)


def test_gemv_untransposed_against_numpy():
    rng = np.random.default_rng(4)
    W = rng.standard_normal((40, 16)).astype(np.float32)
    x = rng.standard_normal(16)
    np.testing.assert_allclose(O.gemv(W.ravel(), x, 40, 16), W.astype(np.float64) @ x, atol=1e-12)


# ----------------------------------------------------------------- residual
def test_residual_add_examples():
    g = gold("p1_residual_add.json")
    assert O.residual_add(g["a"], g["b"]).tolist() == g["out"]
    rng = np.random.default_rng(5)
    a = rng.standard_normal(g["large_n"]).astype(np.float32)
    b = rng.standard_normal(g["large_n"]).astype(np.float32)
    assert np.abs(O.residual_add(a, b) - (a + b)).max() == g["large_max_delta"]


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_form_constant_vector():
    # x = c everywhere: mean(x^2) = c^2, so y = c / sqrt(c^2 + eps) * g
    c, n, eps = 3.0, 16, 1e-5
    g = np.linspace(0.5, 1.5, n).astype(np.float32)
    y = O.rmsnorm(np.full(n, c), g, eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps) * g.astype(np.float64), rtol=1e-14)


def test_rmsnorm_matches_torch_expression():
    rng = np.random.default_rng(6)
    x = rng.standard_normal(4096)
    w = (1 + 0.1 * rng.standard_normal(4096)).astype(np.float32)
    t = torch.from_numpy(x)
    ref = (t * torch.rsqrt(t.pow(2).mean() + 1e-5) * torch.from_numpy(w).double()).numpy()
    np.testing.assert_allclose(O.rmsnorm(x, w), ref, rtol=1e-12)


def test_add_rmsnorm_updates_residual_then_normalises():
    rng = np.random.default_rng(7)
    r = rng.standard_normal(4096).astype(np.float32)
    x = rng.standard_normal(4096).astype(np.float32)
    w = (1 + 0.1 * rng.standard_normal(4096)).astype(np.float32)
    r2, h = O.add_rmsnorm(r, x, w)
    assert np.array_equal(r2, r + x)
    np.testing.assert_allclose(h, O.rmsnorm(r2.astype(np.float64), w), rtol=1e-15)
    r3, h3 = O.add_rmsnorm(r, None, w)
    assert np.array_equal(r3, r)


# ----------------------------------------------------------------- SiLU
def test_silu_mul_matches_torch_and_fixed_points():
    rng = np.random.default_rng(8)
    g = rng.standard_normal(1000) * 4
    u = rng.standard_normal(1000)
    ref = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    np.testing.assert_allclose(O.silu_mul(g, u), ref, rtol=1e-13, atol=1e-15)
    assert O.silu_mul([0.0], [5.0])[0] == 0.0
    assert O.silu_mul([1.0], [1.0])[0] == pytest.approx(1 / (1 + math.exp(-1)), rel=1e-15)


def test_exp_of_zero_is_exactly_one():
    # "decode-ops", "API - Method": exp(0) == 1 exactly; the oracle's
    # softmax relies on it for the maximum's weight
    assert math.exp(0.0) == 1.0
    out = O.gqa_attention(np.zeros(2), np.array([0, 0, 0, 0], np.float32),
                          np.array([7, 7, 3, 3], np.float32), O.DT_F32, 2, 1, 1, 2)
    assert out.tolist() == [5.0, 5.0]  # equal scores -> exact mean


# ----------------------------------------------------------------- RoPE
@pytest.mark.parametrize("layout", [O.ROPE_HALF_SPLIT, O.ROPE_INTERLEAVED])
def test_rope_position_zero_is_identity(layout):
    v = np.random.default_rng(9).standard_normal(8 * 128)
    assert np.array_equal(O.rope(v, 8, 128, 0, 1e4, layout), v)


def test_rope_head_dim_two_turns_by_pos_radians():
    # one pair per head, frequency base^0 = 1, so the angle is pos itself
    for pos in (1, 5, 123):
        out = O.rope([1.0, 0.0, 0.0, 2.0], 2, 2, pos, 1e4, O.ROPE_INTERLEAVED)
        c, s = math.cos(pos), math.sin(pos)
        np.testing.assert_allclose(out, [c, s, -2 * s, 2 * c], atol=1e-15)


def test_rope_pair_frequency_and_layouts():
    hd, pos, base = 8, 7, 10000.0
    for p in range(hd // 2):
        theta = pos * base ** (-2.0 * p / hd)
        # interleaved: pair (2p, 2p+1)
        e = np.zeros(hd)
        e[2 * p] = 1.0
        out = O.rope(e, 1, hd, pos, base, O.ROPE_INTERLEAVED)
        assert out[2 * p] == pytest.approx(math.cos(theta), abs=1e-15)
        assert out[2 * p + 1] == pytest.approx(math.sin(theta), abs=1e-15)
        # half-split: pair (p, p + hd/2)
        e = np.zeros(hd)
        e[p] = 1.0
        out = O.rope(e, 1, hd, pos, base, O.ROPE_HALF_SPLIT)
        assert out[p] == pytest.approx(math.cos(theta), abs=1e-15)
        assert out[p + hd // 2] == pytest.approx(math.sin(theta), abs=1e-15)


def test_rope_preserves_pair_norms_and_is_relative():
    rng = np.random.default_rng(10)
    hd = 128
    q = rng.standard_normal(hd)
    k = rng.standard_normal(hd)
    for layout in (O.ROPE_HALF_SPLIT, O.ROPE_INTERLEAVED):
        r = O.rope(q, 1, hd, 4321, 1e4, layout)
        assert np.linalg.norm(r) == pytest.approx(np.linalg.norm(q), rel=1e-13)
        # <R(m) q, R(n) k> depends only on m - n
        d1 = O.rope(q, 1, hd, 100, 1e4, layout) @ O.rope(k, 1, hd, 37, 1e4, layout)
        d2 = O.rope(q, 1, hd, 63, 1e4, layout) @ O.rope(k, 1, hd, 0, 1e4, layout)
        assert d1 == pytest.approx(d2, rel=1e-10)


def test_rope_half_split_is_interleaved_under_permutation():
    rng = np.random.default_rng(11)
    hd = 16
    v = rng.standard_normal(hd)
    perm = np.empty(hd, dtype=int)  # interleaved slot 2p <- p, 2p+1 <- p+hd/2
    perm[0::2] = np.arange(hd // 2)
    perm[1::2] = np.arange(hd // 2) + hd // 2
    a = O.rope(v, 1, hd, 99, 500000.0, O.ROPE_HALF_SPLIT)
    b = O.rope(v[perm], 1, hd, 99, 500000.0, O.ROPE_INTERLEAVED)
    np.testing.assert_allclose(a[perm], b, atol=1e-15)


# Long-context RoPE scaling as Llama 3.1 checkpoints define it (not on the
# pages): pinned by reductions, band limits, continuity and invariants.
LLAMA31_SCALING = {"factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
                   "original_max_position": 8192.0}


def test_rope_scaling_with_factor_one_is_the_unscaled_rope():
    sc = dict(LLAMA31_SCALING, factor=1.0)
    for p in range(64):
        f = 500000.0 ** (-2.0 * p / 128)
        assert O.rope_freq(p, 128, 500000.0, sc) == pytest.approx(f, rel=1e-15)
    v = np.random.default_rng(12).standard_normal(128)
    np.testing.assert_allclose(O.rope(v, 1, 128, 777, 500000.0, O.ROPE_HALF_SPLIT, sc),
                               O.rope(v, 1, 128, 777, 500000.0, O.ROPE_HALF_SPLIT), atol=1e-12)


def test_rope_scaling_bands_on_the_llama31_parameters():
    """Wavelength 2 pi / f below 8192 / 4 keeps f; above 8192 / 1 divides it
    by 8; in between it lies strictly inside, and the ratio to the unscaled
    frequency never rises as the pairs slow down."""
    hd, base = 128, 500000.0
    ratios = []
    n_keep = n_slow = n_mid = 0
    for p in range(hd // 2):
        f = base ** (-2.0 * p / hd)
        g = O.rope_freq(p, hd, base, LLAMA31_SCALING)
        w = 2 * math.pi / f
        if w < 2048.0:
            assert g == f
            n_keep += 1
        elif w > 8192.0:
            assert g == pytest.approx(f / 8.0, rel=1e-15)
            n_slow += 1
        else:
            assert f / 8.0 < g < f
            n_mid += 1
        ratios.append(g / f)
    assert all(a >= b for a, b in zip(ratios, ratios[1:]))
    assert n_keep > 0 and n_slow > 0 and n_mid > 0
    assert O.rope_freq(0, hd, base, LLAMA31_SCALING) == 1.0  # the fastest pair turns one radian per position


@pytest.mark.parametrize("edge", ["high", "low"])
def test_rope_scaling_is_continuous_at_both_band_edges(edge):
    """Move original_max_position across the value that puts pair p's
    wavelength exactly on a band edge: the frequency must not jump (it meets
    f at the high-frequency edge and f / factor at the low-frequency edge)."""
    hd, base, p = 128, 500000.0, 40
    f = base ** (-2.0 * p / hd)
    w = 2 * math.pi / f
    sc = dict(LLAMA31_SCALING)
    at = w * (sc["high_freq_factor"] if edge == "high" else sc["low_freq_factor"])
    want = f if edge == "high" else f / sc["factor"]
    for eps in (-1e-9, 1e-9):
        sc["original_max_position"] = at * (1 + eps)
        assert O.rope_freq(p, hd, base, sc) == pytest.approx(want, rel=1e-7)


def test_scaled_rope_is_relative_and_identity_at_zero():
    rng = np.random.default_rng(13)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    sc = LLAMA31_SCALING
    assert np.array_equal(O.rope(q, 1, 128, 0, 500000.0, O.ROPE_HALF_SPLIT, sc), q)
    d1 = O.rope(q, 1, 128, 9000, 500000.0, O.ROPE_HALF_SPLIT, sc) @ O.rope(k, 1, 128, 8000, 500000.0,
                                                                           O.ROPE_HALF_SPLIT, sc)
    d2 = O.rope(q, 1, 128, 1000, 500000.0, O.ROPE_HALF_SPLIT, sc) @ O.rope(k, 1, 128, 0, 500000.0,
                                                                           O.ROPE_HALF_SPLIT, sc)
    assert d1 == pytest.approx(d2, rel=1e-9)
    # and the scaling matters at long range: the slow pairs turn 8 times less
    assert not np.allclose(O.rope(q, 1, 128, 9000, 500000.0, O.ROPE_HALF_SPLIT, sc),
                           O.rope(q, 1, 128, 9000, 500000.0, O.ROPE_HALF_SPLIT), atol=1e-3)


# ----------------------------------------------------------------- KV cache
def test_kv_cache_append_worked_example():
    g = gold("p1_kv_cache_append.json")
    cache = np.zeros(g["n"], dtype=np.float32)
    cache[:g["cache_len"]] = g["cache"]
    assert O.kv_cache_append(cache, O.DT_F32, g["cache_len"], g["new_vals"], g["n_new"]) == 560
    assert cache.tolist() == g["out"]


def test_kv_cache_append_refusals():
    cache = np.zeros(8, dtype=np.float32)
    assert O.kv_cache_append(cache, O.DT_F32, 6, [1.0, 2.0, 3.0], 3) == 571
    assert O.kv_cache_append(cache, O.DT_F32, 0, [], 0) == 561
    assert O.kv_cache_append(cache, O.DT_F32, 0, [1.0, 2.0], 3, new_len=2) == 567
    assert not cache.any()


def test_kv_cache_append_bf16_rounds_to_nearest_even():
    cache = np.zeros(4, dtype=np.uint16)
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5])
    assert O.kv_cache_append(cache, O.DT_BF16, 0, vals, 4) == 560
    assert cache.tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020]


# ----------------------------------------------------------------- attention
def test_attention_single_position_returns_v():
    rng = np.random.default_rng(12)
    q = rng.standard_normal(4 * 8)
    k = rng.standard_normal(2 * 8).astype(np.float32)
    v = rng.standard_normal(2 * 8).astype(np.float32)
    out = O.gqa_attention(q, k, v, O.DT_F32, 1, 4, 2, 8)
    np.testing.assert_array_equal(out.reshape(4, 8), v.reshape(2, 8)[[0, 0, 1, 1]])


def test_attention_identical_keys_average_values():
    rng = np.random.default_rng(13)
    T, hd = 9, 8
    q = rng.standard_normal(hd)
    k = np.tile(rng.standard_normal(hd), T).astype(np.float32)
    v = rng.standard_normal(T * hd).astype(np.float32)
    out = O.gqa_attention(q, k, v, O.DT_F32, T, 1, 1, hd)
    np.testing.assert_allclose(out, v.reshape(T, hd).astype(np.float64).mean(0), atol=1e-15)


def test_attention_group_mapping_is_integer_division():
    # 4 query heads share 2 KV heads: heads 0,1 -> kv 0 and heads 2,3 -> kv 1
    # (a modulo mapping would give 0,1,0,1)
    hd, T = 2, 3
    rng = np.random.default_rng(14)
    k = rng.standard_normal(T * 2 * hd).astype(np.float32)
    v = np.zeros((T, 2, hd), dtype=np.float32)
    v[:, 0, :] = 1.0
    v[:, 1, :] = 2.0
    out = O.gqa_attention(rng.standard_normal(4 * hd), k, v.ravel(), O.DT_F32, T, 4, 2, hd)
    np.testing.assert_allclose(out.reshape(4, hd)[:, 0], [1, 1, 2, 2], atol=1e-14)


def test_attention_matches_scipy_softmax_brute_force():
    rng = np.random.default_rng(15)
    nq, nkv, hd, T = 8, 2, 16, 37
    q = rng.standard_normal(nq * hd)
    K = rng.standard_normal((T, nkv, hd)).astype(np.float32)
    V = rng.standard_normal((T, nkv, hd)).astype(np.float32)
    out = O.gqa_attention(q, K.ravel(), V.ravel(), O.DT_F32, T, nq, nkv, hd).reshape(nq, hd)
    for h in range(nq):
        g = h // (nq // nkv)
        w = scipy.special.softmax(K[:, g, :].astype(np.float64) @ q[h * hd:(h + 1) * hd] / math.sqrt(hd))
        np.testing.assert_allclose(out[h], w @ V[:, g, :].astype(np.float64), atol=1e-13)


def test_attention_paged_equals_contiguous():
    rng = np.random.default_rng(16)
    nq, nkv, hd, bt, nblk = 4, 2, 8, 4, 6
    T = 21
    K = rng.standard_normal((nblk * bt, nkv * hd)).astype(np.float32)
    V = rng.standard_normal((nblk * bt, nkv * hd)).astype(np.float32)
    table = np.array([[4, 0, 5, 2, 1, 3]], dtype=np.int32)
    # gather the sequence's rows into contiguous order
    rows = np.concatenate([np.arange(b * bt, (b + 1) * bt) for b in table[0]])
    q = rng.standard_normal(nq * hd)
    paged = O.gqa_attention(q, K.ravel(), V.ravel(), O.DT_F32, T, nq, nkv, hd,
                            block_table=table, max_blocks=6, block_tokens=bt)
    contig = O.gqa_attention(q, K[rows].ravel(), V[rows].ravel(), O.DT_F32, T, nq, nkv, hd)
    np.testing.assert_array_equal(paged, contig)


# ----------------------------------------------------------------- argmax
def test_argmax_worked_examples():
    for case in gold("p1_greedy_argmax.json")["cases"]:
        i, m = O.argmax(case["logits"])
        assert (i, m) == (case["token_id"], case["logit"])


def test_argmax_matches_torch_with_ties_and_nan():
    rng = np.random.default_rng(17)
    for trial in range(20):
        l = np.round(rng.standard_normal(1000) * 3).astype(np.float32)  # many ties
        assert O.argmax(l)[0] == int(torch.argmax(torch.from_numpy(l)))
    l = rng.standard_normal(151936).astype(np.float32)
    l[12095] = 50.0
    assert O.argmax(l)[0] == 12095
    l = np.array([1.0, np.nan, 5.0, np.nan], dtype=np.float32)
    assert O.argmax(l)[0] == int(torch.argmax(torch.from_numpy(l))) == 1


# ----------------------------------------------------------------- sampler
def _hf_warper_probs(logits, T, k, p):
    """Token probabilities after temperature -> top-k -> top-p with torch's
    own sort/softmax/cumsum (descending order, ties by lower index)."""
    l = torch.from_numpy(np.asarray(logits, np.float32)).double() / T
    order = sorted(range(len(l)), key=lambda i: (-float(l[i]), i))
    keep = order[:k] if 0 < k < len(l) else order
    probs = torch.softmax(l[keep], 0)
    cum = torch.cumsum(probs, 0)
    n_keep = int((cum - probs < p).sum()) if p < 1 else len(keep)
    n_keep = max(n_keep, 1)
    kept = keep[:n_keep]
    pr = probs[:n_keep] / probs[:n_keep].sum()
    return kept, pr.numpy()


@pytest.mark.parametrize("T,k,p", [(0.8, 5, 0.95), (1.3, 0, 0.7), (0.5, 3, 1.0), (1.0, 12, 0.5)])
def test_sampler_frequencies_match_warper_probabilities(T, k, p):
    rng = np.random.default_rng(18)
    logits = rng.standard_normal(12).astype(np.float32) * 2
    kept, pr = _hf_warper_probs(logits, T, k, p)
    n = 20000
    counts = {}
    prev_rank = 0
    for j in range(n):
        u = (j + 0.5) / n
        tok, _ = O.sample(logits, T, k, p, u)
        counts[tok] = counts.get(tok, 0) + 1
        rank = kept.index(tok)
        assert rank >= prev_rank  # inverse CDF walks the survivors in order
        prev_rank = rank
    assert set(counts) <= set(kept)
    for tok, prob in zip(kept, pr):
        assert abs(counts.get(tok, 0) / n - prob) <= 2.0 / n


def test_sampler_special_cases():
    rng = np.random.default_rng(19)
    l = rng.standard_normal(500).astype(np.float32)
    top = O.argmax(l)[0]
    assert O.sample(l, 0.8, 1, 0.95, 0.99)[0] == top        # top_k = 1
    assert O.sample(l, 0.8, 50, 1e-6, 0.99)[0] == top       # tiny top_p
    assert O.sample(l, 0.8, 50, 0.95, 0.0)[0] == top        # u = 0
    assert O.sample(l, 0.0, 50, 0.95, 0.7)[0] == top        # T <= 0: greedy
    assert O.sample(l, 0.8, 50, 0.0, 0.5)[0] == -1          # top_p out of domain
    assert O.sample(l, 0.8, 50, 0.9, 1.0)[0] == -1          # u out of domain


def test_sampler_topk_ties_keep_lower_indices():
    l = np.array([1.0, 3.0, 3.0, 3.0, 0.0, 3.0], dtype=np.float32)
    # top-2 of four tied 3.0s keeps ids 1 and 2; with equal mass, u below 1/2
    # picks id 1 and above picks id 2
    assert O.sample(l, 1.0, 2, 1.0, 0.25)[0] == 1
    assert O.sample(l, 1.0, 2, 1.0, 0.75)[0] == 2


def test_sampler_flat_vocabulary_inverse_cdf_is_exact():
    """A flat distribution over the whole 128,256-entry vocabulary: every
    survivor has mass 1/n, so the draw (j + 1/2) / n must pick token j, and a
    top-p cut of 0.3 keeps exactly the first 38,477 ids (i/n < 0.3), over
    which the draw (j + 1/2) / 38477 picks token j.  Running sums carried in
    fp32 drift by far more than 1/(2n) over this many terms and fail here."""
    n = 128256
    l = np.full(n, 0.25, dtype=np.float32)
    for j in (0, 1, 777, 50000, 99999, 128000, n - 1):
        tok, margin = O.sample(l, 1.0, 0, 1.0, (j + 0.5) / n)
        assert tok == j and margin > 0.4 / n
    kept = 38477
    for j in (0, 12345, 30000, kept - 1):
        tok, _ = O.sample(l, 1.0, 0, 0.3, (j + 0.5) / kept)
        assert tok == j
    assert O.sample(l, 1.0, 0, 0.3, 0.999999)[0] == kept - 1
    # top-k over ties keeps the lowest ids: the 1000 survivors are ids 0..999
    assert O.sample(l, 1.0, 1000, 1.0, 0.9995)[0] == 999


@pytest.mark.parametrize("T,k,p", [(1.0, 0, 0.9), (0.7, 400, 0.95)])
def test_sampler_frequencies_over_a_wide_vocabulary(T, k, p):
    """The warper's probabilities over 1,000 logits, top-k off or wide: the
    draw grid's token frequencies match them to within one grid step."""
    rng = np.random.default_rng(21)
    logits = rng.standard_normal(1000).astype(np.float32)
    kept, pr = _hf_warper_probs(logits, T, k, p)
    n = 8000
    counts = {}
    for j in range(n):
        tok, _ = O.sample(logits, T, k, p, (j + 0.5) / n)
        counts[tok] = counts.get(tok, 0) + 1
    assert set(counts) <= set(kept)
    cum_want = np.cumsum(pr)
    cum_got = np.cumsum([counts.get(t, 0) for t in kept]) / n
    assert np.max(np.abs(cum_want - cum_got)) <= 1.0 / n + 1e-9


def test_sampler_fixed_draw_gives_fixed_token():
    rng = np.random.default_rng(20)
    l = rng.standard_normal(128256).astype(np.float32)
    a = O.sample(l, 0.8, 50, 0.95, 0.3141)
    b = O.sample(l, 0.8, 50, 0.95, 0.3141)
    assert a == b and a[0] >= 0
