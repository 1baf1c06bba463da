"""Per-op parity of the CUDA kernels (through the C ABI) against the oracle,
at the pages' op-level sizes and at small ragged sizes that span several
tiles."""
import numpy as np
import pytest
import torch

import oracle as O
from autoregressive_decode_step_gb300 import synth
from tests.gpu_util import FP32_TOL, host, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def A():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from autoregressive_decode_step_gb300 import abi
    return abi


def dev(t):
    return t.to("cuda")


# ----------------------------------------------------------------- GEMV
@pytest.mark.parametrize("rows,cols,dt", [
    (2, 3, torch.float32),          # the page's worked example (plain-load path)
    (300, 300, torch.float32), (128, 1536, torch.float32),  # the page's parity shapes
    (777, 1000, torch.float32),     # ragged last band, uneven split
    (1, 8, torch.float32), (5, 4, torch.float32),
    (4096, 4096, torch.float32), (4096, 14336, torch.float32),  # op-level sizes
    (4096, 6144, torch.bfloat16), (14336, 4096, torch.bfloat16), (1000, 264, torch.bfloat16),
])
def test_gemv_transposed_matches_oracle(A, rows, cols, dt):
    if (rows, cols) == (2, 3):
        Ah = torch.tensor([1, 2, 3, 4, 5, 6], dtype=torch.float32)
        xh = torch.ones(2)
    else:
        Ah = synth.normal((rows * cols,), seed=rows + cols, dtype=dt)
        xh = synth.normal((rows,), seed=rows * 3 + 1)
    Ad, xd = dev(Ah), dev(xh)
    y = torch.full((cols,), float("nan"), device="cuda")
    ws = A.workspace(A.ds_gemv_workspace_bytes(rows, cols, A.dtype_code(Ad)))
    A.ds_gemv_transposed(Ad, xd, rows, cols, y, ws)
    got = host(y)
    ref = O.gemv_transposed(synth.to_numpy_storage(Ah), xh.double().numpy(), rows, cols,
                            O.DT_BF16 if dt == torch.bfloat16 else O.DT_F32)
    if (rows, cols) == (2, 3):
        assert got.tolist() == [5.0, 7.0, 9.0]
    assert rel_err(got, ref) <= FP32_TOL
    # bit-stable from run to run
    y2 = torch.empty_like(y)
    A.ds_gemv_transposed(Ad, xd, rows, cols, y2, ws)
    assert torch.equal(y, y2)
    assert A.ds_workspace_error(ws) == 0


@pytest.mark.parametrize("rows,cols,dt", [(40, 16, torch.float32), (1000, 4096, torch.float32),
                                          (128256, 4096, torch.bfloat16), (151936, 1024, torch.bfloat16),
                                          (37, 12, torch.float32)])
def test_gemv_untransposed_matches_oracle(A, rows, cols, dt):
    Wh = synth.normal((rows * cols,), seed=rows, dtype=dt)
    xh = synth.normal((cols,), seed=cols)
    y = torch.full((rows,), float("nan"), device="cuda")
    A.ds_gemv(dev(Wh), dev(xh), rows, cols, y)
    ref = O.gemv(synth.to_numpy_storage(Wh), xh.double().numpy(), rows, cols,
                 O.DT_BF16 if dt == torch.bfloat16 else O.DT_F32)
    assert rel_err(host(y), ref) <= FP32_TOL


# ----------------------------------------------------------------- glue
def test_residual_add_is_exact(A):
    for n in (6, 4096, 100003):
        a = synth.normal((n,), seed=n)
        b = synth.normal((n,), seed=n + 1)
        out = torch.empty(n, device="cuda")
        A.ds_residual_add(dev(a), dev(b), out, n)
        assert np.abs(host(out) - O.residual_add(a.numpy(), b.numpy())).max() == 0.0
    a = torch.arange(6, dtype=torch.float32)
    b = 10 - a
    out = torch.empty(6, device="cuda")
    A.ds_residual_add(dev(a), dev(b), out, 6)
    assert host(out).tolist() == [10.0] * 6


@pytest.mark.parametrize("n,with_x,wdt", [(4096, True, torch.float32), (4096, False, torch.float32),
                                          (1024, True, torch.bfloat16), (17, True, torch.float32)])
def test_add_rmsnorm_matches_oracle(A, n, with_x, wdt):
    r = synth.normal((n,), seed=1)
    x = synth.normal((n,), seed=2) if with_x else None
    w = synth.normal((n,), seed=3, mean=1.0, std=0.1, dtype=wdt)
    rd = dev(r)
    h = torch.empty(n, device="cuda")
    A.ds_add_rmsnorm(rd, None if x is None else dev(x), dev(w), 1e-5, h, n)
    r_ref, h_ref = O.add_rmsnorm(r.numpy(), None if x is None else x.numpy(), synth.to_numpy_storage(w),
                                 1e-5, O.DT_BF16 if wdt == torch.bfloat16 else O.DT_F32)
    assert np.array_equal(host(rd), r_ref)
    assert rel_err(host(h), h_ref) <= FP32_TOL


def test_silu_mul_matches_oracle(A):
    n = 14336
    g = synth.normal((n,), seed=4, std=4.0)
    u = synth.normal((n,), seed=5)
    out = torch.empty(n, device="cuda")
    A.ds_silu_mul(dev(g), dev(u), out, n)
    assert rel_err(host(out), O.silu_mul(g.double().numpy(), u.double().numpy())) <= FP32_TOL
    z = torch.zeros(4, device="cuda")
    o = torch.empty(4, device="cuda")
    A.ds_silu_mul(z, z + 3, o, 4)
    assert host(o).tolist() == [0.0] * 4


@pytest.mark.parametrize("layout", [0, 1])
def test_rope_matches_oracle_at_random_positions(A, layout):
    nq, nk, hd = 32, 8, 128
    gen = torch.Generator().manual_seed(7)
    for trial in range(6):
        pos = int(torch.randint(0, 8192, (1,), generator=gen)) if trial else 0
        q = synth.normal((nq * hd,), seed=10 + trial)
        k = synth.normal((nk * hd,), seed=20 + trial)
        qd, kd = dev(q), dev(k)
        A.ds_rope(qd, kd, pos, nq, nk, hd, 10000.0, layout)
        q_ref = O.rope(q.double().numpy(), nq, hd, pos, 10000.0, layout)
        k_ref = O.rope(k.double().numpy(), nk, hd, pos, 10000.0, layout)
        assert rel_err(host(qd), q_ref) <= FP32_TOL
        assert rel_err(host(kd), k_ref) <= FP32_TOL
        if pos == 0:
            assert torch.equal(qd.cpu(), q)


def test_kv_cache_append_example_and_bf16_rounding(A):
    cache = torch.zeros(9, device="cuda")
    cache[:6] = torch.arange(6, dtype=torch.float32, device="cuda")
    A.ds_kv_cache_append(cache, 9, 6, dev(torch.tensor([100.0, 101.0, 102.0])), 3)
    assert host(cache).tolist() == [0, 1, 2, 3, 4, 5, 100, 101, 102]
    vals = synth.normal((4096,), seed=9, std=3.0)
    cb = torch.zeros(8192, dtype=torch.bfloat16, device="cuda")
    A.ds_kv_cache_append(cb, 8192, 1000, dev(vals), 4096)
    ref = np.zeros(8192, dtype=np.uint16)
    assert O.kv_cache_append(ref, O.DT_BF16, 1000, vals.double().numpy(), 4096) == 560
    assert np.array_equal(host(cb), ref)
    with pytest.raises(A.DecodeStepError) as e:
        A.ds_kv_cache_append(cb, 8192, 8000, dev(vals), 4096)
    assert e.value.code == A.DS_CACHE_CAPACITY_EXCEEDED


# ----------------------------------------------------------------- attention
def _attn_case(A, n_qh, n_kvh, hd, lens, kv_dt, block_tokens, paged, seed):
    n_seqs = len(lens)
    max_ctx = max(lens)
    max_blocks = (max_ctx + block_tokens - 1) // block_tokens
    n_blocks = n_seqs * max_blocks
    rows = n_blocks * block_tokens
    K = synth.normal((rows, n_kvh * hd), seed=seed, dtype=kv_dt)
    V = synth.normal((rows, n_kvh * hd), seed=seed + 1, dtype=kv_dt)
    q = synth.normal((n_seqs, n_qh * hd), seed=seed + 2)
    table = None
    if paged:
        g = torch.Generator().manual_seed(seed)
        table = torch.randperm(n_blocks, generator=g).to(torch.int32).reshape(n_seqs, max_blocks)
    out = torch.full((n_seqs, n_qh * hd), float("nan"), device="cuda")
    ws = A.workspace(A.ds_attention_workspace_bytes(n_seqs, n_qh, n_kvh, hd, max_blocks * block_tokens))
    lens_d = dev(torch.tensor(lens, dtype=torch.int32))
    scale = 1.0 / np.sqrt(hd)
    A.ds_gqa_decode_attn(dev(q), dev(K), dev(V), rows, None if table is None else dev(table), max_blocks,
                         block_tokens, lens_d, n_seqs, n_qh, n_kvh, hd, scale, out, ws)
    dt = O.DT_BF16 if kv_dt == torch.bfloat16 else O.DT_F32
    Kn, Vn = synth.to_numpy_storage(K), synth.to_numpy_storage(V)
    got = host(out)
    for s in range(n_seqs):
        ref = O.gqa_attention(q[s].double().numpy(), Kn, Vn, dt, lens[s], n_qh, n_kvh, hd, scale,
                              block_table=None if table is None else table.numpy(), max_blocks=max_blocks,
                              block_tokens=block_tokens, seq=s)
        assert rel_err(got[s], ref) <= FP32_TOL, (s, lens[s])
    assert A.ds_workspace_error(ws) == 0
    return out


@pytest.mark.parametrize("lens,paged", [([1], False), ([17], False), ([1024], False), ([4099], True),
                                        ([8192], False), ([5, 300, 1], True)])
def test_attention_8b_heads_bf16(A, lens, paged):
    _attn_case(A, 32, 8, 128, lens, torch.bfloat16, 16, paged, seed=len(lens) * 100 + lens[0])


def test_attention_many_sequences_paged_pool(A):
    """64 sequences, contexts 1..600, 16-position blocks scattered over the
    pool: the whole-block streaming kernel with its even split of blocks over
    the SMs and the per-sequence merge."""
    lens = synth.context_lengths(64, 1, 600, seed=21)
    _attn_case(A, 32, 8, 128, lens, torch.bfloat16, 16, True, seed=22)


def test_attention_fp32_cache_two_heads_per_group(A):
    _attn_case(A, 16, 8, 128, [5, 300, 1, 64, 17, 33], torch.float32, 16, True, seed=23)


@pytest.mark.parametrize("n_qh,n_kvh,hd", [(4, 2, 4), (16, 8, 128), (8, 8, 64), (8, 1, 32)])
def test_attention_fp32_shapes(A, n_qh, n_kvh, hd):
    _attn_case(A, n_qh, n_kvh, hd, [1, 29, 64], torch.float32, 4, False, seed=hd)


def test_attention_single_position_returns_v_and_is_deterministic(A):
    a = _attn_case(A, 32, 8, 128, [700], torch.bfloat16, 16, False, seed=3)
    b = _attn_case(A, 32, 8, 128, [700], torch.bfloat16, 16, False, seed=3)
    assert torch.equal(a, b)


# ----------------------------------------------------------------- argmax / sample
def test_argmax_ties_go_to_lowest_index(A):
    n = 128256
    rows = []
    for seed in range(4):
        l, planted = synth.logits_with_ties(n, 3, seed=seed)
        rows.append((l, planted))
    L = torch.stack([r[0] for r in rows])
    ids = torch.empty(4, dtype=torch.int32, device="cuda")
    mx = torch.empty(4, device="cuda")
    ws = A.workspace(A.ds_argmax_workspace_bytes(4, n))
    A.ds_greedy_argmax(dev(L), 4, n, ids, mx, ws)
    for r, (l, planted) in enumerate(rows):
        i, m = O.argmax(l.numpy())
        assert int(ids[r]) == i == planted[0] == int(torch.argmax(l))
        assert float(mx[r]) == m


def test_argmax_page_examples_and_nan(A):
    for vals, want in (([1.0, 9.0, 3.0], 1), ([2.0, 7.0, 7.0, 1.0], 1), ([1.0, float("nan"), 5.0, float("nan")], 1)):
        l = torch.tensor(vals)
        ids = torch.empty(1, dtype=torch.int32, device="cuda")
        ws = A.workspace(A.ds_argmax_workspace_bytes(1, len(vals)))
        A.ds_greedy_argmax(dev(l), 1, len(vals), ids, None, ws)
        assert int(ids[0]) == want == O.argmax(l.numpy())[0] == int(torch.argmax(l))


# A draw (or a top-p cut) closer than this to a boundary of the oracle's CDF,
# as a fraction of the mass, may go either way: CUDA's expf and the C
# library's differ by up to 2.5 ulp (1.5e-7 relative) per term, which moves a
# normalised running sum by at most about twice that; the kernel's
# fixed-point rounding adds under 1e-9.
SAMPLE_MARGIN = 4e-7


def _sample_check(A, logits, T, k, p, u, min_compared=None):
    n_rows, n = logits.shape
    ids = torch.empty(n_rows, dtype=torch.int32, device="cuda")
    ws = A.workspace(A.ds_sample_workspace_bytes(n_rows, n))
    A.ds_sample(dev(logits), n_rows, n, T, k, p, dev(u), ids, ws)
    got = host(ids)
    compared = 0
    for r in range(n_rows):
        want, margin = O.sample(logits[r].numpy(), T, k, p, float(u[r]))
        if margin < SAMPLE_MARGIN:
            continue  # the draw or the cut sits on a CDF boundary: either neighbour is a valid pick
        assert got[r] == want, (r, got[r], want, margin)
        compared += 1
    need = n_rows - max(1, n_rows // 20) if min_compared is None else min_compared
    assert compared >= need, (compared, n_rows)
    assert A.ds_workspace_error(ws) == 0
    return got


def test_sampler_matches_oracle_at_the_page_settings(A):
    n = 128256
    L = torch.stack([synth.normal((n,), seed=100 + r) for r in range(64)])
    u = synth.uniform_draws(64, seed=0)
    _sample_check(A, L, 0.8, 50, 0.95, u)


@pytest.mark.parametrize("T,k,p", [(0.8, 0, 0.9), (1.0, 5000, 0.95), (0.8, 50, 0.95), (1.2, 0, 1.0)])
def test_sampler_whole_vocabulary_settings(A, T, k, p):
    """64 rows of 128,256 logits: top-k off, wide, or the page's 50, with
    top-p cuts that keep tens of thousands of survivors."""
    n = 128256
    L = torch.stack([synth.normal((n,), seed=300 + r) for r in range(64)])
    u = synth.uniform_draws(64, seed=2)
    _sample_check(A, L, T, k, p, u, min_compared=40)


@pytest.mark.parametrize("n,k", [(151936, 0), (300000, 0), (300000, 2000), (777, 0), (40, 3)])
def test_sampler_other_vocabulary_sizes(A, n, k):
    """The Qwen vocabulary, a row too long for the keys to stay in shared
    memory (read again from memory at every level), and small rows."""
    rows = 8
    # the 300,000-wide rows get a wider spread, so that their CDFs' steps near
    # the cut and the draw are far wider than the comparison margin
    std = 3.0 if n > 200000 else 1.5
    L = torch.stack([synth.normal((n,), seed=400 + r, std=std) for r in range(rows)])
    u = synth.uniform_draws(rows, seed=3)
    _sample_check(A, L, 0.9, k, 0.92, u, min_compared=5)


def test_sampler_flat_vocabulary_is_exact(A):
    """128,256 equal logits: every exponential is exactly 1, so the draw
    (j + 1/2) / n must pick token j, a top-p cut of 0.3 keeps ids
    0..38,476, and a top-k of 1,000 over the tie keeps ids 0..999."""
    n = 128256
    js = [0, 1, 777, 50000, 99999, 128000, n - 1]
    L = torch.full((len(js), n), 0.25)
    u = torch.tensor([(j + 0.5) / n for j in js], dtype=torch.float32)
    assert _sample_check(A, L, 1.0, 0, 1.0, u).tolist() == js
    kept = 38477
    js = [0, 12345, 30000, kept - 1]
    L = torch.full((len(js), n), 0.25)
    u = torch.tensor([(j + 0.5) / kept for j in js], dtype=torch.float32)
    assert _sample_check(A, L, 1.0, 0, 0.3, u).tolist() == js
    L = torch.full((2, n), -3.0)
    u = torch.tensor([0.0005, 0.9995])
    assert _sample_check(A, L, 1.0, 1000, 1.0, u).tolist() == [0, 999]


def test_sampler_topk_boundary_ties_at_full_width(A):
    """The k-th largest value planted 40 times across the row: the survivors
    among its copies are the lowest-index ones; top-p off so every survivor
    can be drawn."""
    n, rows = 128256, 16
    L = torch.stack([synth.normal((n,), seed=500 + r) for r in range(rows)])
    g = torch.Generator().manual_seed(501)
    for r in range(rows):
        v = float(torch.sort(L[r], descending=True).values[30])
        L[r, torch.randperm(n, generator=g)[:40]] = v
    u = torch.linspace(0.01, 0.99, rows)
    _sample_check(A, L, 1.0, 50, 1.0, u, min_compared=12)


def test_sampler_greedy_and_degenerate_rows(A):
    n = 128256
    L = synth.normal((3, n), seed=600)
    L[0, [10, 90000, 120000]] = 9.0   # greedy: the first of the planted maxima
    L[1, 5000] = float("nan")          # a NaN ranks above every number
    L[2, [70000, 80000]] = float("inf")
    ids = torch.empty(3, dtype=torch.int32, device="cuda")
    ws = A.workspace(A.ds_sample_workspace_bytes(3, n))
    A.ds_sample(dev(L[:1]), 1, n, 0.0, 50, 0.95, dev(torch.zeros(1)), ids, ws)
    assert int(ids[0]) == 10 == O.argmax(L[0].numpy())[0]
    assert A.ds_workspace_error(ws) == 0
    A.ds_sample(dev(L[1:]), 2, n, 0.8, 0, 0.9, dev(torch.tensor([0.3, 0.6])), ids, ws)
    assert host(ids)[:2].tolist() == [5000, 70000]
    assert A.ds_workspace_error(ws) == A.DS_ERR_SAMPLING


@pytest.mark.parametrize("T,k,p", [(0.8, 1, 0.95), (0.8, 50, 1e-6), (1.5, 1024, 0.9), (0.7, 0, 0.8),
                                   (1.0, 7, 1.0)])
def test_sampler_special_settings(A, T, k, p):
    n = 1000 if k in (0,) else 50000
    L = torch.stack([synth.normal((n,), seed=200 + r, std=2.0) for r in range(8)])
    u = synth.uniform_draws(8, seed=1)
    got = _sample_check(A, L, T, k, p, u, min_compared=6)
    if k == 1 or p < 1e-3:
        assert all(got[r] == int(torch.argmax(L[r])) for r in range(8))


def test_sampler_u_zero_and_topk_ties(A):
    l = torch.tensor([[1.0, 3.0, 3.0, 3.0, 0.0, 3.0]] * 2)
    u = torch.tensor([0.25, 0.75])
    got = _sample_check(A, l, 1.0, 2, 1.0, u)
    assert got.tolist() == [1, 2]
    L = synth.normal((1, 128256), seed=5)
    got = _sample_check(A, L, 0.8, 50, 0.95, torch.zeros(1))
    assert got[0] == int(torch.argmax(L[0]))
