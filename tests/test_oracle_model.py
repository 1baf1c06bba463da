"""Pins of the oracle's decode step: the tiny decoder's printed result, cached
decode against full recompute, an independent pure-Python statement of the
same model, and closed forms on degenerate models.  CPU only."""
import json
import os

import numpy as np
import pytest

import oracle as O
from autoregressive_decode_step_gb300 import configs as C
from autoregressive_decode_step_gb300 import synth
from tests.toy_reference import ToyDecoder, first_argmax

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def toy_model(cfg=C.TOY, seed=0):
    Wp4 = synth.p4_toy_weights(cfg, seed)
    st = synth.p4_to_storage(Wp4, cfg)
    ocfg = dict(cfg, max_blocks=cfg["max_seq"], block_tokens=1)
    return Wp4, st, O.Model(ocfg, st)


def test_toy_greedy_output_matches_page():
    g = json.load(open(os.path.join(GOLD, "p4_toy_decoder.json")))
    _, _, m = toy_model()
    out, _ = O.greedy_generate(m, g["prompt"], g["n_new"])
    assert out[:len(g["generated_prefix"])] == g["generated_prefix"]


def test_toy_cached_decode_equals_full_recompute():
    g = json.load(open(os.path.join(GOLD, "p4_toy_decoder.json")))
    for prompt in (g["prompt"], synth.toy_prompt(0)):
        _, _, m = toy_model()
        fast, step_logits = O.greedy_generate(m, prompt, g["n_new"])
        seq = list(prompt)
        for i in range(g["n_new"]):
            lg = m.recompute(seq)
            np.testing.assert_allclose(lg, step_logits[i], rtol=0, atol=1e-12)
            seq.append(O.argmax(lg.astype(np.float32))[0])
        assert fast == seq[len(prompt):]


def test_toy_oracle_agrees_with_independent_python_model():
    Wp4, st, m = toy_model()
    # the independent model reads the same fp32-rounded weights
    W32 = {"emb": st["emb"].reshape(40, 16).astype(np.float64).tolist(),
           "out": st["out"].reshape(40, 16).astype(np.float64).tolist(), "norm": [1.0] * 16,
           "layers": []}
    for L in Wp4["layers"]:
        W32["layers"].append({k: np.asarray(v, np.float64).astype(np.float32).astype(np.float64).tolist()
                              for k, v in L.items()})
    ref = ToyDecoder(dict(C.TOY), W32)
    prompt = synth.toy_prompt(0)
    seq = list(prompt)
    for pos in range(len(prompt) + 16):
        a = m.step(seq[pos], pos)
        b = np.array(ref.logits(seq[pos], pos))
        # the oracle stores the residual in fp32 and KV through fp32; the
        # Python model keeps fp64 throughout
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-5 * np.abs(b).max())
        if pos + 1 >= len(seq):
            seq.append(first_argmax(list(b)))
            assert O.argmax(a.astype(np.float32))[0] == seq[-1]


def test_kv_bytes_per_token():
    g = json.load(open(os.path.join(GOLD, "p4_toy_decoder.json")))
    assert C.kv_bytes_per_token(C.TOY, 2) == g["kv_bytes_per_token_fp16"]
    assert C.kv_bytes_per_token(dict(C.TOY, n_kvh=4), 2) == g["kv_bytes_per_token_fp16_full_mha"]


def small_cfg(**kw):
    cfg = dict(vocab=97, d=64, n_layer=2, n_qh=4, n_kvh=2, head_dim=16, ff=96,
               rope_base=10000.0, rope_layout=O.ROPE_HALF_SPLIT, tied=0, w_dtype=O.DT_F32,
               kv_dtype=O.DT_F32, eps=1e-5, max_blocks=32, block_tokens=1, weight_std=0.1)
    cfg.update(kw)
    return cfg


def random_storage(cfg, seed):
    W = synth.model_weights(cfg, seed=seed)
    return synth.weights_to_numpy(W)


def test_layerless_model_is_head_of_normalised_embedding():
    cfg = small_cfg(n_layer=0)
    st = random_storage(cfg, 1)
    m = O.Model(cfg, st)
    E = st["emb"].reshape(cfg["vocab"], cfg["d"]).astype(np.float64)
    Wout = st["out"].reshape(cfg["vocab"], cfg["d"]).astype(np.float64)
    x = E[5]
    h = x / np.sqrt(np.mean(x * x) + 1e-5)
    np.testing.assert_allclose(m.step(5, 0), Wout @ h, rtol=1e-12)


def test_zero_output_projections_make_layers_identity():
    cfg = small_cfg()
    st = random_storage(cfg, 2)
    for l in range(cfg["n_layer"]):
        st["wo"][l] = np.zeros_like(st["wo"][l])
        st["wd"][l] = np.zeros_like(st["wd"][l])
    m = O.Model(cfg, st)
    m0 = O.Model(dict(cfg, n_layer=0), st)
    for pos, t in enumerate([3, 9, 27]):
        np.testing.assert_array_equal(m.step(t, pos), m0.step(t, pos))


def test_tied_head_uses_embedding():
    cfg = small_cfg(tied=1)
    st = random_storage(cfg, 3)
    st_untied = dict(st, out=st["emb"].copy())
    a = O.Model(cfg, st).step(7, 0)
    b = O.Model(dict(cfg, tied=0), st_untied).step(7, 0)
    np.testing.assert_array_equal(a, b)


def test_bf16_model_cached_equals_recompute_and_paged_equals_contiguous():
    cfg = small_cfg(w_dtype=O.DT_BF16, kv_dtype=O.DT_BF16)
    st = random_storage(cfg, 4)
    m = O.Model(cfg, st)
    bt = 4
    table = np.array([[5, 2, 7, 0, 1, 3, 6, 4]], dtype=np.int32)
    mp = O.Model(dict(cfg, block_tokens=bt, max_blocks=8, block_table=table, n_blocks=8), st)
    toks = [11, 3, 50, 50, 8, 90, 1, 13, 2, 71, 64]
    for pos, t in enumerate(toks):
        a = m.step(t, pos)
        b = mp.step(t, pos)
        np.testing.assert_array_equal(a, b)
    np.testing.assert_allclose(m.recompute(toks), a, rtol=0, atol=0)


# QK-norm as Qwen3 checkpoints define it (not on the pages): every q and k
# head RMS-normalised over head_dim with the layer's q_norm / k_norm weight,
# before RoPE.
def qk_norm_storage(cfg, seed):
    st = random_storage(cfg, seed)
    rng = np.random.default_rng(seed)
    st["q_norm"] = [rng.normal(1.0, 0.3, cfg["head_dim"]).astype(np.float32) for _ in range(cfg["n_layer"])]
    st["k_norm"] = [rng.normal(1.0, 0.3, cfg["head_dim"]).astype(np.float32) for _ in range(cfg["n_layer"])]
    return st


def test_qk_norm_k_row_is_each_head_normalised_then_rotated():
    """Layer 0's K row at position 5, rebuilt from the separately pinned
    primitives: RMSNorm of the embedding, the k columns of the projection,
    each KV head normalised with k_norm (not q_norm), then rotated."""
    cfg = small_cfg()
    st = qk_norm_storage(cfg, 6)
    m = O.Model(cfg, st)
    tok, pos = 17, 5
    m.step(tok, pos)
    d, hd, nq, nkv = cfg["d"], cfg["head_dim"], cfg["n_qh"] * cfg["head_dim"], cfg["n_kvh"] * cfg["head_dim"]
    x = st["emb"].reshape(cfg["vocab"], d)[tok].astype(np.float64)
    h = O.rmsnorm(x, st["n1"][0], 1e-5)
    qkv = O.gemv_transposed(st["wqkv"][0], h, d, nq + 2 * nkv)
    k = qkv[nq:nq + nkv].copy()
    for g in range(cfg["n_kvh"]):
        k[g * hd:(g + 1) * hd] = O.rmsnorm(k[g * hd:(g + 1) * hd], st["k_norm"][0], 1e-5)
    want = O.rope(k, cfg["n_kvh"], hd, pos, cfg["rope_base"], cfg["rope_layout"])
    got = m.k[0][pos * nkv:(pos + 1) * nkv].astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-7)
    # the same row without QK-norm is far from it
    plain = O.Model(cfg, random_storage(cfg, 6))
    plain.step(tok, pos)
    assert not np.allclose(plain.k[0][pos * nkv:(pos + 1) * nkv], got, rtol=1e-2)


def test_qk_norm_makes_every_head_scale_free():
    """Scaling one q head's and one k head's projection columns leaves every
    logit unchanged under QK-norm (eps tiny), and changes them without it."""
    cfg = small_cfg(eps=1e-12)
    st = qk_norm_storage(cfg, 7)
    hd, nq = cfg["head_dim"], cfg["n_qh"] * cfg["head_dim"]
    cols = nq + 2 * cfg["n_kvh"] * hd
    scaled = dict(st, wqkv=[w.copy() for w in st["wqkv"]])
    for l in range(cfg["n_layer"]):
        w = scaled["wqkv"][l].reshape(cfg["d"], cols)
        w[:, 1 * hd:2 * hd] *= 4.0          # q head 1 (powers of two: exact in fp32)
        w[:, nq:nq + hd] *= 0.25            # k of KV head 0
    toks = [4, 60, 60, 13, 88]
    a, b = O.Model(cfg, st), O.Model(cfg, scaled)
    for pos, t in enumerate(toks):
        # equal up to eps's share and the fp32 rounding of the stored K/V
        np.testing.assert_allclose(b.step(t, pos), a.step(t, pos), rtol=1e-6, atol=1e-9)
    plain = {k: v for k, v in st.items() if k not in ("q_norm", "k_norm")}
    plain_scaled = {k: v for k, v in scaled.items() if k not in ("q_norm", "k_norm")}
    pa, pb = O.Model(cfg, plain), O.Model(cfg, plain_scaled)
    diff = max(np.max(np.abs(pa.step(t, pos) - pb.step(t, pos))) for pos, t in enumerate(toks))
    assert diff > 1e-3


def test_qk_norm_cached_decode_equals_recompute():
    cfg = small_cfg()
    st = qk_norm_storage(cfg, 8)
    m = O.Model(cfg, st)
    toks = [5, 9, 2, 77, 31, 31, 60]
    for pos, t in enumerate(toks):
        last = m.step(t, pos)
    np.testing.assert_allclose(m.recompute(toks), last, rtol=0, atol=0)
