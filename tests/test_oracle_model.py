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
