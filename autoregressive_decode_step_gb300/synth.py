"""Seeded synthetic inputs shared by the CUDA path's tests and the oracle.

This module makes random numbers and lays them out; it holds none of the
decode step's arithmetic.  Everything is reproducible from a seed.
"""
import random

import numpy as np
import torch

from . import configs as C


# ------------------------------------------------------------------ toy model
def p4_toy_weights(cfg=C.TOY, seed=0):
    """Weights of the tiny decoder drawn as "The forward pass end to end"
    ("The code": init_weights) draws them: one ``random.Random(seed)`` stream of
    Gaussian(0, std) values, row by row, matrices in the order emb, out, then
    per layer wq, wk, wv, wo, gate, up, down.  Matrices are [out][in] lists;
    norm weights are 1.0."""
    rng = random.Random(seed)
    std = cfg["weight_std"]
    hd = cfg["head_dim"]

    def draw(r, c):
        return [[rng.gauss(0, std) for _ in range(c)] for _ in range(r)]

    W = {"emb": draw(cfg["vocab"], cfg["d"]), "out": draw(cfg["vocab"], cfg["d"]),
         "norm": [1.0] * cfg["d"], "layers": []}
    for _ in range(cfg["n_layer"]):
        layer = {}
        layer["wq"] = draw(cfg["n_qh"] * hd, cfg["d"])
        layer["wk"] = draw(cfg["n_kvh"] * hd, cfg["d"])
        layer["wv"] = draw(cfg["n_kvh"] * hd, cfg["d"])
        layer["wo"] = draw(cfg["d"], cfg["n_qh"] * hd)
        layer["gate"] = draw(cfg["ff"], cfg["d"])
        layer["up"] = draw(cfg["ff"], cfg["d"])
        layer["down"] = draw(cfg["d"], cfg["ff"])
        layer["n1"] = [1.0] * cfg["d"]
        layer["n2"] = [1.0] * cfg["d"]
        W["layers"].append(layer)
    return W


def p4_to_storage(W, cfg=C.TOY):
    """[out][in] matrices -> the storage layout (float32, [in, out] row-major
    for projections, q|k|v and gate|up concatenated column-wise)."""
    f32 = lambda a: np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))
    st = {"emb": f32(W["emb"]).ravel(), "out": f32(W["out"]).ravel(),
          "norm": f32(W["norm"]), "n1": [], "wqkv": [], "wo": [], "n2": [], "wgu": [], "wd": []}
    for L in W["layers"]:
        st["n1"].append(f32(L["n1"]))
        st["n2"].append(f32(L["n2"]))
        st["wqkv"].append(f32(np.concatenate([L["wq"], L["wk"], L["wv"]], axis=0).T).ravel())
        st["wo"].append(f32(np.asarray(L["wo"]).T).ravel())
        st["wgu"].append(f32(np.concatenate([L["gate"], L["up"]], axis=0).T).ravel())
        st["wd"].append(f32(np.asarray(L["down"]).T).ravel())
    return st


def toy_prompt(seed=0, n=6, vocab=40):
    """Six ids uniform in [0, vocab) from their own ``random.Random(seed)``."""
    rng = random.Random(seed)
    return [rng.randrange(vocab) for _ in range(n)]


P4_PROMPT = [3, 14, 15, 9, 2, 6]


# ------------------------------------------------------------------ models
def _tdtype(code):
    return torch.float32 if code == C.F32 else torch.bfloat16


def model_weights(cfg, seed=0, device="cpu"):
    """Random-init weights in the storage layout as torch tensors on `device`:
    N(0, weight_std) in the model's weight dtype, norm weights 1.0."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    wdt = _tdtype(cfg["w_dtype"])
    std = cfg["weight_std"]
    d, ff, hd = cfg["d"], cfg["ff"], cfg["head_dim"]

    def randn(*shape):
        t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        return t.mul_(std).to(wdt)

    ones = lambda: torch.ones(d, device=device, dtype=torch.float32)
    W = {"emb": randn(cfg["vocab"], d)}
    W["out"] = W["emb"] if cfg["tied"] else randn(cfg["vocab"], d)
    W["norm"] = ones()
    for k in ("n1", "wqkv", "wo", "n2", "wgu", "wd"):
        W[k] = []
    for _ in range(cfg["n_layer"]):
        W["n1"].append(ones())
        W["wqkv"].append(randn(d, C.qkv_cols(cfg)))
        W["wo"].append(randn(cfg["n_qh"] * hd, d))
        W["n2"].append(ones())
        W["wgu"].append(randn(d, 2 * ff))
        W["wd"].append(randn(ff, d))
    return W


def qk_norm_weights(cfg, seed=0, device="cpu", std=0.3):
    """Per-layer QK-norm weights (fp32 [head_dim], N(1, std)) as the
    ``q_norm`` and ``k_norm`` lists of a weight dict."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    hd = cfg["head_dim"]
    mk = lambda: torch.randn(hd, generator=g, device=device, dtype=torch.float32).mul_(std).add_(1.0)
    return {"q_norm": [mk() for _ in range(cfg["n_layer"])], "k_norm": [mk() for _ in range(cfg["n_layer"])]}


def to_numpy_storage(t):
    """A torch tensor as the oracle's numpy storage: float32, or uint16 bits
    for bf16."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).ravel()
    return t.to(torch.float32).numpy().ravel()


def weights_to_numpy(W):
    out = {}
    for k, v in W.items():
        out[k] = [to_numpy_storage(t) for t in v] if isinstance(v, list) else to_numpy_storage(v)
    return out


def prompt_ids(cfg, n, seed=0):
    """n token ids uniform in [0, vocab)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, cfg["vocab"], (n,), generator=g, dtype=torch.int64).tolist()


def synthetic_kv(cfg, n_rows, seed=0, device="cpu", std=1.0):
    """Per-layer K and V caches of n_rows rows (n_kvh * head_dim values each),
    N(0, std) in the cache dtype — a stand-in for a prefilled context."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = _tdtype(cfg["kv_dtype"])
    row = cfg["n_kvh"] * cfg["head_dim"]
    ks, vs = [], []
    for _ in range(cfg["n_layer"]):
        ks.append(torch.randn(n_rows, row, generator=g, device=device).mul_(std).to(dt))
        vs.append(torch.randn(n_rows, row, generator=g, device=device).mul_(std).to(dt))
    return ks, vs


def uniform_draws(n, seed=0):
    """n float32 draws in [0, 1), torch CPU generator."""
    g = torch.Generator().manual_seed(seed)
    return torch.rand(n, generator=g, dtype=torch.float32)


def normal(shape, seed=0, device="cpu", mean=0.0, std=1.0, dtype=torch.float32):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return t.mul_(std).add_(mean).to(dtype)


def logits_with_ties(n, n_ties=3, seed=0, device="cpu"):
    """N(0,1) logits with the maximum planted at `n_ties` random distinct
    indices; returns (logits, sorted planted indices)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    l = torch.randn(n, generator=g, dtype=torch.float32)
    idx = torch.randperm(n, generator=g)[:n_ties].sort().values
    l[idx] = float(l.max()) + 1.0
    return l.to(device), idx.tolist()


def context_lengths(n_seqs, lo, hi, seed=0):
    """n_seqs context lengths uniform in [lo, hi] (the batched workload's mix)."""
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, (n_seqs,), generator=g, dtype=torch.int64).tolist()


def paged_block_table(n_seqs, max_blocks, seed=0):
    """int32 [n_seqs, max_blocks]: a seeded permutation of the pool's
    n_seqs * max_blocks physical blocks, so consecutive blocks of a sequence
    are scattered over the pool."""
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(n_seqs * max_blocks, generator=g).to(torch.int32).view(n_seqs, max_blocks)
