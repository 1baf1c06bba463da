"""Decode-step oracle — TEST INFRASTRUCTURE ONLY.

Python face of ``oracle.c``: a plain, slow CPU statement of the single-token
decode step.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg may import this package; the product path never does, and it
shares no code with the CUDA library.

Arrays are numpy.  Stored operands are float32 arrays, or uint16 arrays that
hold raw bf16 bits (numpy has no bfloat16); ``DT_F32`` / ``DT_BF16`` say which.
"""
import ctypes
import os

import numpy as np

from . import build as _build

DT_F32 = 0
DT_BF16 = 1
ROPE_HALF_SPLIT = 0
ROPE_INTERLEAVED = 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        D = ctypes.c_double
        L.or_threads.restype = ctypes.c_int
        L.or_set_threads.argtypes = [ctypes.c_int]
        L.or_f32_to_bf16.argtypes = [ctypes.c_float]
        L.or_f32_to_bf16.restype = ctypes.c_uint16
        L.or_residual_dims_check.argtypes = [I64, I64, I64]
        L.or_gemv_transposed.argtypes = [P, ctypes.c_int, P, I64, I64, P]
        L.or_gemv.argtypes = [P, ctypes.c_int, P, I64, I64, P]
        L.or_residual_add.argtypes = [P, P, P, I64]
        L.or_rmsnorm.argtypes = [P, P, ctypes.c_int, I64, D, P]
        L.or_add_rmsnorm.argtypes = [P, P, P, ctypes.c_int, I64, D, P]
        L.or_silu_mul.argtypes = [P, P, P, I64]
        L.or_rope.argtypes = [P, I64, I64, I64, D, ctypes.c_int, P]
        L.or_rope_freq.argtypes = [I64, I64, D, P]
        L.or_rope_freq.restype = D
        L.or_kv_cache_append.argtypes = [P, ctypes.c_int, I64, I64, P, I64, I64]
        L.or_gqa_attention.argtypes = [P, P, P, ctypes.c_int, P, I64, I64, I64, I64, I64, I64, I64, D, P]
        L.or_argmax.argtypes = [P, I64, P]
        L.or_argmax.restype = I64
        L.or_sample.argtypes = [P, I64, ctypes.c_float, I64, ctypes.c_float, ctypes.c_float, P]
        L.or_sample.restype = I64
        L.or_decode_step.argtypes = [P, P, P, P, P, P, I64, I64, I64, P]
        L.or_recompute_logits.argtypes = [P, P, P, P, P, P, I64, P]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _stored(a, dt):
    """A stored operand: float32 values, or uint16 raw bf16 bits."""
    return _c(a, np.float32 if dt == DT_F32 else np.uint16)


def threads():
    """Threads the oracle's parallel loops use."""
    return lib().or_threads()


def set_threads(n):
    """Threads for the oracle's later parallel loops (timing only: every
    output element is computed the same way whatever the count)."""
    lib().or_set_threads(int(n))


# ---------------------------------------------------------------- elements
def f32_to_bf16_bits(x):
    """Round float32 values to bf16 (nearest, ties to even); returns uint16 bits."""
    x = np.asarray(x, dtype=np.float32).ravel()
    f = lib().or_f32_to_bf16
    return np.array([f(float(v)) for v in x], dtype=np.uint16)


def bf16_bits_to_f64(bits):
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def widen(a, dt):
    return np.asarray(a, dtype=np.float64) if dt == DT_F32 else bf16_bits_to_f64(a)


# ---------------------------------------------------------------- contract
def residual_dims_check(n, a_len, b_len):
    return lib().or_residual_dims_check(n, a_len, b_len)


# ---------------------------------------------------------------- ops
def gemv_transposed(A, x, rows, cols, dt=DT_F32):
    A = _stored(A, dt)
    x = _c(x, np.float64)
    assert A.size == rows * cols and x.size == rows
    y = np.empty(cols, dtype=np.float64)
    lib().or_gemv_transposed(_ptr(A), dt, _ptr(x), rows, cols, _ptr(y))
    return y


def gemv(W, x, rows, cols, dt=DT_F32):
    W = _stored(W, dt)
    x = _c(x, np.float64)
    assert W.size == rows * cols and x.size == cols
    y = np.empty(rows, dtype=np.float64)
    lib().or_gemv(_ptr(W), dt, _ptr(x), rows, cols, _ptr(y))
    return y


def residual_add(a, b):
    a = _c(a, np.float32)
    b = _c(b, np.float32)
    out = np.empty_like(a)
    lib().or_residual_add(_ptr(a), _ptr(b), _ptr(out), a.size)
    return out


def rmsnorm(x, g, eps=1e-5, g_dt=DT_F32):
    x = _c(x, np.float64)
    g = _stored(g, g_dt)
    y = np.empty_like(x)
    lib().or_rmsnorm(_ptr(x), _ptr(g), g_dt, x.size, eps, _ptr(y))
    return y


def add_rmsnorm(residual, x, w, eps=1e-5, w_dt=DT_F32):
    """Returns (updated residual float32, h float64)."""
    r = _c(residual, np.float32).copy()
    xx = None if x is None else _c(x, np.float32)
    w = _stored(w, w_dt)
    h = np.empty(r.size, dtype=np.float64)
    lib().or_add_rmsnorm(_ptr(r), _ptr(xx), _ptr(w), w_dt, r.size, eps, _ptr(h))
    return r, h


def silu_mul(gate, up):
    g = _c(gate, np.float64)
    u = _c(up, np.float64)
    out = np.empty_like(g)
    lib().or_silu_mul(_ptr(g), _ptr(u), _ptr(out), g.size)
    return out


def rope_scaling_vector(scaling):
    """{factor, low_freq_factor, high_freq_factor, original_max_position} as
    the oracle's four doubles; None: no scaling (factor 0)."""
    if not scaling:
        return np.zeros(4, dtype=np.float64)
    return np.array([scaling["factor"], scaling["low_freq_factor"], scaling["high_freq_factor"],
                     scaling["original_max_position"]], dtype=np.float64)


def rope_freq(p, head_dim, base, scaling=None):
    """Rotation frequency of pair p, optionally with long-context scaling."""
    sc = rope_scaling_vector(scaling)
    return lib().or_rope_freq(p, head_dim, base, _ptr(sc))


def rope(vec, n_heads, head_dim, pos, base, layout, scaling=None):
    v = _c(vec, np.float64).copy()
    assert v.size == n_heads * head_dim
    sc = rope_scaling_vector(scaling)
    lib().or_rope(_ptr(v), n_heads, head_dim, pos, base, layout, _ptr(sc))
    return v


def kv_cache_append(cache, dt, cache_len, new_vals, n_new, new_len=None):
    """In place on `cache` (float32 or uint16 bf16 bits); returns the status."""
    nv = _c(new_vals, np.float64)
    return lib().or_kv_cache_append(_ptr(cache), dt, cache.size, cache_len, _ptr(nv),
                                    nv.size if new_len is None else new_len, n_new)


def gqa_attention(q, k_cache, v_cache, kv_dt, n_ctx, n_qh, n_kvh, head_dim, scale=None,
                  block_table=None, max_blocks=None, block_tokens=None, seq=0):
    q = _c(q, np.float64)
    k_cache = _stored(k_cache, kv_dt)
    v_cache = _stored(v_cache, kv_dt)
    if block_tokens is None:
        block_tokens = 1
        max_blocks = k_cache.size // (n_kvh * head_dim)
    bt = None if block_table is None else _c(block_table, np.int32)
    out = np.empty(n_qh * head_dim, dtype=np.float64)
    if scale is None:
        scale = 1.0 / np.sqrt(head_dim)
    lib().or_gqa_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), kv_dt, _ptr(bt), max_blocks,
                           block_tokens, seq, n_ctx, n_qh, n_kvh, head_dim, scale, _ptr(out))
    return out


def argmax(logits):
    l = _c(logits, np.float32)
    m = np.zeros(1, dtype=np.float32)
    i = lib().or_argmax(_ptr(l), l.size, _ptr(m))
    return int(i), float(m[0])


def sample(logits, temperature, top_k, top_p, u):
    """Returns (token id, margin); the id is -1 for a parameter out of domain."""
    l = _c(logits, np.float32)
    margin = np.zeros(1, dtype=np.float64)
    t = lib().or_sample(_ptr(l), l.size, float(temperature), int(top_k), float(top_p), float(u),
                        _ptr(margin))
    return int(t), float(margin[0])


# ---------------------------------------------------------------- model
class Model:
    """Oracle model: weights in the shared storage layout (see oracle.c), its
    own host KV caches, and one ``step`` per decode step.

    ``cfg`` keys: vocab, d, n_layer, n_qh, n_kvh, head_dim, ff, rope_base,
    rope_layout, tied, w_dtype, kv_dtype, eps, optional rope_scaling (see
    ``rope_scaling_vector``); cache geometry
    block_tokens / max_blocks (a sequence's capacity is their product) and
    n_seqs; optional block_table (int32 [n_seqs, max_blocks]) for a paged pool
    with ``n_blocks`` physical blocks.

    ``weights`` keys: emb, out (absent when tied), norm, and per layer lists
    n1, wqkv, wo, n2, wgu, wd — flat float32 arrays or uint16 bf16 bits;
    optional per layer lists q_norm and k_norm (float32 [head_dim]) turn on
    the QK-norm of every q and k head before RoPE.
    """

    def __init__(self, cfg, weights):
        self.cfg = dict(cfg)
        c = self.cfg
        c.setdefault("eps", 1e-5)
        c.setdefault("tied", 0)
        c.setdefault("block_tokens", 1)
        c.setdefault("n_seqs", 1)
        c.setdefault("max_blocks", c.get("capacity", 64))
        wdt = c["w_dtype"]
        keep = []

        def hold(a, dt):
            a = _stored(a, dt)
            keep.append(a)
            return a.ctypes.data

        ptrs = [hold(weights["emb"], wdt),
                hold(weights["emb"] if c["tied"] else weights["out"], wdt),
                hold(weights["norm"], DT_F32)]
        for l in range(c["n_layer"]):
            ptrs += [hold(weights["n1"][l], DT_F32), hold(weights["wqkv"][l], wdt),
                     hold(weights["wo"][l], wdt), hold(weights["n2"][l], DT_F32),
                     hold(weights["wgu"][l], wdt), hold(weights["wd"][l], wdt)]
        qk_norm = "q_norm" in weights
        if qk_norm:
            for l in range(c["n_layer"]):
                ptrs += [hold(weights["q_norm"][l], DT_F32), hold(weights["k_norm"][l], DT_F32)]
        self._keep = keep
        self._wptrs = (ctypes.c_void_p * len(ptrs))(*ptrs)
        self._iv = np.array([c["vocab"], c["d"], c["n_layer"], c["n_qh"], c["n_kvh"],
                             c["head_dim"], c["ff"], c["rope_layout"], c["tied"], wdt,
                             c["kv_dtype"], c["block_tokens"], c["max_blocks"], int(qk_norm)], dtype=np.int64)
        self._dv = np.concatenate([np.array([c["rope_base"], c["eps"]], dtype=np.float64),
                                   rope_scaling_vector(c.get("rope_scaling"))])
        bt = c.get("block_table")
        self._bt = None if bt is None else _c(bt, np.int32)
        n_blocks = c.get("n_blocks", c["n_seqs"] * c["max_blocks"])
        rows = n_blocks * c["block_tokens"]
        kvdt = np.float32 if c["kv_dtype"] == DT_F32 else np.uint16
        row = c["n_kvh"] * c["head_dim"]
        self.k = [np.zeros(rows * row, dtype=kvdt) for _ in range(c["n_layer"])]
        self.v = [np.zeros(rows * row, dtype=kvdt) for _ in range(c["n_layer"])]

    def _cache_ptrs(self, caches):
        return (ctypes.c_void_p * len(caches))(*[a.ctypes.data for a in caches])

    def step(self, token, pos, seq=0):
        """Logits (float64 [vocab]) of `token` at `pos`; appends its K/V."""
        logits = np.empty(self.cfg["vocab"], dtype=np.float64)
        rc = lib().or_decode_step(_ptr(self._iv), _ptr(self._dv), self._wptrs,
                                  self._cache_ptrs(self.k), self._cache_ptrs(self.v),
                                  _ptr(self._bt), seq, int(token), int(pos), _ptr(logits))
        if rc:
            raise ValueError("oracle decode step refused token %d at pos %d" % (token, pos))
        return logits

    def recompute(self, tokens):
        """Logits of the last of `tokens`, recomputed from scratch (fresh,
        contiguous caches; no reuse of this model's caches)."""
        c = self.cfg
        toks = _c(tokens, np.int32)
        iv = self._iv.copy()
        iv[11] = 1
        iv[12] = len(toks)
        kvdt = np.float32 if c["kv_dtype"] == DT_F32 else np.uint16
        row = c["n_kvh"] * c["head_dim"]
        ks = [np.zeros(len(toks) * row, dtype=kvdt) for _ in range(c["n_layer"])]
        vs = [np.zeros(len(toks) * row, dtype=kvdt) for _ in range(c["n_layer"])]
        logits = np.empty(c["vocab"], dtype=np.float64)
        rc = lib().or_recompute_logits(_ptr(iv), _ptr(self._dv), self._wptrs,
                                       self._cache_ptrs(ks), self._cache_ptrs(vs), _ptr(toks),
                                       len(toks), _ptr(logits))
        if rc:
            raise ValueError("oracle recompute refused")
        return logits


def top2_gap(logits):
    """Gap between the largest and second-largest logit."""
    s = np.sort(np.asarray(logits, dtype=np.float64))
    return float(s[-1] - s[-2])


def greedy_generate(model, prompt, n_new):
    """Prefill one token at a time, then n_new greedy steps; returns
    (generated ids, per-step logits)."""
    logits = None
    for pos, t in enumerate(prompt):
        logits = model.step(t, pos)
    out, all_logits = [], []
    for i in range(n_new):
        tok, _ = argmax(logits.astype(np.float32))
        out.append(tok)
        all_logits.append(logits)
        logits = model.step(tok, len(prompt) + i)
    return out, all_logits
