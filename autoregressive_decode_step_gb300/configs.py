"""Workload descriptions: model shapes, dtypes and the op-level sizes.

Plain data only.  Dtype and layout codes match ``include/decode_step.h``.

Storage layout of a model's weights (the format both the CUDA library and the
tests' oracle read):

* ``emb``  [vocab, d] — token embedding; also the output head when ``tied``.
* ``out``  [vocab, d] — output head (untied models), applied untransposed.
* ``norm`` [d] fp32 — final RMSNorm weight.
* per layer: ``n1``/``n2`` [d] fp32 RMSNorm weights;
  ``wqkv`` [d, (n_qh + 2 n_kvh) head_dim] — q columns, then k, then v;
  ``wo`` [n_qh head_dim, d]; ``wgu`` [d, 2 ff] — gate columns, then up;
  ``wd`` [ff, d].  Projections are [in, out] row-major and applied as
  y = A^T x (the transposed mat-vec of the "LLM inference kernels" page).
"""

F32 = 0
BF16 = 1
ROPE_HALF_SPLIT = 0
ROPE_INTERLEAVED = 1

DTYPE_BYTES = {F32: 4, BF16: 2}

# The tiny Llama-style decoder of "The forward pass end to end" ("The code":
# Config): vocab 40, d 16, 2 layers, 4 query heads sharing 2 KV heads, head_dim
# 4, SwiGLU hidden 24, max_seq 64; Gaussian(0, 0.15) weights from seed 0,
# interleaved RoPE base 10000, fp32.
TOY = dict(name="toy-llama-d16", vocab=40, d=16, n_layer=2, n_qh=4, n_kvh=2, head_dim=4, ff=24,
           max_seq=64, rope_base=10000.0, rope_layout=ROPE_INTERLEAVED, tied=0, w_dtype=F32,
           kv_dtype=F32, eps=1e-5, weight_std=0.15)

# Qwen3-0.6B-shaped random-init decoder (tied embeddings, half-split RoPE).
QWEN3_0_6B = dict(name="qwen3-0.6b-shape", vocab=151936, d=1024, n_layer=28, n_qh=16, n_kvh=8,
                  head_dim=128, ff=3072, max_seq=768, rope_base=1e6,
                  rope_layout=ROPE_HALF_SPLIT, tied=1, w_dtype=BF16, kv_dtype=F32, eps=1e-5,
                  weight_std=0.02)

# Llama-3-8B-shaped random-init decoder, bf16 weights and bf16 KV cache.
LLAMA3_8B = dict(name="llama3-8b-shape", vocab=128256, d=4096, n_layer=32, n_qh=32, n_kvh=8,
                 head_dim=128, ff=14336, max_seq=8192 + 256, rope_base=500000.0,
                 rope_layout=ROPE_HALF_SPLIT, tied=0, w_dtype=BF16, kv_dtype=BF16, eps=1e-5,
                 weight_std=0.02)

# Batched continuous decode on the 8B shape.
BATCHED_8B = dict(model=LLAMA3_8B, n_seqs=64, ctx_lo=128, ctx_hi=4096, block_tokens=16,
                  steps=128, temperature=0.8, top_k=50, top_p=0.95)

# Op-level decode glue at the pages' measured sizes (fp32, N(0,1) inputs).
OPS = dict(gemv_shapes=[(4096, 4096), (4096, 14336)], rmsnorm_n=4096, rope_q_heads=32,
           rope_k_heads=8, rope_head_dim=128, rope_base=10000.0, rope_max_pos=8192,
           argmax_n=128256, sample_temperature=0.8, sample_top_k=50, sample_top_p=0.95)


def qkv_cols(cfg):
    return (cfg["n_qh"] + 2 * cfg["n_kvh"]) * cfg["head_dim"]


def layer_params(cfg):
    d, ff, hd = cfg["d"], cfg["ff"], cfg["head_dim"]
    return d * qkv_cols(cfg) + cfg["n_qh"] * hd * d + d * 2 * ff + ff * d


def weight_bytes_per_step(cfg):
    """Bytes of weights one decode step reads once: projections of every layer
    plus the output head (norm weights are counted too; they are tiny)."""
    wb = DTYPE_BYTES[cfg["w_dtype"]]
    total = cfg["n_layer"] * layer_params(cfg) * wb
    total += cfg["vocab"] * cfg["d"] * wb
    total += (2 * cfg["n_layer"] + 1) * cfg["d"] * 4
    return total


def kv_bytes_per_token(cfg, dtype_bytes=None):
    """K and V bytes one cached position occupies across all layers."""
    b = DTYPE_BYTES[cfg["kv_dtype"]] if dtype_bytes is None else dtype_bytes
    return 2 * cfg["n_layer"] * cfg["n_kvh"] * cfg["head_dim"] * b


def step_bytes(cfg, n_ctx):
    """Algorithmic HBM bytes of one batch-1 decode step attending over n_ctx
    positions: every weight byte once plus the K/V of every position."""
    return weight_bytes_per_step(cfg) + n_ctx * kv_bytes_per_token(cfg)
