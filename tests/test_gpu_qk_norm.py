"""QK-norm (every q and k head RMS-normalised with its layer's q_norm / k_norm
weight before RoPE, as Qwen3 checkpoints define it) on every path of the
decode step, through the C ABI against the oracle: the persistent batch-1
kernel, the per-kernel launch sequence, the batched tensor-core step and
prompt chunks (ds_step_seq)."""
import numpy as np
import pytest
import torch

import oracle as O
from autoregressive_decode_step_gb300 import configs as C
from autoregressive_decode_step_gb300 import synth
from tests.gpu_util import BF16_TOL, FP32_TOL, TIE_GAP, host, rel_err, top2_gap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from autoregressive_decode_step_gb300 import model
    return model


def weights(cfg, seed):
    W = synth.model_weights(cfg, seed=seed, device="cuda")
    W.update(synth.qk_norm_weights(cfg, seed=seed + 100, device="cuda"))
    return W, synth.weights_to_numpy(W)


def teacher_forced(M, cfg, W, st, prompt, n_new, capacity, tol, block_tokens=16):
    g = M.DecodeModel(cfg, W, capacity=capacity, block_tokens=block_tokens)
    o = O.Model(dict(cfg, block_tokens=block_tokens, max_blocks=(g.capacity + block_tokens - 1) // block_tokens),
                st)
    seq = list(prompt)
    compared = 0
    for pos in range(len(prompt) + n_new):
        g.set_state([seq[pos]], [pos])
        g.step()
        ref = o.step(seq[pos], pos)
        assert rel_err(host(g.logits[0]), ref) <= tol, pos
        want = O.argmax(ref.astype(np.float32))[0]
        if top2_gap(ref) > TIE_GAP:
            assert int(g.next_ids[0]) == want, pos
            compared += 1
        if pos + 1 >= len(seq) and len(seq) < len(prompt) + n_new:
            seq.append(want)
    # every K row written holds the normalised, rotated k
    n = len(prompt) + n_new
    row = cfg["n_kvh"] * cfg["head_dim"]
    for l in range(cfg["n_layer"]):
        kg = host(g.k_cache[l]).ravel()[:n * row]
        ko = o.k[l][:n * row]
        if kg.dtype == np.uint16:
            kg, ko = O.bf16_bits_to_f64(kg), O.bf16_bits_to_f64(ko)
        assert rel_err(kg, ko) <= tol
    assert g.error_word() == 0
    return compared


def test_batch1_step_kernel_qwen_width(M):
    """The persistent step kernel at Qwen3-0.6B widths (2 layers), bf16
    weights, fp32 K/V."""
    cfg = dict(C.QWEN3_0_6B, n_layer=2)
    W, st = weights(cfg, 0)
    prompt = synth.prompt_ids(cfg, 21, seed=0)
    assert teacher_forced(M, cfg, W, st, prompt, 6, capacity=64, tol=BF16_TOL) >= 20


@pytest.mark.parametrize("head_dim,layout", [(64, C.ROPE_HALF_SPLIT), (16, C.ROPE_INTERLEAVED)])
def test_batch1_step_kernel_narrow_heads(M, head_dim, layout):
    """Heads narrower than a warp (16) and half a band (64): the per-head
    square sums take their lane-group and warp-group forms."""
    cfg = dict(C.QWEN3_0_6B, n_layer=2, vocab=4096, d=512, head_dim=head_dim, n_qh=8, n_kvh=4, ff=768,
               rope_layout=layout, kv_dtype=C.BF16)
    W, st = weights(cfg, 1)
    prompt = synth.prompt_ids(cfg, 12, seed=1)
    teacher_forced(M, cfg, W, st, prompt, 6, capacity=32, tol=BF16_TOL)


def test_per_kernel_path(M):
    """head_dim 256 takes the per-kernel launch sequence (the standalone
    transposed GEMV's q|k|v epilogue); bf16 weights, fp32 K/V."""
    cfg = dict(name="wide-head", vocab=2000, d=512, n_layer=2, n_qh=4, n_kvh=2, head_dim=256, ff=1024,
               max_seq=64, rope_base=10000.0, rope_layout=C.ROPE_HALF_SPLIT, tied=0, w_dtype=C.BF16,
               kv_dtype=C.F32, eps=1e-5, weight_std=0.02)
    W, st = weights(cfg, 2)
    prompt = synth.prompt_ids(cfg, 10, seed=2)
    teacher_forced(M, cfg, W, st, prompt, 6, capacity=32, tol=BF16_TOL)


def test_toy_fp32_tolerance(M):
    """The tiny decoder's shape (head_dim 4, fp32 throughout) at the fp32
    tolerance."""
    cfg = dict(C.TOY, weight_std=0.15)
    W, st = weights(cfg, 4)
    prompt = synth.prompt_ids(cfg, 8, seed=4)
    teacher_forced(M, cfg, W, st, prompt, 8, capacity=32, tol=FP32_TOL, block_tokens=4)


def _pool_pair(M, cfg, W, st, n_seqs, cap, block_tokens, seed):
    mb = (cap + block_tokens - 1) // block_tokens
    n_blocks = n_seqs * mb
    table = synth.paged_block_table(n_seqs, mb, seed=seed)
    g = M.DecodeModel(cfg, W, capacity=cap, block_tokens=block_tokens, block_table=table.cuda(), n_blocks=n_blocks,
                      max_seqs=n_seqs)
    o = O.Model(dict(cfg, block_tokens=block_tokens, max_blocks=mb, block_table=table.numpy(), n_blocks=n_blocks,
                     n_seqs=n_seqs), st)
    ks, vs = synth.synthetic_kv(cfg, n_blocks * block_tokens, seed=seed + 1, device="cuda")
    for l in range(cfg["n_layer"]):
        g.k_cache[l].copy_(ks[l])
        g.v_cache[l].copy_(vs[l])
        o.k[l][:] = host(ks[l]).ravel()
        o.v[l][:] = host(vs[l]).ravel()
    return g, o


def test_batched_tensor_core_step(M):
    """8 sequences at Qwen3-0.6B widths (2 layers) on the batched path: the
    tensor-core q|k|v epilogue normalises each head before RoPE."""
    cfg = dict(C.QWEN3_0_6B, n_layer=2, kv_dtype=C.BF16)
    W, st = weights(cfg, 5)
    n = 8
    ctx = synth.context_lengths(n, 4, 60, seed=5)
    g, o = _pool_pair(M, cfg, W, st, n, max(ctx) + 4, 16, 6)
    toks = synth.prompt_ids(cfg, 3 * n, seed=7)
    for t in range(3):
        tk = toks[t * n:(t + 1) * n]
        pos = [c + t for c in ctx]
        g.set_state(tk, pos)
        g.step(n_seqs=n)
        got = host(g.logits[:n])
        ids = host(g.next_ids[:n])
        for s in range(n):
            ref = o.step(tk[s], pos[s], seq=s)
            assert rel_err(got[s], ref) <= BF16_TOL, (t, s)
            if top2_gap(ref) > TIE_GAP:
                assert int(ids[s]) == O.argmax(ref.astype(np.float32))[0], (t, s)
    assert g.error_word() == 0


def test_prompt_chunks(M):
    """A 40-token prompt as chunks of 16 rows (ds_step_seq) at Qwen3-0.6B
    widths: every prompt position's K row, the last logits and the pick."""
    cfg = dict(C.QWEN3_0_6B, n_layer=2, kv_dtype=C.BF16)
    W, st = weights(cfg, 8)
    g, o = _pool_pair(M, cfg, W, st, 16, 64, 16, 9)
    prompt = synth.prompt_ids(cfg, 40, seed=10)
    g.step_seq(prompt, seq=3, offset=0)
    torch.cuda.synchronize()
    ref = None
    for t, tok in enumerate(prompt):
        ref = o.step(int(tok), t, seq=3)
    assert rel_err(host(g.logits[3]), ref) <= BF16_TOL
    if top2_gap(ref) > TIE_GAP:
        assert int(g.next_ids[3]) == O.argmax(ref.astype(np.float32))[0]
    assert g.error_word() == 0
