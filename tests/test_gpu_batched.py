"""The batched decode step — projections on the tensor cores, K/V in a paged
pool, one token per sequence — through the C ABI against the oracle's decode
step, sequence by sequence.  Both sides receive the same synthetic prefilled
pool and the same (teacher-forced) tokens."""
import numpy as np
import pytest
import torch

import oracle as O
from autoregressive_decode_step_gb300 import configs as C
from autoregressive_decode_step_gb300 import synth
from tests.gpu_util import BF16_TOL, TIE_GAP, host, rel_err, top2_gap

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from autoregressive_decode_step_gb300 import model
    return model


class Pair:
    """A batched GPU model and the oracle over the same weights and the same
    synthetic paged pool."""

    def __init__(self, M, cfg, n_seqs, ctx, n_steps, block_tokens, seed):
        self.cfg, self.n, self.ctx = cfg, n_seqs, list(ctx)
        W = synth.model_weights(cfg, seed=seed, device="cuda")
        st = synth.weights_to_numpy(W)
        cap = max(ctx) + n_steps + 1
        mb = (cap + block_tokens - 1) // block_tokens
        n_blocks = n_seqs * mb
        table = synth.paged_block_table(n_seqs, mb, seed=seed + 1)
        self.g = M.DecodeModel(cfg, W, capacity=cap, block_tokens=block_tokens, block_table=table.cuda(),
                               n_blocks=n_blocks, max_seqs=n_seqs)
        self.o = O.Model(dict(cfg, block_tokens=block_tokens, max_blocks=mb, block_table=table.numpy(),
                              n_blocks=n_blocks, n_seqs=n_seqs), st)
        ks, vs = synth.synthetic_kv(cfg, n_blocks * block_tokens, seed=seed + 2, device="cuda")
        for l in range(cfg["n_layer"]):
            self.g.k_cache[l].copy_(ks[l])
            self.g.v_cache[l].copy_(vs[l])
            self.o.k[l][:] = host(ks[l]).ravel()
            self.o.v[l][:] = host(vs[l]).ravel()
        del W, ks, vs
        self.t = 0

    def step(self, tokens, sampling=None, u=None):
        """One batched step at positions ctx[s] + t; returns (gpu logits,
        oracle logits) as [n, vocab] arrays."""
        pos = [c + self.t for c in self.ctx]
        self.g.set_state(tokens, pos)
        if u is not None:
            self.g.u[:self.n].copy_(torch.as_tensor(u))
        self.g.step(n_seqs=self.n, sampling=sampling)
        got = host(self.g.logits[:self.n])
        ref = np.stack([self.o.step(tokens[s], pos[s], seq=s) for s in range(self.n)])
        self.t += 1
        return got, ref


def check_logits_and_ids(p, got, ref):
    worst = 0.0
    compared = 0
    ids = host(p.g.next_ids[:p.n])
    for s in range(p.n):
        e = rel_err(got[s], ref[s])
        worst = max(worst, e)
        assert e <= BF16_TOL, (s, e)
        if top2_gap(ref[s]) > TIE_GAP:
            assert int(ids[s]) == O.argmax(ref[s].astype(np.float32))[0], s
            compared += 1
    return worst, compared


def test_batched_tiny_shape_all_sequences(M):
    """The tiny decoder's shape with bf16 weights and K/V, 64 sequences at
    contexts 1..60 in a paged pool of 4-position blocks, 3 steps."""
    cfg = dict(C.TOY, w_dtype=C.BF16, kv_dtype=C.BF16)
    ctx = synth.context_lengths(64, 1, 60, seed=3)
    p = Pair(M, cfg, 64, ctx, 3, block_tokens=4, seed=5)
    toks = synth.prompt_ids(cfg, 64 * 3, seed=6)
    compared = 0
    for t in range(3):
        got, ref = p.step(toks[64 * t:64 * (t + 1)])
        _, c = check_logits_and_ids(p, got, ref)
        compared += c
    assert compared >= 150
    assert p.g.error_word() == 0


def test_batched_llama8b_shape_two_layers_paged(M):
    """8B widths (q|k|v 4096 x 6144, gate|up 4096 x 28672, down 14336 x 4096,
    head 128,256 x 4096), 2 layers, 16 sequences at contexts 1..300 in a
    paged pool of 16-position blocks, 2 steps; K/V written at each position
    checked against the oracle's cache."""
    cfg = dict(C.LLAMA3_8B, n_layer=2)
    ctx = synth.context_lengths(16, 1, 300, seed=7)
    p = Pair(M, cfg, 16, ctx, 2, block_tokens=16, seed=8)
    toks = synth.prompt_ids(cfg, 32, seed=9)
    for t in range(2):
        got, ref = p.step(toks[16 * t:16 * (t + 1)])
        worst, compared = check_logits_and_ids(p, got, ref)
        assert compared >= 10
    # the K/V rows this step wrote, sequence 3, both layers
    row_len = cfg["n_kvh"] * cfg["head_dim"]
    table = host(p.g.block_table)
    for s in (0, 3, 15):
        pos = ctx[s] + 1
        row = int(table[s][pos // 16]) * 16 + pos % 16
        for l in range(2):
            kg = O.bf16_bits_to_f64(host(p.g.k_cache[l][row]))
            ko = O.bf16_bits_to_f64(p.o.k[l][row * row_len:(row + 1) * row_len])
            assert rel_err(kg, ko) <= BF16_TOL
    assert p.g.error_word() == 0


@pytest.mark.parametrize("head_dim,layout,kv", [(64, C.ROPE_INTERLEAVED, C.BF16), (32, C.ROPE_HALF_SPLIT, C.BF16),
                                                (128, C.ROPE_INTERLEAVED, C.F32), (8, C.ROPE_HALF_SPLIT, C.BF16)])
def test_batched_rope_layouts_and_head_sizes(M, head_dim, layout, kv):
    """The q|k|v epilogue's cases: runs of 32 features inside one head
    (interleaved pairs at head_dim 64), runs across the two halves of a head
    (half-split at 32), an fp32 cache (item by item) and heads narrower than
    a run (8); 24 sequences at contexts 1..200, 2 steps, and the K/V rows
    each step wrote."""
    n_qh = 512 // head_dim
    cfg = dict(C.LLAMA3_8B, n_layer=2, vocab=3000, d=512, n_qh=n_qh, n_kvh=max(1, n_qh // 4), head_dim=head_dim,
               ff=768, rope_layout=layout, kv_dtype=kv)
    ctx = synth.context_lengths(24, 1, 200, seed=31)
    p = Pair(M, cfg, 24, ctx, 2, block_tokens=16, seed=32)
    toks = synth.prompt_ids(cfg, 48, seed=33)
    for t in range(2):
        got, ref = p.step(toks[24 * t:24 * (t + 1)])
        _, compared = check_logits_and_ids(p, got, ref)
        assert compared >= 18
    row_len = cfg["n_kvh"] * cfg["head_dim"]
    table = host(p.g.block_table)
    for s in (0, 11, 23):
        pos = ctx[s] + 1
        row = int(table[s][pos // 16]) * 16 + pos % 16
        for l in range(2):
            if kv == C.BF16:
                kg = O.bf16_bits_to_f64(host(p.g.k_cache[l][row]))
                vg = O.bf16_bits_to_f64(host(p.g.v_cache[l][row]))
            else:
                kg = host(p.g.k_cache[l][row]).astype(np.float64)
                vg = host(p.g.v_cache[l][row]).astype(np.float64)
            ko = p.o.k[l][row * row_len:(row + 1) * row_len]
            vo = p.o.v[l][row * row_len:(row + 1) * row_len]
            if kv == C.BF16:
                ko, vo = O.bf16_bits_to_f64(ko), O.bf16_bits_to_f64(vo)
            assert rel_err(kg, ko) <= BF16_TOL and rel_err(vg, vo) <= BF16_TOL
    assert p.g.error_word() == 0


def test_batched_qwen_shape_per_row_sampling(M):
    """Tied Qwen3-0.6B widths, 1 layer, 8 sequences, per-row sampling at
    temperature 0.8 / top_k 50 / top_p 0.95 with one seeded draw per row: the
    GPU's id equals the oracle sampler's on the oracle's logits wherever the
    draw is not within 1e-3 of a CDF boundary."""
    cfg = dict(C.QWEN3_0_6B, n_layer=1)
    ctx = synth.context_lengths(8, 1, 100, seed=10)
    p = Pair(M, cfg, 8, ctx, 2, block_tokens=16, seed=11)
    toks = synth.prompt_ids(cfg, 16, seed=12)
    u = synth.uniform_draws(16, seed=13)
    compared = 0
    for t in range(2):
        uu = u[8 * t:8 * (t + 1)]
        got, ref = p.step(toks[8 * t:8 * (t + 1)], sampling=(0.8, 50, 0.95), u=uu)
        ids = host(p.g.next_ids[:8])
        for s in range(8):
            assert rel_err(got[s], ref[s]) <= BF16_TOL
            want, margin = O.sample(ref[s].astype(np.float32), 0.8, 50, 0.95, float(uu[s]))
            if margin >= 1e-3:
                assert int(ids[s]) == want, s
                compared += 1
    assert compared >= 8


def test_batched_graph_replay_equals_eager_and_is_bit_stable(M):
    cfg = dict(C.LLAMA3_8B, n_layer=1, vocab=4096)
    ctx = synth.context_lengths(32, 1, 64, seed=14)
    runs = []
    for mode in ("eager", "graph", "eager"):
        p = Pair(M, cfg, 32, ctx, 4, block_tokens=16, seed=15)
        p.g.set_state(synth.prompt_ids(cfg, 32, seed=16), ctx)
        ids = []
        if mode == "graph":
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                replay = p.g.graph(n_seqs=32, advance=True, write_logits=True, stream=s)
                for _ in range(4):
                    replay(s)
                    s.synchronize()
                    ids.append(host(p.g.next_ids[:32]).copy())
        else:
            for _ in range(4):
                p.g.step(n_seqs=32, advance=True)
                ids.append(host(p.g.next_ids[:32]).copy())
        assert host(p.g.pos[:32]).tolist() == [c + 4 for c in ctx]
        runs.append((np.stack(ids), host(p.g.logits[:32]).copy()))
    for r in runs[1:]:
        np.testing.assert_array_equal(r[0], runs[0][0])
        np.testing.assert_array_equal(r[1], runs[0][1])


@pytest.mark.slow
def test_batched_full_size_in_the_benchmark_configuration(M):
    """The benchmark's batched workload at full size — 32 layers, 64 sequences
    at contexts uniform in [128, 4096] in a scattered pool of 16-position
    blocks, a captured graph with per-row sampling and the state advanced on
    the device — one step checked against the oracle on three sampled
    sequences (the oracle recomputes one sequence at a time)."""
    cfg = C.LLAMA3_8B
    n = 64
    ctx = synth.context_lengths(n, 128, 4096, seed=0)
    need = [(c + 2 + 15) // 16 for c in ctx]
    mb = max(need)
    n_blocks = sum(need)
    perm = synth.paged_block_table(1, n_blocks, seed=1).view(-1)
    table = torch.zeros(n, mb, dtype=torch.int32)
    at = 0
    for s, k in enumerate(need):
        table[s, :k] = perm[at:at + k]
        at += k
    W = synth.model_weights(cfg, seed=0, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=mb * 16, block_tokens=16, block_table=table.cuda(), n_blocks=n_blocks,
                      max_seqs=n)
    ks, vs = synth.synthetic_kv(cfg, n_blocks * 16, seed=2, device="cuda")
    for l in range(cfg["n_layer"]):
        g.k_cache[l].copy_(ks[l])
        g.v_cache[l].copy_(vs[l])
    toks = synth.prompt_ids(cfg, n, seed=3)
    u = synth.uniform_draws(n, seed=4)
    g.set_state(toks, ctx)
    g.u[:n].copy_(u)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        replay = g.graph(n_seqs=n, sampling=(0.8, 50, 0.95), advance=True, write_logits=True, stream=s)
        replay(s)
    s.synchronize()
    got = host(g.logits[:n])
    ids = host(g.next_ids[:n])
    assert host(g.pos[:n]).tolist() == [c + 1 for c in ctx]
    assert np.isfinite(got).all()
    st = synth.weights_to_numpy(W)
    del W
    o = O.Model(dict(cfg, block_tokens=16, max_blocks=mb, block_table=table.numpy(), n_blocks=n_blocks, n_seqs=n), st)
    for l in range(cfg["n_layer"]):
        o.k[l][:] = host(ks[l]).ravel()
        o.v[l][:] = host(vs[l]).ravel()
    del ks, vs
    for sq in (0, 31, 63):
        ref = o.step(toks[sq], ctx[sq], seq=sq)
        assert rel_err(got[sq], ref) <= BF16_TOL, sq
        want, margin = O.sample(ref.astype(np.float32), 0.8, 50, 0.95, float(u[sq]))
        if margin >= 1e-3:
            assert int(ids[sq]) == want, sq
    assert g.error_word() == 0
