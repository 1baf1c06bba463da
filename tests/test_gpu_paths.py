"""Decode-step paths and configurations beyond the ones the model tests take:
the per-kernel launch sequence (a batch-1 shape the persistent step kernel
does not take), the 8B shape at an 8192-position context, and the error
word's bits for device-fed tokens and positions outside their range."""
import numpy as np
import pytest
import torch

import oracle as O
from autoregressive_decode_step_gb300 import configs as C
from autoregressive_decode_step_gb300 import synth
from tests.gpu_util import BF16_TOL, FP32_TOL, TIE_GAP, host, rel_err, top2_gap

pytestmark = pytest.mark.gpu

# A batch-1 shape with head_dim 256 (as Gemma-style models use): the
# persistent step kernel takes head_dim <= 128 only, so every step of this
# model runs the per-kernel launch sequence (five launches per layer).
WIDE_HEAD = dict(name="wide-head-bf16", vocab=3000, d=512, n_layer=2, n_qh=4, n_kvh=2, head_dim=256, ff=1024,
                 max_seq=128, rope_base=10000.0, rope_layout=C.ROPE_HALF_SPLIT, tied=0, w_dtype=C.BF16,
                 kv_dtype=C.BF16, eps=1e-5, weight_std=0.02)


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from autoregressive_decode_step_gb300 import model
    return model


def oracle_model(cfg, st, capacity, block_tokens=1):
    return O.Model(dict(cfg, block_tokens=block_tokens, max_blocks=(capacity + block_tokens - 1) // block_tokens),
                   st)


def fill_context(g, o, cfg, n_ctx, seed):
    ks, vs = synth.synthetic_kv(cfg, n_ctx, seed=seed, device="cuda")
    for l in range(cfg["n_layer"]):
        g.k_cache[l][:n_ctx].copy_(ks[l])
        g.v_cache[l][:n_ctx].copy_(vs[l])
        if o is not None:
            o.k[l][:ks[l].numel()] = host(ks[l]).ravel()
            o.v[l][:vs[l].numel()] = host(vs[l]).ravel()


@pytest.mark.parametrize("kv_dtype,layout", [(C.BF16, C.ROPE_HALF_SPLIT), (C.F32, C.ROPE_INTERLEAVED)])
def test_per_kernel_launch_sequence_matches_oracle(M, kv_dtype, layout):
    """The per-kernel step (q|k|v with the RMSNorm prologue and the RoPE +
    K/V epilogue, split attention, o + residual, gate|up + SiLU, down +
    residual, head + argmax), teacher-forced over a 12-token prompt and 8
    decoded positions: logits, ids and every K/V row written."""
    from autoregressive_decode_step_gb300 import abi
    cfg = dict(WIDE_HEAD, kv_dtype=kv_dtype, rope_layout=layout)
    W = synth.model_weights(cfg, seed=21, device="cuda")
    st = synth.weights_to_numpy(W)
    g = M.DecodeModel(cfg, W, capacity=64, block_tokens=16)
    with pytest.raises(abi.DecodeStepError) as e:  # not on the persistent kernel: the multi-step launch refuses
        g.steps(2)
    assert e.value.code == abi.DS_BAD_ARGUMENT
    o = oracle_model(cfg, st, g.capacity)
    prompt = synth.prompt_ids(cfg, 12, seed=22)
    seq = list(prompt)
    compared = 0
    for pos in range(len(prompt) + 8):
        g.set_state([seq[pos]], [pos])
        g.step()
        ref = o.step(seq[pos], pos)
        assert rel_err(host(g.logits[0]), ref) <= BF16_TOL, pos
        want = O.argmax(ref.astype(np.float32))[0]
        if top2_gap(ref) > TIE_GAP:
            assert int(g.next_ids[0]) == want, pos
            compared += 1
        if pos + 1 >= len(seq):
            seq.append(want)
    assert compared >= 12
    n = len(prompt) + 8
    row = cfg["n_kvh"] * cfg["head_dim"]
    for l in range(cfg["n_layer"]):
        kg, vg = host(g.k_cache[l][:n]).ravel(), host(g.v_cache[l][:n]).ravel()
        ko, vo = o.k[l][:n * row], o.v[l][:n * row]
        if kv_dtype == C.BF16:
            kg, vg, ko, vo = (O.bf16_bits_to_f64(a) for a in (kg, vg, ko, vo))
        assert rel_err(kg, ko) <= BF16_TOL and rel_err(vg, vo) <= BF16_TOL
    assert g.error_word() == 0


def test_per_kernel_launch_sequence_graph_replay_and_timers(M):
    """The same path captured as a graph and replayed with the token and
    position advanced on the device equals eager steps bit for bit; the
    per-kernel timers run over it."""
    cfg = WIDE_HEAD
    W = synth.model_weights(cfg, seed=23, device="cuda")
    a = M.DecodeModel(cfg, W, capacity=64, block_tokens=16)
    b = M.DecodeModel(cfg, W, capacity=64, block_tokens=16)
    prompt = synth.prompt_ids(cfg, 5, seed=24)
    for m in (a, b):
        m.prefill(prompt)
        m.set_state([int(m.next_ids[0])], [len(prompt)])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        replay = a.graph(advance=True, write_logits=True, stream=s)
        ids_a = []
        for _ in range(6):
            replay(s)
            s.synchronize()
            ids_a.append(int(a.next_ids[0]))
    ids_b = []
    for _ in range(6):
        b.step(advance=True)
        ids_b.append(int(b.next_ids[0]))
    assert ids_a == ids_b and torch.equal(a.logits, b.logits)
    for l in range(cfg["n_layer"]):
        assert torch.equal(a.k_cache[l], b.k_cache[l]) and torch.equal(a.v_cache[l], b.v_cache[l])
    for kind in ("embed", "qkv", "attention", "o_proj", "gate_up", "down", "head"):
        assert b.kernel_time_us(kind, reps=2) > 0.0
    slots = b.profile(reps=2)
    assert len(slots) == 2 + 5 * cfg["n_layer"] and all(t > 0.0 for _, t in slots)
    assert a.error_word() == 0 and b.error_word() == 0


def test_llama8b_widths_at_context_8192(M):
    """8B widths (2 layers) from a synthetic 8192-position context: three
    single steps against the oracle, and the multi-step launch (several
    greedy steps in one kernel, as the benchmark runs it) equal to single
    steps bit for bit at that context."""
    cfg = dict(C.LLAMA3_8B, n_layer=2)
    n_ctx = 8192
    W = synth.model_weights(cfg, seed=41, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=n_ctx + 32, block_tokens=16)
    o = oracle_model(cfg, synth.weights_to_numpy(W), g.capacity)
    fill_context(g, o, cfg, n_ctx, seed=42)
    for i, t in enumerate(synth.prompt_ids(cfg, 3, seed=43)):
        g.set_state([t], [n_ctx + i])
        g.step()
        ref = o.step(t, n_ctx + i)
        assert rel_err(host(g.logits[0]), ref) <= BF16_TOL, i
        if top2_gap(ref) > TIE_GAP:
            assert int(g.next_ids[0]) == O.argmax(ref.astype(np.float32))[0]
    # multi-step launch against single steps from the same state
    a = M.DecodeModel(cfg, W, capacity=n_ctx + 32, block_tokens=16)
    b = M.DecodeModel(cfg, W, capacity=n_ctx + 32, block_tokens=16)
    for m in (a, b):
        fill_context(m, None, cfg, n_ctx, seed=42)
        m.set_state([7], [n_ctx])
    ids = torch.zeros(10, dtype=torch.int32, device="cuda")
    a.steps(10, ids_out=ids)
    want = []
    for _ in range(10):
        b.step(advance=True)
        want.append(int(b.next_ids[0]))
    assert host(ids).tolist() == want
    for l in range(cfg["n_layer"]):
        assert torch.equal(a.k_cache[l], b.k_cache[l]) and torch.equal(a.v_cache[l], b.v_cache[l])
    assert g.error_word() == 0 and a.error_word() == 0 and b.error_word() == 0


@pytest.mark.slow
def test_llama8b_full_size_step_at_context_8192(M):
    """All 32 layers and the full vocabulary at position 8192 over a
    synthetic 8192-position context: one captured-graph step against the
    oracle, and the benchmark's launch (the multi-step kernel) giving the
    same pick and the same K/V row."""
    cfg = C.LLAMA3_8B
    n_ctx = 8192
    W = synth.model_weights(cfg, seed=0, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=n_ctx + 64, block_tokens=16)
    b = M.DecodeModel(cfg, W, capacity=n_ctx + 64, block_tokens=16)
    ks, vs = synth.synthetic_kv(cfg, n_ctx, seed=3, device="cuda")
    for m in (g, b):
        for l in range(cfg["n_layer"]):
            m.k_cache[l][:n_ctx].copy_(ks[l])
            m.v_cache[l][:n_ctx].copy_(vs[l])
    tok = synth.prompt_ids(cfg, 1, seed=5)[0]
    g.set_state([tok], [n_ctx])
    b.set_state([tok], [n_ctx])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        replay = g.graph(advance=True, write_logits=True, stream=s)
        replay(s)
        b.steps(1, stream=s)
    s.synchronize()
    got = host(g.logits[0])
    gid = int(g.next_ids[0])
    assert int(b.next_ids[0]) == gid and int(b.pos[0]) == int(g.pos[0]) == n_ctx + 1
    for l in range(cfg["n_layer"]):
        assert torch.equal(g.k_cache[l][n_ctx], b.k_cache[l][n_ctx])
    st = synth.weights_to_numpy(W)
    del W, b
    o = oracle_model(cfg, st, g.capacity)
    for l in range(cfg["n_layer"]):
        o.k[l][:ks[l].numel()] = host(ks[l]).ravel()
        o.v[l][:vs[l].numel()] = host(vs[l]).ravel()
    ref = o.step(tok, n_ctx)
    assert rel_err(got, ref) <= BF16_TOL
    if top2_gap(ref) > TIE_GAP:
        assert gid == O.argmax(ref.astype(np.float32))[0]
    row = cfg["n_kvh"] * cfg["head_dim"]
    for l in (0, cfg["n_layer"] - 1):
        kg = O.bf16_bits_to_f64(host(g.k_cache[l][n_ctx]))
        ko = O.bf16_bits_to_f64(o.k[l][n_ctx * row:(n_ctx + 1) * row])
        assert rel_err(kg, ko) <= BF16_TOL
    assert g.error_word() == 0


# ------------------------------------------------------------------ error word
BATCHED_SMALL = dict(C.TOY, name="toy-bf16", w_dtype=C.BF16, kv_dtype=C.BF16)


def _models(M, path):
    """A small model on one step path: the persistent step kernel, the
    per-kernel launch sequence or the batched tensor-core path."""
    if path == "persistent":
        st = synth.p4_to_storage(synth.p4_toy_weights(C.TOY, 0), C.TOY)
        w = {k: ([torch.from_numpy(a).cuda() for a in v] if isinstance(v, list) else torch.from_numpy(v).cuda())
             for k, v in st.items()}
        return C.TOY, M.DecodeModel(C.TOY, w, capacity=64, block_tokens=4), 1
    if path == "per_kernel":
        w = synth.model_weights(WIDE_HEAD, seed=25, device="cuda")
        return WIDE_HEAD, M.DecodeModel(WIDE_HEAD, w, capacity=64, block_tokens=16), 1
    w = synth.model_weights(BATCHED_SMALL, seed=26, device="cuda")
    table = synth.paged_block_table(4, 16, seed=27).cuda()
    return BATCHED_SMALL, M.DecodeModel(BATCHED_SMALL, w, capacity=64, block_tokens=4, block_table=table,
                                        n_blocks=64, max_seqs=4), 4


@pytest.mark.parametrize("path", ["persistent", "per_kernel", "batched"])
def test_device_side_token_and_position_range_flags(M, path):
    """A device-fed token outside [0, vocab) is clamped and sets
    DS_ERR_TOKEN_RANGE; a position at or past the cache's end skips the K/V
    write and sets DS_ERR_POSITION.  The step still completes with finite
    logits, and a good step afterwards reports nothing."""
    from autoregressive_decode_step_gb300 import abi
    cfg, g, n = _models(M, path)
    V = cfg["vocab"]
    toks = [3] * n
    pos = [2] * n
    # a prompt so that the cache has contents
    for p in range(2):
        g.set_state([5] * n, [p] * n)
        g.step(n_seqs=n)
    assert g.error_word() == 0
    for bad in (V + 5, -3):
        t = list(toks)
        t[n - 1] = bad
        g.set_state(t, pos)
        g.step(n_seqs=n)
        torch.cuda.synchronize()
        assert g.error_word() == abi.DS_ERR_TOKEN_RANGE, bad
        assert torch.isfinite(g.logits[:n]).all()
        ids = host(g.next_ids[:n])
        assert ((ids >= 0) & (ids < V)).all()
    before = [(k.clone(), v.clone()) for k, v in zip(g.k_cache, g.v_cache)]
    p = list(pos)
    p[0] = g.capacity  # one past the last cached position
    g.set_state(toks, p)
    g.step(n_seqs=n)
    torch.cuda.synchronize()
    assert g.error_word() == abi.DS_ERR_POSITION
    assert torch.isfinite(g.logits[:n]).all()
    if n == 1:  # the only row was the bad one: nothing may have been written
        for (k0, v0), k1, v1 in zip(before, g.k_cache, g.v_cache):
            assert torch.equal(k0, k1) and torch.equal(v0, v1)
    g.set_state(toks, pos)
    g.step(n_seqs=n)
    assert g.error_word() == 0
