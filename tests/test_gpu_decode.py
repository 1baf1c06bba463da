"""Whole decode steps through the C ABI against the oracle: the tiny decoder
(ids exact, logits to 1e-4, cache contents, cache vs recompute), a Qwen3-0.6B-
shaped model at full width, the 8B shape at full size from a synthetic
prefilled context, graph replay and determinism."""
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


def toy_weights_gpu():
    st = synth.p4_to_storage(synth.p4_toy_weights(C.TOY, 0), C.TOY)
    W = {k: ([torch.from_numpy(a).cuda() for a in v] if isinstance(v, list) else torch.from_numpy(v).cuda())
         for k, v in st.items()}
    return st, W


def oracle_model(cfg, st, capacity, block_tokens=1, block_table=None, n_blocks=None):
    ocfg = dict(cfg, block_tokens=block_tokens, max_blocks=(capacity + block_tokens - 1) // block_tokens)
    if block_table is not None:
        ocfg.update(block_table=block_table, n_blocks=n_blocks)
    return O.Model(ocfg, st)


@pytest.mark.parametrize("prompt_kind", ["page", "seeded"])
def test_toy_decoder_matches_oracle_token_for_token(M, prompt_kind):
    st, W = toy_weights_gpu()
    prompt = synth.P4_PROMPT if prompt_kind == "page" else synth.toy_prompt(0)
    g = M.DecodeModel(C.TOY, W, capacity=64, block_tokens=4)
    o = oracle_model(C.TOY, st, 64)
    seq = list(prompt)
    n_new = 16
    for pos in range(len(prompt) + n_new):
        g.set_state([seq[pos]], [pos])
        g.step()
        ref = o.step(seq[pos], pos)
        got = host(g.logits[0])
        assert rel_err(got, ref) <= FP32_TOL, pos
        gid = int(g.next_ids[0])
        assert gid == O.argmax(ref.astype(np.float32))[0]
        if pos + 1 >= len(seq) and len(seq) < len(prompt) + n_new:
            seq.append(gid)
    if prompt_kind == "page":
        assert seq[len(prompt):len(prompt) + 3] == [30, 30, 30]  # the page's printed result
    # KV cache rows written so far match the oracle; the rest stayed zero
    n = len(prompt) + n_new
    for l in range(C.TOY["n_layer"]):
        kg, vg = host(g.k_cache[l]).ravel(), host(g.v_cache[l]).ravel()
        row = C.TOY["n_kvh"] * C.TOY["head_dim"]
        assert rel_err(kg[:n * row], o.k[l][:n * row]) <= FP32_TOL
        assert rel_err(vg[:n * row], o.v[l][:n * row]) <= FP32_TOL
        assert not kg[n * row:].any() and not vg[n * row:].any()
    assert g.error_word() == 0


def test_toy_cached_decode_equals_recompute_on_gpu(M):
    st, W = toy_weights_gpu()
    g = M.DecodeModel(C.TOY, W, capacity=64, block_tokens=4)
    out = g.generate_greedy(synth.P4_PROMPT, 10)
    seq = list(synth.P4_PROMPT)
    for _ in range(10):
        r = M.DecodeModel(C.TOY, W, capacity=64, block_tokens=4)  # fresh cache: no reuse
        r.prefill(seq)
        seq.append(int(r.next_ids[0]))
    assert out == seq[len(synth.P4_PROMPT):]


def test_toy_graph_replay_equals_eager_steps(M):
    _, W = toy_weights_gpu()
    a = M.DecodeModel(C.TOY, W, capacity=64, block_tokens=4)
    b = M.DecodeModel(C.TOY, W, capacity=64, block_tokens=4)
    a.prefill(synth.P4_PROMPT)
    b.prefill(synth.P4_PROMPT)
    p = len(synth.P4_PROMPT)
    for m in (a, b):
        m.set_state([int(m.next_ids[0])], [p])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        replay = a.graph(advance=True, write_logits=True, stream=s)
        ids_a = []
        for _ in range(12):
            replay(s)
            s.synchronize()
            ids_a.append(int(a.next_ids[0]))
    ids_b = []
    for _ in range(12):
        b.step(advance=True)
        ids_b.append(int(b.next_ids[0]))
    assert ids_a == ids_b
    assert int(a.pos[0]) == int(b.pos[0]) == p + 12
    assert torch.equal(a.logits, b.logits)


def small_bf16(cfg, n_layer):
    c = dict(cfg, n_layer=n_layer)
    return c


def _teacher_forced(M, cfg, W, st, prompt, n_new, capacity, block_tokens=16, tol=BF16_TOL):
    g = M.DecodeModel(cfg, W, capacity=capacity, block_tokens=block_tokens)
    o = oracle_model(cfg, st, g.capacity)
    seq = list(prompt)
    compared = 0
    for pos in range(len(prompt) + n_new):
        g.set_state([seq[pos]], [pos])
        g.step()
        ref = o.step(seq[pos], pos)
        got = host(g.logits[0])
        assert rel_err(got, ref) <= tol, pos
        gap = top2_gap(ref)
        want = O.argmax(ref.astype(np.float32))[0]
        if gap > TIE_GAP:
            assert int(g.next_ids[0]) == want, (pos, gap)
            compared += 1
        if pos + 1 >= len(seq) and len(seq) < len(prompt) + n_new:
            seq.append(want)  # the GPU follows the oracle's token
    assert g.error_word() == 0
    return compared


def test_qwen_shape_two_layers_full_width(M):
    cfg = small_bf16(C.QWEN3_0_6B, 2)
    W = synth.model_weights(cfg, seed=0, device="cuda")
    st = synth.weights_to_numpy(W)
    prompt = synth.prompt_ids(cfg, 37, seed=0)
    compared = _teacher_forced(M, cfg, W, st, prompt, 8, capacity=64)
    assert compared >= 30


def test_llama8b_shape_two_layers_full_width(M):
    cfg = small_bf16(C.LLAMA3_8B, 2)
    W = synth.model_weights(cfg, seed=1, device="cuda")
    st = synth.weights_to_numpy(W)
    prompt = synth.prompt_ids(cfg, 21, seed=1)
    compared = _teacher_forced(M, cfg, W, st, prompt, 6, capacity=48)
    assert compared >= 20


@pytest.mark.slow
def test_llama8b_full_size_step_from_synthetic_context(M):
    """All 32 layers and the full vocabulary, in the launch configuration the
    benchmark times (captured graph, advance on device), one step at position
    1024 over a synthetic prefilled context of 1024 positions."""
    cfg = C.LLAMA3_8B
    n_ctx = 1024
    W = synth.model_weights(cfg, seed=0, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=n_ctx + 256, block_tokens=16)
    ks, vs = synth.synthetic_kv(cfg, n_ctx, seed=3, device="cuda")
    for l in range(cfg["n_layer"]):
        g.k_cache[l][:n_ctx].copy_(ks[l])
        g.v_cache[l][:n_ctx].copy_(vs[l])
    tok = synth.prompt_ids(cfg, 1, seed=5)[0]
    g.set_state([tok], [n_ctx])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        replay = g.graph(advance=True, write_logits=True, stream=s)
        replay(s)
    s.synchronize()
    got = host(g.logits[0])
    gid = int(g.next_ids[0])
    assert int(g.pos[0]) == n_ctx + 1 and int(g.tokens[0]) == gid
    # the oracle, from the same weights and the same synthetic context
    st = synth.weights_to_numpy(W)
    del W
    o = oracle_model(cfg, st, g.capacity)
    for l in range(cfg["n_layer"]):
        o.k[l][:ks[l].numel()] = host(ks[l]).ravel()
        o.v[l][:vs[l].numel()] = host(vs[l]).ravel()
    ref = o.step(tok, n_ctx)
    assert rel_err(got, ref) <= BF16_TOL
    if top2_gap(ref) > TIE_GAP:
        assert gid == O.argmax(ref.astype(np.float32))[0]
    # the K/V written at position n_ctx
    row = cfg["n_kvh"] * cfg["head_dim"]
    for l in (0, cfg["n_layer"] - 1):
        kg = O.bf16_bits_to_f64(host(g.k_cache[l][n_ctx]))
        ko = O.bf16_bits_to_f64(o.k[l][n_ctx * row:(n_ctx + 1) * row])
        assert rel_err(kg, ko) <= BF16_TOL
    assert g.error_word() == 0


def test_decode_is_bit_stable(M):
    cfg = small_bf16(C.LLAMA3_8B, 2)
    W = synth.model_weights(cfg, seed=2, device="cuda")
    outs = []
    for _ in range(2):
        g = M.DecodeModel(cfg, W, capacity=32, block_tokens=16)
        g.prefill([1, 2, 3, 4, 5])
        outs.append(g.logits[0].clone())
    assert torch.equal(outs[0], outs[1])


def test_sampled_decode_matches_oracle_sampler(M):
    cfg = small_bf16(C.QWEN3_0_6B, 1)
    W = synth.model_weights(cfg, seed=4, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=32, block_tokens=16)
    u = synth.uniform_draws(6, seed=0)
    toks = synth.prompt_ids(cfg, 6, seed=4)
    o = oracle_model(cfg, synth.weights_to_numpy(W), g.capacity)
    compared = 0
    for pos, t in enumerate(toks):
        g.set_state([t], [pos])
        g.u[0] = u[pos]
        g.step(sampling=(0.8, 50, 0.95))
        ref = o.step(t, pos)
        assert rel_err(host(g.logits[0]), ref) <= BF16_TOL
        # the oracle sampler on the oracle's own logits; draws within 1e-3 of
        # a CDF boundary may go either way given the logits' rounding
        want, margin = O.sample(ref.astype(np.float32), 0.8, 50, 0.95, float(u[pos]))
        if margin >= 1e-3:
            assert int(g.next_ids[0]) == want
            compared += 1
    assert compared >= 3


def test_sampled_decode_over_the_whole_vocabulary(M):
    """Top-p sampling with no top-k cut over the tied 151,936-entry Qwen
    vocabulary, through the model's step: the step's pick equals the
    standalone sampler's on the step's own logits and the same draw (the
    sampler's parity with the oracle is checked op by op)."""
    from autoregressive_decode_step_gb300 import abi
    cfg = small_bf16(C.QWEN3_0_6B, 1)
    W = synth.model_weights(cfg, seed=7, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=32, block_tokens=16)
    u = synth.uniform_draws(5, seed=8)
    ids = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = abi.workspace(abi.ds_sample_workspace_bytes(1, cfg["vocab"]))
    for pos, t in enumerate(synth.prompt_ids(cfg, 5, seed=9)):
        g.set_state([t], [pos])
        g.u[0] = u[pos]
        g.step(sampling=(0.9, 0, 0.9))
        abi.ds_sample(g.logits[0], 1, cfg["vocab"], 0.9, 0, 0.9, g.u[:1], ids, ws)
        assert int(g.next_ids[0]) == int(ids[0])
    assert g.error_word() == 0


def test_multi_step_launch_equals_single_steps(M):
    """ds_decode_steps (n greedy steps in one launch, the pick handed to the
    next step on the device) against n separate single steps: same ids, same
    final state, same K/V written, bit for bit."""
    cfg = small_bf16(C.LLAMA3_8B, 2)
    W = synth.model_weights(cfg, seed=6, device="cuda")
    prompt = synth.prompt_ids(cfg, 9, seed=6)
    a = M.DecodeModel(cfg, W, capacity=48, block_tokens=16)
    b = M.DecodeModel(cfg, W, capacity=48, block_tokens=16)
    for g in (a, b):
        g.prefill(prompt)
        g.set_state([int(g.next_ids[0])], [len(prompt)])
    ids = torch.zeros(12, dtype=torch.int32, device="cuda")
    a.steps(12, ids_out=ids)
    want = []
    for _ in range(12):
        b.step(advance=True)
        want.append(int(b.next_ids[0]))
    assert host(ids).tolist() == want
    assert int(a.pos[0]) == int(b.pos[0]) == len(prompt) + 12
    assert int(a.tokens[0]) == int(b.tokens[0]) == want[-1]
    for l in range(cfg["n_layer"]):
        assert torch.equal(a.k_cache[l], b.k_cache[l]) and torch.equal(a.v_cache[l], b.v_cache[l])
    assert a.error_word() == 0 and b.error_word() == 0


def test_multi_step_launch_reproduces_the_page_on_the_tiny_decoder(M):
    st, W = toy_weights_gpu()
    g = M.DecodeModel(C.TOY, W, capacity=C.TOY["max_seq"], block_tokens=4)
    prompt = [3, 14, 15, 9, 2, 6]
    g.prefill(prompt)
    first = int(g.next_ids[0])
    g.set_state([first], [len(prompt)])
    ids = torch.zeros(9, dtype=torch.int32, device="cuda")
    g.steps(9, ids_out=ids)
    o = oracle_model(C.TOY, st, g.capacity)
    out, _ = O.greedy_generate(o, prompt, 10)
    assert [first] + host(ids).tolist() == out
    assert out[:3] == [30, 30, 30]


@pytest.mark.slow
def test_qwen_full_size_step_from_synthetic_context(M):
    """The Qwen3-0.6B shape at full depth and vocabulary (28 layers, tied
    151,936 x 1024 head, fp32 K/V), in the captured-graph configuration, one
    step at position 512 over a synthetic 512-position context."""
    cfg = C.QWEN3_0_6B
    n_ctx = 512
    W = synth.model_weights(cfg, seed=0, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=n_ctx + 256, block_tokens=16)
    ks, vs = synth.synthetic_kv(cfg, n_ctx, seed=3, device="cuda")
    for l in range(cfg["n_layer"]):
        g.k_cache[l][:n_ctx].copy_(ks[l])
        g.v_cache[l][:n_ctx].copy_(vs[l])
    tok = synth.prompt_ids(cfg, 1, seed=5)[0]
    g.set_state([tok], [n_ctx])
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        replay = g.graph(advance=True, write_logits=True, stream=s)
        replay(s)
    s.synchronize()
    got = host(g.logits[0])
    gid = int(g.next_ids[0])
    st = synth.weights_to_numpy(W)
    del W
    o = oracle_model(cfg, st, g.capacity)
    for l in range(cfg["n_layer"]):
        o.k[l][:ks[l].numel()] = host(ks[l]).ravel()
        o.v[l][:vs[l].numel()] = host(vs[l]).ravel()
    ref = o.step(tok, n_ctx)
    assert rel_err(got, ref) <= BF16_TOL
    if top2_gap(ref) > TIE_GAP:
        assert gid == O.argmax(ref.astype(np.float32))[0]
    assert g.error_word() == 0


@pytest.mark.parametrize("shape,n_ctx", [("llama", 4096), ("qwen", 2048)])
def test_long_context_attention_streamed_through_the_ring(M, shape, n_ctx):
    """Contexts long enough that every attention split fills a K/V stage, so
    the persistent kernel streams the cached K/V through its shared-memory
    ring (bf16 K/V for the 8B widths, fp32 for the Qwen widths): two steps
    from a synthetic prefilled context against the oracle."""
    cfg = small_bf16(C.LLAMA3_8B if shape == "llama" else C.QWEN3_0_6B, 2)
    W = synth.model_weights(cfg, seed=9, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=n_ctx + 16, block_tokens=16)
    ks, vs = synth.synthetic_kv(cfg, n_ctx, seed=10, device="cuda")
    for l in range(cfg["n_layer"]):
        g.k_cache[l][:n_ctx].copy_(ks[l])
        g.v_cache[l][:n_ctx].copy_(vs[l])
    o = oracle_model(cfg, synth.weights_to_numpy(W), g.capacity)
    for l in range(cfg["n_layer"]):
        o.k[l][:ks[l].numel()] = host(ks[l]).ravel()
        o.v[l][:vs[l].numel()] = host(vs[l]).ravel()
    toks = synth.prompt_ids(cfg, 2, seed=11)
    for i, t in enumerate(toks):
        g.set_state([t], [n_ctx + i])
        g.step()
        ref = o.step(t, n_ctx + i)
        assert rel_err(host(g.logits[0]), ref) <= BF16_TOL, i
        if top2_gap(ref) > TIE_GAP:
            assert int(g.next_ids[0]) == O.argmax(ref.astype(np.float32))[0]
    assert g.error_word() == 0


LLAMA31_SCALING = {"factor": 8.0, "low_freq_factor": 1.0, "high_freq_factor": 4.0,
                   "original_max_position": 8192.0}


def test_llama31_rope_scaling_past_the_original_context(M):
    """Long-context RoPE scaling as Llama 3.1 checkpoints define it, in the
    model's RoPE table: 8B widths, 2 layers, two steps at positions 9000 and
    9001 from a synthetic prefilled context.  Logits and the K rows written
    match the scaled oracle; the K rows are far from the unscaled rotation."""
    cfg = dict(small_bf16(C.LLAMA3_8B, 2), rope_scaling=LLAMA31_SCALING)
    n_ctx = 9000
    W = synth.model_weights(cfg, seed=31, device="cuda")
    g = M.DecodeModel(cfg, W, capacity=n_ctx + 16, block_tokens=16)
    ks, vs = synth.synthetic_kv(cfg, n_ctx, seed=32, device="cuda")
    for l in range(cfg["n_layer"]):
        g.k_cache[l][:n_ctx].copy_(ks[l])
        g.v_cache[l][:n_ctx].copy_(vs[l])
    st = synth.weights_to_numpy(W)
    o = oracle_model(cfg, st, g.capacity)
    plain = oracle_model(dict(cfg, rope_scaling=None), st, g.capacity)
    for oo in (o, plain):
        for l in range(cfg["n_layer"]):
            oo.k[l][:ks[l].numel()] = host(ks[l]).ravel()
            oo.v[l][:vs[l].numel()] = host(vs[l]).ravel()
    row = cfg["n_kvh"] * cfg["head_dim"]
    for i, t in enumerate(synth.prompt_ids(cfg, 2, seed=33)):
        pos = n_ctx + i
        g.set_state([t], [pos])
        g.step()
        ref = o.step(t, pos)
        plain.step(t, pos)
        assert rel_err(host(g.logits[0]), ref) <= BF16_TOL, i
        if top2_gap(ref) > TIE_GAP:
            assert int(g.next_ids[0]) == O.argmax(ref.astype(np.float32))[0]
        kg = O.bf16_bits_to_f64(host(g.k_cache[0][pos]))
        assert rel_err(kg, O.bf16_bits_to_f64(o.k[0][pos * row:(pos + 1) * row])) <= BF16_TOL
        assert rel_err(kg, O.bf16_bits_to_f64(plain.k[0][pos * row:(pos + 1) * row])) > 0.1
    assert g.error_word() == 0
