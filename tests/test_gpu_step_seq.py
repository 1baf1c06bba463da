"""stepSeq — a prompt of one sequence run as chunks of rows on the batched
path (ds_step_seq) — through the C ABI against the oracle decoding the same
tokens one at a time ("Inside the engine", section 1: prefill is a chunk of
prompt tokens run as a batch of rows; decode is the one-token chunk of the
same step).  Both sides start from the same synthetic paged pool; after the
prompt, the K/V rows of every prompt position, the last token's logits and
the greedy pick must agree."""
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


def make_pair(M, cfg, n_seqs, cap, block_tokens, seed):
    W = synth.model_weights(cfg, seed=seed, device="cuda")
    st = synth.weights_to_numpy(W)
    mb = (cap + block_tokens - 1) // block_tokens
    n_blocks = n_seqs * mb
    table = synth.paged_block_table(n_seqs, mb, seed=seed + 1)
    g = M.DecodeModel(cfg, W, capacity=cap, block_tokens=block_tokens, block_table=table.cuda(), n_blocks=n_blocks,
                      max_seqs=n_seqs)
    o = O.Model(dict(cfg, block_tokens=block_tokens, max_blocks=mb, block_table=table.numpy(), n_blocks=n_blocks,
                     n_seqs=n_seqs), st)
    ks, vs = synth.synthetic_kv(cfg, n_blocks * block_tokens, seed=seed + 2, device="cuda")
    for l in range(cfg["n_layer"]):
        g.k_cache[l].copy_(ks[l])
        g.v_cache[l].copy_(vs[l])
        o.k[l][:] = host(ks[l]).ravel()
        o.v[l][:] = host(vs[l]).ravel()
    return g, o, table


def kv_values(a):
    """Cache row as fp64: bf16 caches come back as their bit patterns."""
    a = np.asarray(a)
    return O.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def check_prompt(g, o, table, cfg, seq, offset, prompt, block_tokens):
    """Run the prompt through ds_step_seq and through the oracle token by
    token; compare K/V rows of every prompt position, last logits, pick."""
    g.step_seq(prompt, seq=seq, offset=offset)
    torch.cuda.synchronize()
    ref = None
    for t, tok in enumerate(prompt):
        ref = o.step(int(tok), offset + t, seq=seq)
    got = host(g.logits[seq])
    assert rel_err(got, ref) <= BF16_TOL
    if top2_gap(ref) > TIE_GAP:
        assert int(host(g.next_ids[seq:seq + 1])[0]) == O.argmax(ref.astype(np.float32))[0]
    row_len = cfg["n_kvh"] * cfg["head_dim"]
    tab = table.numpy()
    for t in range(len(prompt)):
        pos = offset + t
        row = int(tab[seq][pos // block_tokens]) * block_tokens + pos % block_tokens
        for l in range(cfg["n_layer"]):
            for gc, oc in ((g.k_cache[l], o.k[l]), (g.v_cache[l], o.v[l])):
                kg = kv_values(host(gc[row]))
                ko = kv_values(oc[row * row_len:(row + 1) * row_len])
                assert rel_err(kg, ko) <= BF16_TOL, (t, l)
    assert g.error_word() == 0


def test_step_seq_tiny_shape_from_position_zero_ragged_chunks(M):
    """The tiny decoder's shape with bf16 weights and K/V, 4 rows per chunk:
    a 21-token prompt from position 0 runs as chunks of 4, 4, 4, 4, 4 and 1
    rows (the fallback attention kernel, head_dim 4)."""
    cfg = dict(C.TOY, w_dtype=C.BF16, kv_dtype=C.BF16)
    g, o, table = make_pair(M, cfg, 4, 32, block_tokens=4, seed=21)
    prompt = synth.prompt_ids(cfg, 21, seed=22)
    check_prompt(g, o, table, cfg, 2, 0, prompt, 4)


def test_step_seq_llama8b_shape_after_a_cached_context(M):
    """8B widths, 2 layers, 8 rows per chunk: a 20-token prompt appended to a
    sequence that already holds 37 cached positions (chunks of 8, 8, 4 on the
    paged tensor-core attention); then one ordinary decode step of that
    sequence continues from the prompt."""
    cfg = dict(C.LLAMA3_8B, n_layer=2)
    g, o, table = make_pair(M, cfg, 8, 64, block_tokens=16, seed=23)
    prompt = synth.prompt_ids(cfg, 21, seed=24)
    check_prompt(g, o, table, cfg, 5, 37, prompt[:20], 16)
    # the next token through the decode step, rows 0..7 with row 5 the one checked
    g.set_state([int(prompt[20])] * 8, [57] * 8)
    g.step(n_seqs=8)
    ref = o.step(int(prompt[20]), 57, seq=5)
    assert rel_err(host(g.logits[5]), ref) <= BF16_TOL


def test_step_seq_refusals(M):
    cfg = dict(C.TOY, w_dtype=C.BF16, kv_dtype=C.BF16)
    g, _, _ = make_pair(M, cfg, 4, 16, block_tokens=4, seed=25)
    with pytest.raises(M.abi.DecodeStepError) as e:
        g.step_seq([1] * 17, seq=0, offset=0)  # past the 16 positions of the cache
    assert e.value.code == M.abi.DS_CACHE_CAPACITY_EXCEEDED
    with pytest.raises(M.abi.DecodeStepError) as e:
        g.step_seq([1, 2], seq=4, offset=0)  # no such sequence
    assert e.value.code == M.abi.DS_BAD_ARGUMENT
    with pytest.raises(M.abi.DecodeStepError) as e:
        g.step_seq([], seq=0, offset=0)
    assert e.value.code == M.abi.DS_EMPTY_DIMENSION


def test_step_seq_full_chunks_of_256_rows(M):
    """Qwen3-0.6B widths (1 layer, vocab cut to 4,096), 256 rows per chunk —
    the largest batch the tensor-core projections take: a 300-token prompt
    from position 0 runs as chunks of 256 and 44 rows."""
    cfg = dict(C.QWEN3_0_6B, n_layer=1, vocab=4096)
    g, o, table = make_pair(M, cfg, 256, 320, block_tokens=16, seed=26)
    prompt = synth.prompt_ids(cfg, 300, seed=27)
    check_prompt(g, o, table, cfg, 7, 0, prompt, 16)
