"""The continuous-batching scheduler slice driving the GPU step ("Inside the
engine", section 2: admission by free blocks, prompt chunks, preemption of
the youngest request, first-in first-out resume by recompute).  Every plan
of ds_sched_plan runs on the GPU: its prompt chunks (and the chunks of a
resumed request's recomputed prefix) through ds_step_seq, its decode rows as
one batched ds_decode_step, both over the plan's block table on one shared
paged pool.  Each request's generated ids are then checked against the
oracle decoding that request alone."""
import numpy as np
import pytest
import torch

import oracle as O
from autoregressive_decode_step_gb300 import configs as C
from autoregressive_decode_step_gb300 import synth
from tests.gpu_util import TIE_GAP, top2_gap

pytestmark = pytest.mark.gpu

CFG = dict(C.QWEN3_0_6B, name="sched-test", n_layer=2, vocab=2048, d=256, n_qh=4, n_kvh=2, head_dim=64, ff=512,
           kv_dtype=C.BF16)
# (prompt length, tokens to generate) per request; a pool of 10 blocks of 16
# positions for 4 running requests forces preemptions
REQUESTS = [(30, 24), (21, 30), (40, 20), (17, 28), (33, 25), (25, 22)]
N_BLOCKS, BLOCK_TOKENS, MAX_BLOCKS, MAX_RUNNING, CHUNK = 10, 16, 8, 4, 16


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from autoregressive_decode_step_gb300 import model
    return model


def run_trace(M):
    from autoregressive_decode_step_gb300.sched import Scheduler
    W = synth.model_weights(CFG, seed=31, device="cuda")
    table_dev = torch.full((MAX_RUNNING, MAX_BLOCKS), -1, dtype=torch.int32, device="cuda")
    g = M.DecodeModel(CFG, W, capacity=MAX_BLOCKS * BLOCK_TOKENS, block_tokens=BLOCK_TOKENS, block_table=table_dev,
                      n_blocks=N_BLOCKS, max_seqs=MAX_RUNNING)
    sched = Scheduler(N_BLOCKS, BLOCK_TOKENS, MAX_BLOCKS, MAX_RUNNING, CHUNK, 1)
    prompts = {i: synth.prompt_ids(CFG, pl, seed=40 + i) for i, (pl, _) in enumerate(REQUESTS)}
    tokens = {i: list(p) for i, p in prompts.items()}  # prompt, then generated ids
    for i, (pl, mn) in enumerate(REQUESTS):
        sched.submit(i, pl, mn)
    preempted, steps = [], 0
    while True:
        st = sched.stats()
        if st["running"] == 0 and st["waiting"] == 0:
            break
        rows, table, gone = sched.plan()
        preempted += gone
        # chunk rows: the request's tokens at [offset, offset + count) through
        # stepSeq, its blocks at table row `slot`
        table_dev.copy_(torch.from_numpy(table))
        picks = {}
        for req, slot, off, cnt, dec, yields in rows:
            if dec:
                continue
            g.step_seq(tokens[req][off:off + cnt], seq=slot, offset=off)
            if yields:
                picks[req] = int(g.next_ids[slot])
        # decode rows: one batched step, row r addressing its request's blocks
        # through row r of a reordered table
        dec_rows = [r for r in rows if r[4]]
        if dec_rows:
            perm = np.full_like(table, -1)
            for r, (req, slot, off, cnt, dec, yields) in enumerate(dec_rows):
                perm[r] = table[slot]
            table_dev.copy_(torch.from_numpy(perm))
            g.set_state([tokens[r[0]][r[2]] for r in dec_rows], [r[2] for r in dec_rows])
            g.step(n_seqs=len(dec_rows))
            ids = g.next_ids[:len(dec_rows)].cpu().tolist()
            for r, row in enumerate(dec_rows):
                picks[row[0]] = ids[r]
        for req, t in picks.items():
            tokens[req].append(t)
        sched.commit()
        steps += 1
        assert steps < 500
    assert g.error_word() == 0
    return prompts, tokens, preempted, W


def test_scheduler_plans_on_gpu_match_oracle(M):
    prompts, tokens, preempted, W = run_trace(M)
    assert len(preempted) >= 2, preempted  # the trace exercises resume by recompute
    st = synth.weights_to_numpy(W)
    compared = 0
    for i, (pl, mn) in enumerate(REQUESTS):
        seq = tokens[i]
        assert len(seq) == pl + mn, (i, len(seq))
        o = O.Model(dict(CFG, block_tokens=1, max_blocks=pl + mn), st)
        for pos in range(pl + mn - 1):
            ref = o.step(seq[pos], pos)
            if pos >= pl - 1 and top2_gap(ref) > TIE_GAP:
                assert seq[pos + 1] == O.argmax(ref.astype(np.float32))[0], (i, pos)
                compared += 1
    assert compared >= 0.9 * sum(mn for _, mn in REQUESTS)
