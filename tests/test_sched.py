"""The continuous-batching scheduler slice ("Inside the engine", section 2):
the oracle pinned by a worked example and by invariants on random traces,
then the library's ds_sched_* against the oracle, decision for decision.
CPU only."""
import ctypes
import random

import numpy as np
import pytest

from oracle.sched import SchedulerOracle

# A hand-worked example: 4 blocks of 2 positions, 2 rows, chunks of 2, one
# block of headroom.  A (id 1): prompt 3, 3 new tokens; B (id 2): prompt 1,
# 4 new tokens.  Rows are (request, slot, offset, count, decode, yields).
WORKED = [
    # both admitted: A takes blocks 0, 1 (3 tokens) leaving 2 >= 1 + headroom
    # for B, which takes block 2; A runs a chunk of 2, B its one prompt token
    dict(rows=[(1, 0, 0, 2, 0, 0), (2, 1, 0, 1, 0, 1)], table=[[0, 1, -1, -1], [2, -1, -1, -1]], gone=[]),
    # A's last prompt token yields; B decodes its first token (position 1)
    dict(rows=[(1, 0, 2, 1, 0, 1), (2, 1, 1, 1, 1, 1)], table=[[0, 1, -1, -1], [2, -1, -1, -1]], gone=[]),
    # B's position 2 needs a block: the last free one, 3
    dict(rows=[(1, 0, 3, 1, 1, 1), (2, 1, 2, 1, 1, 1)], table=[[0, 1, -1, -1], [2, 3, -1, -1]], gone=[]),
    # A's position 4 needs a block and none is free: B, the youngest, is
    # preempted; A takes block 2 and produces its 3rd and last token
    dict(rows=[(1, 0, 4, 1, 1, 1)], table=[[0, 1, 2, -1], [-1] * 4], gone=[2]),
    # A finished; B resumes with its 4 tokens (prompt + 3 generated) in
    # blocks 0, 1 of row 0, recomputed in chunks of 2
    dict(rows=[(2, 0, 0, 2, 0, 0)], table=[[0, 1, -1, -1], [-1] * 4], gone=[]),
    dict(rows=[(2, 0, 2, 2, 0, 1)], table=[[0, 1, -1, -1], [-1] * 4], gone=[]),
]


def worked_run(sched):
    sched.submit(1, 3, 3)
    sched.submit(2, 1, 4)
    out = []
    for _ in WORKED:
        rows, table, gone = sched.plan()
        out.append(dict(rows=[tuple(r) for r in rows], table=[list(map(int, t)) for t in table],
                        gone=list(gone)))
        sched.commit()
    return out


def test_oracle_follows_the_worked_example():
    o = SchedulerOracle(n_blocks=4, block_tokens=2, max_blocks=4, max_running=2, chunk=2, headroom_blocks=1)
    assert worked_run(o) == WORKED
    assert o.stats() == dict(free_blocks=4, running=0, waiting=0, finished=2, preemptions=1)
    assert o.generated(1) == 3 and o.generated(2) == 4


def random_trace(seed, n_requests=40, steps=400):
    """Seeded submissions (prompt 1..40, 1..24 new tokens, arriving over the
    first half of the run) and occasional early finishes."""
    rng = random.Random(seed)
    arrivals = sorted(rng.randrange(steps // 2) for _ in range(n_requests))
    reqs = [(100 + i, rng.randint(1, 40), rng.randint(1, 24), arrivals[i]) for i in range(n_requests)]
    cancel = {rng.randrange(steps): rng.randrange(n_requests) for _ in range(4)}
    return reqs, cancel


CONFIGS = [dict(n_blocks=24, block_tokens=4, max_blocks=16, max_running=6, chunk=8, headroom_blocks=1),
           dict(n_blocks=17, block_tokens=2, max_blocks=32, max_running=4, chunk=5, headroom_blocks=2),
           dict(n_blocks=64, block_tokens=16, max_blocks=4, max_running=8, chunk=16, headroom_blocks=0)]


def drive(sched, cfg, seed, check=None):
    reqs, cancel = random_trace(seed)
    # positions a request may feed: one block-table row, and the pool less the headroom
    cap = min(cfg["max_blocks"], cfg["n_blocks"] - cfg["headroom_blocks"]) * cfg["block_tokens"]
    log = []
    t = 0
    while True:
        for rid, p, m, at in reqs:
            if at == t:
                m = min(m, cap)
                sched.submit(rid, max(1, min(p, cap - m + 1)), m)
        rows, table, gone = sched.plan()
        if check:
            check(sched, rows, table, gone)
        fin = []
        if t in cancel:
            fin = [reqs[cancel[t]][0]]
        sched.commit(fin)
        log.append(([tuple(r) for r in rows], [list(map(int, x)) for x in table], list(gone)))
        t += 1
        st = sched.stats()
        if t > max(at for *_, at in reqs) and st["running"] == 0 and st["waiting"] == 0:
            break
        assert t < 5000, "the trace does not drain"
    return log, sched.stats(), {rid: sched.generated(rid) for rid, *_ in reqs}


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_oracle_invariants_on_random_traces(cfg, seed):
    """Blocks are conserved and never shared, a row never maps another's
    blocks, every preemption takes the youngest running request, resumes
    keep preemption order ahead of new requests, and every request that is
    not cancelled ends with exactly max_new tokens."""
    seen_preempted = []

    def check(o, rows, table, gone):
        held = [b for r in o.req.values() if r["state"] == "running" for b in r["blocks"]]
        assert len(held) == len(set(held))
        assert len(held) + len(o._free_blocks()) == cfg["n_blocks"]
        mapped = [b for row in table for b in row if b >= 0]
        assert sorted(mapped) == sorted(held)
        for i in gone:
            younger = [j for j in o._running() if o.req[j]["arrival"] > o.req[i]["arrival"]]
            assert not younger, "an older request was preempted while a younger one runs"
        seen_preempted.extend(gone)
        # decode rows have their position's block
        for (rid, slot, off, cnt, dec, yl) in rows:
            r = o.req[rid]
            assert (off + cnt - 1) // cfg["block_tokens"] < len(r["blocks"])
            assert 1 <= cnt <= cfg["chunk"]

    o = SchedulerOracle(**cfg)
    log, st, gen = drive(o, cfg, seed, check)
    reqs, cancel = random_trace(seed)
    cancelled = {reqs[i][0] for i in cancel.values()}
    for rid, p, m, at in reqs:
        if rid not in cancelled:
            assert gen[rid] == m, rid
    assert st["free_blocks"] == cfg["n_blocks"]
    assert st["finished"] == len(reqs)


@pytest.fixture(scope="module")
def lib_sched():
    from autoregressive_decode_step_gb300 import build
    build.build()
    from autoregressive_decode_step_gb300.sched import Scheduler
    return Scheduler


def test_library_follows_the_worked_example(lib_sched):
    s = lib_sched(n_blocks=4, block_tokens=2, max_blocks=4, max_running=2, chunk=2, headroom_blocks=1)
    assert worked_run(s) == WORKED
    assert s.stats() == dict(free_blocks=4, running=0, waiting=0, finished=2, preemptions=1)


@pytest.mark.parametrize("cfg", CONFIGS)
@pytest.mark.parametrize("seed", [0, 1, 2, 3, 4])
def test_library_matches_the_oracle_step_for_step(lib_sched, cfg, seed):
    a = drive(SchedulerOracle(**cfg), cfg, seed)
    b = drive(lib_sched(**cfg), cfg, seed)
    for t, (x, y) in enumerate(zip(a[0], b[0])):
        assert x == y, t
    assert len(a[0]) == len(b[0])
    assert a[1] == b[1] and a[2] == b[2]


def test_library_refusals(lib_sched):
    from autoregressive_decode_step_gb300 import abi
    L = abi.lib
    h = ctypes.c_void_p()
    c = abi.SchedConfig(4, 2, 4, 2, 2, 1)
    assert L.ds_sched_create(None, ctypes.byref(h)) == abi.DS_BAD_ARGUMENT
    assert L.ds_sched_create(ctypes.byref(abi.SchedConfig(0, 2, 4, 2, 2, 1)), ctypes.byref(h)) == \
        abi.DS_EMPTY_DIMENSION
    assert L.ds_sched_create(ctypes.byref(c), ctypes.byref(h)) == abi.DS_OK
    try:
        assert L.ds_sched_submit(h, 1, 0, 3) == abi.DS_EMPTY_DIMENSION
        assert L.ds_sched_submit(h, 1, 8, 2) == abi.DS_CACHE_CAPACITY_EXCEEDED   # 9 positions > 4 x 2
        assert L.ds_sched_submit(h, 1, 7, 1) == abi.DS_CACHE_CAPACITY_EXCEEDED   # 4 blocks + 1 headroom > 4
        assert L.ds_sched_submit(h, 1, 3, 2) == abi.DS_OK
        assert L.ds_sched_submit(h, 1, 2, 2) == abi.DS_BAD_ARGUMENT              # id still live
        assert L.ds_sched_commit(h, None, 0) == abi.DS_BAD_ARGUMENT              # nothing planned
        rows = (abi.SchedRow * 2)()
        table = np.empty((2, 4), dtype=np.int32)
        n = ctypes.c_int32()
        tp = table.ctypes.data_as(ctypes.c_void_p)
        assert L.ds_sched_plan(h, rows, 1, ctypes.byref(n), tp, None, None) == abi.DS_WORKSPACE_TOO_SMALL
        assert L.ds_sched_plan(h, rows, 2, ctypes.byref(n), tp, None, None) == abi.DS_OK
        assert L.ds_sched_plan(h, rows, 2, ctypes.byref(n), tp, None, None) == abi.DS_BAD_ARGUMENT  # uncommitted
        assert L.ds_sched_commit(h, None, 0) == abi.DS_OK
    finally:
        L.ds_sched_destroy(h)
