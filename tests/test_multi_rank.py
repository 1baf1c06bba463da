"""The benchmark's multi-rank host logic on CPU with two gloo ranks: the
process-group set-up from the launcher's environment, the barrier, the
slowest-rank timing (max over ranks) and the rule that only rank 0 runs and
prints the reference arm."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    r, w, local = bench.dist_init()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # each rank "timed" a different duration; everyone sees the slowest
    slowest = bench.max_over_ranks(10.0 + rank, w)

    class A:
        steps, warmup, ctx = 2, 1, 16
    # rank 1 leaves the reference arm at once, without work or output
    rc = bench.run_reference(A, rank, w) if rank == 1 else 0
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((rank, slowest, rc))


@pytest.mark.timeout(180)
def test_two_gloo_ranks_share_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(150)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0, 0), (1, 11.0, 0)]
