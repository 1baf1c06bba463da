"""The continuous-batching scheduler slice (``ds_sched_*``) from Python:
argument marshalling only; every decision is made by the library."""
import ctypes

import numpy as np

from . import abi


class Scheduler:
    """Plans steps over a paged K/V pool of ``n_blocks`` blocks of
    ``block_tokens`` positions for at most ``max_running`` requests, each
    mapping at most ``max_blocks`` blocks ("Inside the engine", section 2)."""

    def __init__(self, n_blocks, block_tokens, max_blocks, max_running, chunk, headroom_blocks=1):
        c = abi.SchedConfig()
        c.n_blocks, c.block_tokens, c.max_blocks = n_blocks, block_tokens, max_blocks
        c.max_running, c.chunk, c.headroom_blocks = max_running, chunk, headroom_blocks
        self.cfg = c
        h = ctypes.c_void_p()
        abi.check(abi.lib.ds_sched_create(ctypes.byref(c), ctypes.byref(h)), "ds_sched_create")
        self._h = h
        self._rows = (abi.SchedRow * max_running)()
        self._table = np.empty((max_running, max_blocks), dtype=np.int32)
        self._gone = (ctypes.c_int64 * max_running)()

    def __del__(self):
        if getattr(self, "_h", None):
            abi.lib.ds_sched_destroy(self._h)
            self._h = None

    def submit(self, request, prompt_len, max_new):
        abi.check(abi.lib.ds_sched_submit(self._h, request, prompt_len, max_new), "ds_sched_submit")

    def plan(self):
        """Returns (rows, block_table, preempted): rows as tuples (request,
        slot, offset, count, decode, yields), oldest request first; the
        block table as int32 [max_running, max_blocks] (-1 unused); the ids
        this plan preempted."""
        n = ctypes.c_int32()
        ng = ctypes.c_int32()
        abi.check(abi.lib.ds_sched_plan(self._h, self._rows, len(self._rows), ctypes.byref(n),
                                        self._table.ctypes.data_as(ctypes.c_void_p), self._gone,
                                        ctypes.byref(ng)), "ds_sched_plan")
        rows = [(r.request, r.slot, r.offset, r.count, r.decode, r.yields) for r in self._rows[:n.value]]
        return rows, self._table.copy(), list(self._gone[:ng.value])

    def commit(self, finished=()):
        ids = (ctypes.c_int64 * max(len(finished), 1))(*finished)
        abi.check(abi.lib.ds_sched_commit(self._h, ids, len(finished)), "ds_sched_commit")

    def stats(self):
        out = (ctypes.c_int64 * 5)()
        abi.check(abi.lib.ds_sched_stats(self._h, out), "ds_sched_stats")
        return dict(zip(("free_blocks", "running", "waiting", "finished", "preemptions"), list(out)))

    def generated(self, request):
        return int(abi.lib.ds_sched_generated(self._h, request))
