"""Test infrastructure: the oracle of the continuous-batching scheduler slice.

Only the tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline leg
use this package; the product never does.

A plain restatement of the scheduling policy of "Inside the engine", section
2 (admission, chunks, preemption, resume), for a paged K/V pool whose blocks
each hold every layer's K/V of ``block_tokens`` positions.  Slow and direct:
plain lists, every choice re-derived from the whole state each time.

The policy, in the page's order:

* Admission.  A waiting request is admitted only when the free blocks cover
  its whole uncached suffix — for a waiting request that is all its tokens,
  the prompt plus whatever it generated before a preemption — plus the decode
  headroom; the blocks are taken at admission.  Waiting requests are served
  first come first served: preempted ones first, in the order they were
  preempted, then new ones in submission order; admission stops at the first
  one that does not fit (no overtaking, so none starves).  A request also
  needs a free block-table row.
* Chunks.  A request with uncached tokens advances by at most ``chunk`` of
  them per step; the step that reaches its last token produces its next
  token.  A request whose tokens are all cached except the last one (a
  decoding request) advances by that one token.
* Preemption.  When a decoding request's next position lies past its blocks
  and the pool has no free block, the youngest running request (the last
  submitted) is preempted, until a block is free or the requester itself was
  the youngest.  Older requests are served first, so older work is never
  sacrificed for newer.  A preempted request loses its blocks, its row and
  its cache.
* Resume.  Preempted requests wait ahead of new ones, first preempted first,
  and recompute their prefix through the chunked path.
* Completion.  After a step, a request that has produced ``max_new`` tokens,
  or that the caller reports finished, releases its blocks and row; they
  admit waiting requests at the next plan.
"""


class SchedulerOracle:
    def __init__(self, n_blocks, block_tokens, max_blocks, max_running, chunk, headroom_blocks=1):
        self.n_blocks, self.bt, self.max_blocks = n_blocks, block_tokens, max_blocks
        self.max_running, self.chunk, self.headroom = max_running, chunk, headroom_blocks
        self.req = {}            # id -> dict of the request's state
        self.submitted = 0
        self.preempt_count = 0
        self.finished_count = 0
        self.last_plan = None

    # ------------------------------------------------------------ helpers
    def _blocks_for(self, positions):
        return -(-positions // self.bt)

    def _tokens(self, r):
        return r["prompt"] + r["generated"]

    def _held_blocks(self):
        return [b for r in self.req.values() if r["state"] == "running" for b in r["blocks"]]

    def _free_blocks(self):
        held = set(self._held_blocks())
        return [b for b in range(self.n_blocks) if b not in held]

    def _free_rows(self):
        used = {r["slot"] for r in self.req.values() if r["state"] == "running"}
        return [s for s in range(self.max_running) if s not in used]

    def _running(self):
        """Running request ids, oldest (first submitted) first."""
        ids = [i for i, r in self.req.items() if r["state"] == "running"]
        return sorted(ids, key=lambda i: self.req[i]["arrival"])

    def _waiting(self):
        """Waiting ids in service order: preempted by preemption order, then new by submission."""
        pre = [i for i, r in self.req.items() if r["state"] == "waiting" and r["preempted_at"] is not None]
        new = [i for i, r in self.req.items() if r["state"] == "waiting" and r["preempted_at"] is None]
        return (sorted(pre, key=lambda i: self.req[i]["preempted_at"]) +
                sorted(new, key=lambda i: self.req[i]["arrival"]))

    # ------------------------------------------------------------ API
    def submit(self, request, prompt_len, max_new):
        if request in self.req and self.req[request]["state"] != "finished":
            raise ValueError("request %r is live" % request)
        self.req[request] = dict(arrival=self.submitted, prompt=prompt_len, max_new=max_new, generated=0,
                                 cached=0, state="waiting", slot=-1, blocks=[], preempted_at=None)
        self.submitted += 1

    def plan(self):
        assert self.last_plan is None, "the previous plan is not committed"
        # 1. admission, strictly in service order
        for i in self._waiting():
            r = self.req[i]
            need = self._blocks_for(self._tokens(r))
            free, rows = self._free_blocks(), self._free_rows()
            if not rows or len(free) < need + self.headroom:
                break
            r["state"], r["slot"], r["blocks"], r["cached"] = "running", rows[0], free[:need], 0
        # 2. decoding requests claim the block of their next position, oldest first
        preempted = []
        for i in self._running():
            r = self.req[i]
            if r["state"] != "running":
                continue  # preempted earlier in this loop
            if r["cached"] != self._tokens(r) - 1 or r["cached"] < len(r["blocks"]) * self.bt:
                continue
            while not self._free_blocks() and r["state"] == "running":
                victim = self._running()[-1]
                v = self.req[victim]
                v["state"], v["slot"], v["blocks"], v["cached"] = "waiting", -1, [], 0
                v["preempted_at"] = self.preempt_count
                self.preempt_count += 1
                preempted.append(victim)
            if r["state"] == "running":
                r["blocks"] = r["blocks"] + [self._free_blocks()[0]]
        # 3. one row per running request, oldest first
        rows = []
        for i in self._running():
            r = self.req[i]
            n = self._tokens(r)
            count = min(self.chunk, n - r["cached"])
            rows.append((i, r["slot"], r["cached"], count,
                         int(r["cached"] == n - 1 and r["generated"] >= 1), int(r["cached"] + count == n)))
        table = [[-1] * self.max_blocks for _ in range(self.max_running)]
        for i in self._running():
            r = self.req[i]
            for j, b in enumerate(r["blocks"]):
                table[r["slot"]][j] = b
        self.last_plan = rows
        return rows, table, preempted

    def commit(self, finished=()):
        assert self.last_plan is not None, "nothing planned"
        for (i, slot, offset, count, decode, yields) in self.last_plan:
            r = self.req[i]
            r["cached"] += count
            if yields:
                r["generated"] += 1
        for i, r in self.req.items():
            if r["state"] == "finished":
                continue
            if (r["state"] == "running" and r["generated"] >= r["max_new"]) or i in finished:
                r["state"], r["slot"], r["blocks"] = "finished", -1, []
                self.finished_count += 1
        self.last_plan = None

    def stats(self):
        return dict(free_blocks=len(self._free_blocks()), running=len(self._running()),
                    waiting=len(self._waiting()), finished=self.finished_count, preemptions=self.preempt_count)

    def generated(self, request):
        return self.req[request]["generated"] if request in self.req else -1
