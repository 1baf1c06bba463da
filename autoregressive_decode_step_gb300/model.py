"""Decode driver over the C ABI: model creation, KV cache, single steps,
captured-graph replay, per-kernel timing and a greedy generation loop.

PyTorch supplies device memory and streams; every step of the decode runs in
the library's kernels (``ds_decode_step`` / ``ds_step_graph_*``).
"""
import ctypes

import torch

from . import abi
from . import configs as C


def _ptr_array(tensors):
    return (ctypes.c_void_p * max(1, len(tensors)))(*[t.data_ptr() for t in tensors])


class DecodeModel:
    """A model resident on the GPU plus its KV cache and decode state.

    ``weights``: dict in the storage layout of ``configs`` (torch tensors on
    the device).  ``capacity``: positions the KV cache reserves per sequence
    (rounded up to whole blocks).  ``block_table``: optional device int32
    [max_seqs, max_blocks] mapping a sequence's blocks to physical blocks of a
    pool with ``n_blocks`` blocks.
    """

    def __init__(self, cfg, weights, capacity, device="cuda", block_tokens=16, block_table=None, n_blocks=None,
                 max_seqs=1):
        self.cfg = dict(cfg)
        self.device = torch.device(device)
        self.weights = weights
        c = self.cfg
        self.block_tokens = block_tokens
        self.max_blocks = (capacity + block_tokens - 1) // block_tokens
        self.capacity = self.max_blocks * block_tokens
        self.max_seqs = max_seqs
        mc = abi.ModelConfig()
        mc.vocab, mc.d, mc.n_layer = c["vocab"], c["d"], c["n_layer"]
        mc.n_qh, mc.n_kvh, mc.head_dim, mc.ff = c["n_qh"], c["n_kvh"], c["head_dim"], c["ff"]
        mc.rope_layout, mc.rope_base, mc.eps = c["rope_layout"], c["rope_base"], c.get("eps", 1e-5)
        mc.tied, mc.w_dtype, mc.kv_dtype = c["tied"], c["w_dtype"], c["kv_dtype"]
        mc.max_seqs, mc.max_ctx = max_seqs, self.capacity
        sc = c.get("rope_scaling")
        if sc:
            mc.rope_factor, mc.rope_low_freq_factor = sc["factor"], sc["low_freq_factor"]
            mc.rope_high_freq_factor, mc.rope_orig_max_pos = sc["high_freq_factor"], sc["original_max_position"]
        self._mc = mc
        W = weights
        names = ("n1", "wqkv", "wo", "n2", "wgu", "wd") + (("q_norm", "k_norm") if "q_norm" in W else ())
        self._arrays = {k: _ptr_array(W[k]) for k in names}
        mw = abi.ModelWeights()
        mw.emb = W["emb"].data_ptr()
        mw.out = W["out"].data_ptr()
        mw.final_norm = W["norm"].data_ptr()
        for k, arr in self._arrays.items():
            setattr(mw, k, ctypes.cast(arr, ctypes.c_void_p))
        self._mw = mw
        ws_bytes = abi.lib.ds_model_workspace_bytes(ctypes.byref(mc))
        if ws_bytes == 0:
            raise abi.DecodeStepError(abi.DS_BAD_ARGUMENT, "ds_model_workspace_bytes")
        self.ws = abi.workspace(ws_bytes, self.device)
        handle = ctypes.c_void_p()
        abi.check(abi.lib.ds_model_create(ctypes.byref(mc), ctypes.byref(mw), abi.ptr(self.ws), ws_bytes,
                                          ctypes.byref(handle)), "ds_model_create")
        self._h = handle
        # KV cache
        kvdt = torch.float32 if c["kv_dtype"] == C.F32 else torch.bfloat16
        row = c["n_kvh"] * c["head_dim"]
        if block_table is None:
            rows = self.capacity * max_seqs
        else:
            rows = n_blocks * block_tokens
        self.kv_rows = rows
        self.k_cache = [torch.zeros(rows, row, dtype=kvdt, device=self.device) for _ in range(c["n_layer"])]
        self.v_cache = [torch.zeros(rows, row, dtype=kvdt, device=self.device) for _ in range(c["n_layer"])]
        self.block_table = block_table
        self._kv_arrays = (_ptr_array(self.k_cache), _ptr_array(self.v_cache))
        kv = abi.KVCache()
        kv.k = ctypes.cast(self._kv_arrays[0], ctypes.c_void_p)
        kv.v = ctypes.cast(self._kv_arrays[1], ctypes.c_void_p)
        kv.rows = rows
        kv.block_tokens = block_tokens
        kv.max_blocks = self.max_blocks
        kv.block_table = None if block_table is None else block_table.data_ptr()
        self._kv = kv
        # decode state on the device
        self.tokens = torch.zeros(max_seqs, dtype=torch.int32, device=self.device)
        self.pos = torch.zeros(max_seqs, dtype=torch.int32, device=self.device)
        self.next_ids = torch.zeros(max_seqs, dtype=torch.int32, device=self.device)
        self.u = torch.zeros(max_seqs, dtype=torch.float32, device=self.device)
        self.logits = torch.zeros(max_seqs, c["vocab"], dtype=torch.float32, device=self.device)
        self._graphs = {}

    def __del__(self):
        try:
            for g in self._graphs.values():
                abi.lib.ds_step_graph_destroy(g)
            if getattr(self, "_h", None):
                abi.lib.ds_model_destroy(self._h)
        except Exception:
            pass

    # -------------------------------------------------------------- steps
    def _sampling(self, sampling):
        if sampling is None:
            return None
        s = abi.Sampling()
        s.temperature, s.top_k, s.top_p = sampling
        return ctypes.byref(s)

    def step(self, n_seqs=1, sampling=None, advance=False, write_logits=True, stream=None, phase_times=False,
             trace=False):
        """One decode step of tokens[:n_seqs] at pos[:n_seqs]; ids go to
        next_ids (and logits to self.logits)."""
        flags = ((abi.DS_STEP_ADVANCE if advance else 0) | (abi.DS_STEP_PHASE_TIMES if phase_times else 0) |
                 (abi.DS_STEP_TRACE if trace else 0))
        abi.check(abi.lib.ds_decode_step(self._h, ctypes.byref(self._kv), abi.ptr(self.tokens), abi.ptr(self.pos),
                                         n_seqs, self._sampling(sampling), abi.ptr(self.u), abi.ptr(self.next_ids),
                                         abi.ptr(self.logits) if write_logits else None, flags,
                                         abi.stream_handle(stream)), "ds_decode_step")

    def steps(self, n_steps, ids_out=None, advance=True, stream=None):
        """n_steps greedy steps of sequence 0 in one launch (ds_decode_steps);
        ids_out: optional device int32 tensor receiving every step's pick."""
        flags = abi.DS_STEP_ADVANCE if advance else 0
        abi.check(abi.lib.ds_decode_steps(self._h, ctypes.byref(self._kv), abi.ptr(self.tokens), abi.ptr(self.pos),
                                          n_steps, abi.ptr(ids_out), abi.ptr(self.next_ids), flags,
                                          abi.stream_handle(stream)), "ds_decode_steps")

    def step_seq(self, tokens, seq=0, offset=0, stream=None):
        """stepSeq: the tokens of sequence `seq` at positions offset,
        offset + 1, ... run as chunks of up to max_seqs rows on the batched
        path (ds_step_seq).  The greedy pick after the last token goes to
        next_ids[seq] and that token's logits to logits[seq]."""
        t = torch.as_tensor(tokens, dtype=torch.int32).to(self.device)
        # addresses, not views: the library itself refuses a sequence outside the model
        pick = ctypes.c_void_p(self.next_ids.data_ptr() + 4 * seq)
        logits = ctypes.c_void_p(self.logits.data_ptr() + 4 * seq * self.cfg["vocab"])
        abi.check(abi.lib.ds_step_seq(self._h, ctypes.byref(self._kv), abi.ptr(t), t.numel(), seq, offset,
                                      t.numel(), pick, logits, abi.stream_handle(stream)), "ds_step_seq")
        return t

    def graph(self, n_seqs=1, sampling=None, advance=True, write_logits=False, stream=None):
        """A captured step (created once per argument set); returns a
        callable that replays it on `stream`."""
        key = (n_seqs, sampling, advance, write_logits)
        if key not in self._graphs:
            stream = stream or torch.cuda.current_stream()
            if stream == torch.cuda.default_stream():
                raise ValueError("capture needs a non-default stream")
            h = ctypes.c_void_p()
            flags = abi.DS_STEP_ADVANCE if advance else 0
            abi.check(abi.lib.ds_step_graph_create(self._h, ctypes.byref(self._kv), abi.ptr(self.tokens),
                                                   abi.ptr(self.pos), n_seqs, self._sampling(sampling),
                                                   abi.ptr(self.u), abi.ptr(self.next_ids),
                                                   abi.ptr(self.logits) if write_logits else None, flags,
                                                   abi.stream_handle(stream), ctypes.byref(h)),
                      "ds_step_graph_create")
            self._graphs[key] = h
        h = self._graphs[key]

        def replay(stream=None):
            abi.check(abi.lib.ds_step_graph_launch(h, abi.stream_handle(stream)), "ds_step_graph_launch")

        return replay

    def profile(self, reps=3, n_seqs=1, sampling=None, advance=True, stream=None):
        """Mean duration (ms) of every kernel launch slot of one step, each
        launch bracketed by CUDA events (launches serialised)."""
        cap = 16 + 5 * self.cfg["n_layer"]
        ms = (ctypes.c_float * cap)()
        kinds = (ctypes.c_int32 * cap)()
        n = ctypes.c_int(0)
        flags = abi.DS_STEP_ADVANCE if advance else 0
        abi.check(abi.lib.ds_decode_step_profile(self._h, ctypes.byref(self._kv), abi.ptr(self.tokens),
                                                 abi.ptr(self.pos), n_seqs, self._sampling(sampling),
                                                 abi.ptr(self.u), abi.ptr(self.next_ids), None, flags, reps, ms,
                                                 kinds, cap, ctypes.byref(n), abi.stream_handle(stream)),
                  "ds_decode_step_profile")
        return [(abi.KIND_NAMES[kinds[i]], ms[i]) for i in range(n.value)]

    def phase_times_us(self, stream=None):
        """Per-phase durations (µs) of the last step run with phase_times=True:
        [("embed", t), ("qkv", t), ("attention", t), ..., ("head", t)]."""
        n_layer = self.cfg["n_layer"]
        cap = 5 * n_layer + 4
        buf = (ctypes.c_uint64 * cap)()
        n = ctypes.c_int(0)
        abi.check(abi.lib.ds_model_phase_times(self._h, buf, cap, ctypes.byref(n), abi.stream_handle(stream)),
                  "ds_model_phase_times")
        names = ["embed"] + ["qkv", "attention", "o_proj", "gate_up", "down"] * n_layer + ["head"]
        ts = [buf[i] for i in range(n.value)]
        return [(names[i], (ts[i + 1] - ts[i]) / 1000.0) for i in range(min(len(names), len(ts) - 1))]

    def trace(self, stream=None):
        """Per-CTA timestamps of the last traced step as an int64 tensor
        [phase, cta, 5] (see ds_model_trace)."""
        n_layer = self.cfg["n_layer"]
        n_phase = 5 * n_layer + 4
        cap = n_phase * 1024 * 5
        buf = (ctypes.c_uint64 * cap)()
        nw = ctypes.c_size_t(0)
        nc = ctypes.c_int(0)
        abi.check(abi.lib.ds_model_trace(self._h, buf, cap, ctypes.byref(nw), ctypes.byref(nc),
                                         abi.stream_handle(stream)), "ds_model_trace")
        t = torch.tensor(list(buf[:nw.value]), dtype=torch.int64)
        return t.reshape(-1, nc.value, 5)

    def kernel_time_us(self, kind, reps=4, stream=None):
        """Mean microseconds per launch of one kernel kind ("qkv", "attention",
        "o_proj", "gate_up", "down", "head", "embed"), launched back to back
        over every layer (see ds_decode_kernel_time)."""
        us = ctypes.c_float(0.0)
        abi.check(abi.lib.ds_decode_kernel_time(self._h, ctypes.byref(self._kv), abi.ptr(self.tokens),
                                                abi.ptr(self.pos), abi.KIND_NAMES.index(kind), reps,
                                                ctypes.byref(us), abi.stream_handle(stream)),
                  "ds_decode_kernel_time")
        return us.value

    def error_word(self, stream=None):
        return abi.ds_workspace_error(self.ws, stream)

    # -------------------------------------------------------------- helpers
    def set_state(self, tokens, pos):
        self.tokens[:len(tokens)].copy_(torch.as_tensor(tokens, dtype=torch.int32))
        self.pos[:len(pos)].copy_(torch.as_tensor(pos, dtype=torch.int32))

    def prefill(self, prompt, seq=0):
        """Token-at-a-time prefill through the decode step (the page's
        prefill loop); returns the logits of the last prompt token."""
        for p, t in enumerate(prompt):
            self.set_state([t], [p])
            self.step()
        return self.logits[0].clone()

    def generate_greedy(self, prompt, n_new):
        """Prefill, then greedy decoding with the host reading each id; the
        last prefill step's fused argmax already picked the first new token."""
        self.prefill(prompt)
        out = []
        tok = int(self.next_ids[0].item())
        for i in range(n_new):
            out.append(tok)
            if i + 1 == n_new:
                break
            self.set_state([tok], [len(prompt) + i])
            self.step()
            tok = int(self.next_ids[0].item())
        return out
