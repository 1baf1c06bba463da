#!/usr/bin/env python
"""Batch-1 decode benchmark of the Llama-3-8B-shaped random-init decoder.

One step = one whole single-token decode step (32 layers of q|k|v, RoPE+KV
write, attention, o, gate|up+SiLU, down, then the output head and greedy
argmax) replayed from a captured CUDA graph with the token and position
advanced on the device.  The context starts at --ctx prefilled positions
(a random prompt run through the same decode step) and grows by one per step.

Prints one JSON line (see the keys below).  `--impl reference` times the CPU
oracle on the host cores instead (a bounded sample per step, scaled to the
same metric).  Under torchrun each rank decodes its own replica (no data-path
communication); rank 0 prints the aggregate.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "batch-1 decode tokens/s and % of GB300 HBM roofline; per-op us vs CPU oracle"
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=256)
    p.add_argument("--warmup", type=int, default=8)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--ctx", type=int, default=1024, help="prefilled context before the first timed step")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-batched", action="store_true", help="skip the batched (64-sequence) decode measurement")
    p.add_argument("--batched-only", action="store_true",
                   help="time only the batched (64-sequence) decode (a profiling case; the line's batch-1 keys are "
                        "then absent)")
    p.add_argument("--no-ops", action="store_true", help="skip the op-level timings")
    p.add_argument("--no-legs", action="store_true",
                   help="skip the extra batch-1 legs (8B at contexts 4096 and 8192, the Qwen3-0.6B shape, the tiny "
                        "decoder)")
    p.add_argument("--ops-only", action="store_true",
                   help="time only the op-level decode glue (a profiling case: no step, no CPU baseline)")
    p.add_argument("--ops-reps", type=int, default=200, help="timed launches per op in the op-level leg")
    p.add_argument("--prompt-only", action="store_true",
                   help="time only the chunked prompt (stepSeq) leg (a profiling case)")
    p.add_argument("--batched-steps", type=int, default=None,
                   help="timed steps of the batched decode (default: the workload's 128)")
    p.add_argument("--chunk", type=int, default=32,
                   help="greedy steps per kernel launch in the timed region (the picks hand over on the device); "
                        "1 = one captured-graph replay per step")
    p.add_argument("--layers", type=int, default=None,
                   help="decoder layers (default: the model's 32); fewer layers make a small profiling case, "
                        "not a benchmark number")
    p.add_argument("--kv-fill", choices=["prefill", "synthetic"], default="prefill",
                   help="fill the first --ctx cache positions by prefilling a random prompt through the decode "
                        "step, or with seeded N(0,1) K/V values (same step cost, far fewer launches)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def workload_config(args, cfg):
    from autoregressive_decode_step_gb300 import configs as C
    return {"workload": "llama3-8b-shape random-init decoder, batch-1 greedy decode, context %d + %d decoded "
                        "(positions %d..%d)" % (args.ctx, args.steps, args.ctx, args.ctx + args.steps - 1),
            "context": args.ctx, "batch": 1, "layers": cfg["n_layer"], "d": cfg["d"], "ff": cfg["ff"],
            "heads": "%dq/%dkv x %d" % (cfg["n_qh"], cfg["n_kvh"], cfg["head_dim"]), "vocab": cfg["vocab"],
            "weights": "bf16", "kv_cache": "bf16", "activations": "fp32",
            "l2": "inputs larger than L2 (%.1f GB of weights streamed per step)" % (C.weight_bytes_per_step(cfg) / 1e9),
            "parallelism": "replicas (one independent decoder per GPU)"}


# ------------------------------------------------------------------ distributed
def dist_init():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch
    import torch.distributed as dist
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    dist.init_process_group(backend=backend)
    return dist.get_rank(), ws, int(os.environ.get("LOCAL_RANK", "0"))


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value, world):
    """Largest value over all ranks (timing is taken as the slowest rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id):
        self.samples = []
        self.proc = None
        self.bus_id = bus_id

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.bus_id, "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 - 0.15 <= t <= t1 + 0.15] or [s for (_, s) in self.samples[-3:]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [x.strip() for x in r.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle
class OracleDecoder:
    """The CPU oracle's full-depth decode step on the given weights over a
    synthetic prefilled context of `ctx` positions (seeded N(0,1) K/V rows,
    the same recipe the GPU legs use): greedy, one token at a time from
    position ctx."""

    def __init__(self, cfg, W, ctx, capacity, seed):
        import oracle as O
        from autoregressive_decode_step_gb300 import synth

        self.O = O
        st = synth.weights_to_numpy(W)
        self.m = O.Model(dict(cfg, block_tokens=1, max_blocks=capacity), st)
        dev = W["emb"].device
        ks, vs = synth.synthetic_kv(cfg, ctx, seed=seed, device=dev)
        for l in range(cfg["n_layer"]):
            self.m.k[l][:ks[l].numel()] = synth.to_numpy_storage(ks[l])
            self.m.v[l][:vs[l].numel()] = synth.to_numpy_storage(vs[l])
        del ks, vs
        self.tok, self.pos = 7, ctx

    def step(self):
        """One decode step; returns its wall time in seconds."""
        t = time.perf_counter()
        logits = self.m.step(self.tok, self.pos)
        dt = time.perf_counter() - t
        self.tok, self.pos = self.O.argmax(logits.astype("float32"))[0], self.pos + 1
        return dt


def run_reference(args, rank, world):
    """The oracle as it stands, timed on the host cores: every step is one
    whole 32-layer decode step of the 8B shape (weights once, K/V of every
    attended position), the same workload as the GPU arm."""
    import oracle as O
    import torch
    from autoregressive_decode_step_gb300 import configs as C
    from autoregressive_decode_step_gb300 import synth

    if rank != 0:
        return 0
    cfg = C.LLAMA3_8B
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    W = synth.model_weights(cfg, seed=0, device=dev)
    od = OracleDecoder(cfg, W, args.ctx, args.ctx + args.warmup + args.steps + 1, seed=1)
    del W
    for _ in range(args.warmup):
        od.step()
    times = [od.step() for _ in range(args.steps)]
    total = sum(times)
    value = args.steps / total
    sample = ("every step a whole decode step of the oracle (32 layers + the 128,256-row head, greedy) at positions "
              "%d..%d after %d untimed steps, over a synthetic %d-position context; %d threads"
              % (args.ctx + args.warmup, args.ctx + args.warmup + args.steps - 1, args.warmup, args.ctx, O.threads()))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(args, cfg),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": O.threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm
STEP_TRAFFIC = os.path.join(ROOT, "profiles", "step_kernel_llama3_8b.json")


def kernel_source_sha():
    """sha256 over the sources of the persistent step kernel (the dominant
    kernel); the committed traffic record names the value it was taken on."""
    from autoregressive_decode_step_gb300.ncu_record import kernel_source_sha as sha
    return sha()


def traffic_ratio(kernel_src_sha):
    """DRAM bytes over algorithmic bytes of the step kernel from the committed
    ncu record, when it was taken on the current kernel source (else None).
    Traffic is proportional to the bytes streamed, so a launch's traffic is
    this ratio times its algorithmic bytes."""
    try:
        with open(STEP_TRAFFIC) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_src_sha:
        return None
    return float(rec["dram_bytes"]) / float(rec["algorithmic_bytes"])


def time_batch1(model, cfg, K, chunk, first, ctx, stream):
    """K greedy decode steps of one sequence from position ctx, in launches of
    up to `chunk` steps each (the picks handed over on the device), between
    CUDA events on `stream`; returns (ms, launches)."""
    import torch

    chunks = []
    left = K
    while left > 0:
        chunks.append(min(chunk, left))
        left -= chunks[-1]
    model.set_state([first], [ctx])
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for n in chunks:
        model.steps(n, stream=stream)
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1), len(chunks)


def run_batch1_leg(cfg, W, dev, ctx, K, warmup, chunk, kv_seed, prompt=None):
    """Batch-1 greedy decode of `cfg` from a context of ctx positions (a
    random prompt prefilled through the decode step when `prompt` is given,
    else seeded N(0,1) K/V rows), K steps timed as in the main leg; the
    roofline is every weight byte once plus the K/V of every attended
    position, over the measured HBM bandwidth."""
    import torch

    from autoregressive_decode_step_gb300 import configs as C
    from autoregressive_decode_step_gb300 import synth
    from autoregressive_decode_step_gb300.model import DecodeModel

    model = DecodeModel(cfg, W, capacity=ctx + max(K, warmup) + 8, device=dev, block_tokens=16)
    if prompt is not None:
        model.prefill(prompt)
        first = int(model.next_ids[0])
    else:
        ks, vs = synth.synthetic_kv(cfg, ctx, seed=kv_seed, device=dev)
        for l in range(cfg["n_layer"]):
            model.k_cache[l][:ctx].copy_(ks[l])
            model.v_cache[l][:ctx].copy_(vs[l])
        del ks, vs
        first = synth.prompt_ids(cfg, 1, seed=kv_seed)[0]
    stream = torch.cuda.Stream(device=dev)
    time_batch1(model, cfg, warmup, chunk, first, ctx, stream)
    ms, launches = time_batch1(model, cfg, K, chunk, first, ctx, stream)
    err = model.error_word()
    if err:
        raise RuntimeError("device error word %d" % err)
    alg = sum(C.step_bytes(cfg, ctx + i + 1) for i in range(K)) / K
    peak, kind = peaks()
    achieved = alg / (ms / K / 1e3) / 1e9
    del model
    torch.cuda.empty_cache()
    return {"value": K / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms / K, "steps": K, "warmup": warmup,
            "launches": launches, "context": ctx,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": kind, "algorithmic_bytes_per_step": alg}}


def run_toy_leg(dev, reps=50):
    """The pages' tiny decoder (vocab 40, d 16, 2 layers; P4's seed-0
    weights and prompt): microseconds per greedy step, one captured-graph
    replay per step and 16 steps per launch, and the oracle's microseconds
    per step on one host core."""
    import torch

    import oracle as O
    from autoregressive_decode_step_gb300 import configs as C
    from autoregressive_decode_step_gb300 import synth
    from autoregressive_decode_step_gb300.model import DecodeModel

    cfg = C.TOY
    st = synth.p4_to_storage(synth.p4_toy_weights(cfg, 0), cfg)
    W = {k: ([torch.from_numpy(a).to(dev) for a in v] if isinstance(v, list) else torch.from_numpy(v).to(dev))
         for k, v in st.items()}
    g = DecodeModel(cfg, W, capacity=cfg["max_seq"], device=dev, block_tokens=4)
    prompt = list(synth.P4_PROMPT)
    g.prefill(prompt)
    first = int(g.next_ids[0])
    p0 = len(prompt)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        replay = g.graph(advance=True, write_logits=False, stream=stream)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn):
        best = float("inf")
        for _ in range(3):
            g.set_state([first], [p0])
            torch.cuda.synchronize()
            ev[0].record(stream)
            fn()
            ev[1].record(stream)
            ev[1].synchronize()
            best = min(best, ev[0].elapsed_time(ev[1]) * 1e3)
        return best

    def replays():
        for _ in range(16):
            replay(stream)

    us_graph = timed(replays) / 16
    us_multi = timed(lambda: g.steps(16, stream=stream)) / 16
    ids = torch.zeros(16, dtype=torch.int32, device=dev)
    g.set_state([first], [p0])
    g.steps(16, ids_out=ids)
    gpu_ids = [first] + ids.cpu().tolist()[:15]
    o = O.Model(dict(cfg, block_tokens=1, max_blocks=cfg["max_seq"]), st)
    before = O.threads()
    O.set_threads(1)
    t0 = time.perf_counter()
    want, _ = O.greedy_generate(o, prompt, 16)
    t_oracle = time.perf_counter() - t0
    O.set_threads(before)
    return {"workload": "tiny Llama-style decoder of \"The forward pass end to end\" (vocab 40, d 16, 2 layers, "
                        "4q/2kv x 4, ff 24, fp32, P4's seed-0 weights and prompt [3,14,15,9,2,6]), 16 greedy steps",
            "us_per_step_graph_replay": us_graph, "us_per_step_16_per_launch": us_multi,
            "oracle_us_per_step_one_core": t_oracle * 1e6 / (len(prompt) + 16),
            "ids_equal_oracle": gpu_ids == want, "first_ids": gpu_ids[:4]}


def run_batched(cfg, W, dev, rank, clocks_cls, bus, warmup=3, steps=None):
    """Batched continuous decode on the same 8B-shaped weights: 64 sequences,
    contexts uniform in [128, 4096] (a synthetic prefilled paged pool of
    16-position blocks), one token per sequence per step, per-row sampling at
    temperature 0.8 / top_k 50 / top_p 0.95 with seeded draws, 128 steps
    replayed from a captured graph (tokens and positions advance on the
    device; each step's 64 draws are copied into place before it)."""
    import torch

    from autoregressive_decode_step_gb300 import configs as C
    from autoregressive_decode_step_gb300 import synth
    from autoregressive_decode_step_gb300.model import DecodeModel

    B = C.BATCHED_8B
    n, bt = B["n_seqs"], B["block_tokens"]
    steps = steps or B["steps"]
    ctx = synth.context_lengths(n, B["ctx_lo"], B["ctx_hi"], seed=rank)
    # a compact pool: sequence s owns ceil((ctx + steps + warm-up + 1) / bt)
    # blocks, scattered over the pool by a seeded permutation
    need = [(c + steps + warmup + 1 + bt - 1) // bt for c in ctx]
    max_blocks = max(need)
    n_blocks = sum(need)
    perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(rank + 1)).to(torch.int32)
    table = torch.zeros(n, max_blocks, dtype=torch.int32)
    at = 0
    for s_, k in enumerate(need):
        table[s_, :k] = perm[at:at + k]
        at += k
    model = DecodeModel(cfg, W, capacity=max_blocks * bt, device=dev, block_tokens=bt,
                        block_table=table.to(dev), n_blocks=n_blocks, max_seqs=n)
    ks, vs = synth.synthetic_kv(cfg, n_blocks * bt, seed=rank + 2, device=dev)
    for l in range(cfg["n_layer"]):
        model.k_cache[l].copy_(ks[l])
        model.v_cache[l].copy_(vs[l])
    del ks, vs
    toks = synth.prompt_ids(cfg, n, seed=rank + 3)
    U = synth.uniform_draws((warmup + steps) * n, seed=rank + 4).view(warmup + steps, n).to(dev)
    stream = torch.cuda.Stream(device=dev)
    sampling = (B["temperature"], B["top_k"], B["top_p"])
    with torch.cuda.stream(stream):
        replay = model.graph(n_seqs=n, sampling=sampling, advance=True, write_logits=False, stream=stream)
    model.set_state(toks, ctx)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(warmup):
            model.u[:n].copy_(U[i], non_blocking=True)
            replay(stream)
    stream.synchronize()
    pos0 = [c + warmup for c in ctx]
    clocks = clocks_cls(bus)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            model.u[:n].copy_(U[warmup + i], non_blocking=True)
            replay(stream)
        e1.record(stream)
    e1.synchronize()
    t_wall1 = time.perf_counter()
    ms = e0.elapsed_time(e1)
    time.sleep(0.2)
    clocks.stop()
    err = model.error_word()
    if err:
        raise RuntimeError("device error word %d during the batched timed region" % err)
    assert model.pos[:n].cpu().tolist() == [p + steps for p in pos0]
    kvb = C.kv_bytes_per_token(cfg)
    alg = sum(C.weight_bytes_per_step(cfg) + sum(p + i + 1 for p in pos0) * kvb for i in range(steps)) / steps
    step_ms = ms / steps
    peak, kind = peaks()
    achieved = alg / (step_ms / 1e3) / 1e9
    out = {"workload": "llama3-8b-shape, %d sequences, contexts uniform in [%d, %d] (mean %.0f), paged K/V pool of "
                       "%d-position blocks (%d blocks), sampling T=%.1f top_k=%d top_p=%.2f with seeded draws, %d steps"
                       % (n, B["ctx_lo"], B["ctx_hi"], sum(ctx) / n, bt, n_blocks, sampling[0], sampling[1],
                          sampling[2], steps),
           "value": n * steps / (ms / 1e3), "unit": "tokens/s (all sequences)", "ms_per_step": step_ms,
           "steps": steps, "warmup": warmup,
           "hbm_roofline_step": {"achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                                 "algorithmic_bytes_per_step": alg,
                                 "algorithmic_bytes": "every weight byte once + K/V of every attended position of "
                                                      "every sequence", "peak_source": kind},
           "gpu_launches_per_step": 5 * cfg["n_layer"] + 5,  # embed, first norm, 5 per layer, final norm, head, sampler
           "clocks": clocks.summary(t_wall0, t_wall1)}
    del model
    torch.cuda.empty_cache()
    return out


def run_step_seq(cfg, W, dev, rank, clocks_cls, bus, prompt_len=1024, rows=256, warmup=1, reps=3):
    """A prompt of one sequence through ds_step_seq on the same 8B-shaped
    weights: prompt_len random tokens from position 0, chunks of `rows` rows
    on the batched path (q|k|v, o, gate|up, down as GEMMs over the chunk's
    rows on the tensor cores; each row attends its own causal prefix), then
    the last token's head and greedy pick.  The K/V of the prompt goes to
    one sequence's blocks of a paged pool."""
    import torch

    from autoregressive_decode_step_gb300 import configs as C
    from autoregressive_decode_step_gb300 import synth
    from autoregressive_decode_step_gb300.model import DecodeModel

    bt = 16
    mb = (prompt_len + bt - 1) // bt
    table = torch.zeros(rows, mb, dtype=torch.int32)
    table[0] = torch.randperm(mb, generator=torch.Generator().manual_seed(rank + 5)).to(torch.int32)
    model = DecodeModel(cfg, W, capacity=mb * bt, device=dev, block_tokens=bt, block_table=table.to(dev),
                        n_blocks=mb, max_seqs=rows)
    prompt = synth.prompt_ids(cfg, prompt_len, seed=rank + 6)
    toks = torch.as_tensor(prompt, dtype=torch.int32).to(dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            model.step_seq(toks, seq=0, offset=0, stream=stream)
    stream.synchronize()
    clocks = clocks_cls(bus)
    clocks.start()
    time.sleep(0.3)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    t_wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(reps):
            model.step_seq(toks, seq=0, offset=0, stream=stream)
            ev[i + 1].record(stream)
    ev[-1].synchronize()
    t_wall1 = time.perf_counter()
    ms = ev[0].elapsed_time(ev[-1]) / reps
    time.sleep(0.2)
    clocks.stop()
    err = model.error_word()
    if err:
        raise RuntimeError("device error word %d during the prompt timed region" % err)
    n_chunks = (prompt_len + rows - 1) // rows
    nq = cfg["n_qh"] * cfg["head_dim"]
    # the method's arithmetic: 2 flops per weight per token for the
    # projections, the head once, and q.K plus p.V over each causal prefix
    flops = (2.0 * cfg["n_layer"] * C.layer_params(cfg) * prompt_len + 2.0 * cfg["vocab"] * cfg["d"]
             + 4.0 * cfg["n_layer"] * nq * prompt_len * (prompt_len + 1) / 2)
    wbytes = C.weight_bytes_per_step(cfg)
    alg_bytes = n_chunks * (wbytes - cfg["vocab"] * cfg["d"] * 2) + cfg["vocab"] * cfg["d"] * 2 \
        + prompt_len * C.kv_bytes_per_token(cfg)
    hbm, kind = peaks()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tf_peak, tf_kind = float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        tf_peak, tf_kind = FALLBACK_BF16_TFLOPS, "fallback"
    sec = ms / 1e3
    out = {"workload": "llama3-8b-shape, one sequence, %d-token random prompt from position 0 in chunks of %d rows "
                       "(stepSeq on the batched path), last token's head + greedy pick, paged K/V pool of %d-position "
                       "blocks" % (prompt_len, rows, bt),
           "value": prompt_len / sec, "unit": "prompt tokens/s", "ms_per_prompt": ms, "reps": reps,
           "warmup": warmup, "chunks": n_chunks,
           "tensor_roofline": {"achieved": flops / sec / 1e12, "peak": tf_peak, "unit": "TFLOP/s",
                               "frac": flops / sec / 1e12 / tf_peak, "peak_source": tf_kind,
                               "algorithmic_flops": flops,
                               "note": "the projections multiply each fp32 activation as a bf16 pair hi + lo, so "
                                       "the tensor pipe executes twice these flops"},
           "hbm_roofline": {"achieved": alg_bytes / sec / 1e9, "peak": hbm, "unit": "GB/s",
                            "frac": alg_bytes / sec / 1e9 / hbm, "peak_source": kind,
                            "algorithmic_bytes": alg_bytes},
           "gpu_launches_per_prompt": n_chunks * (5 * cfg["n_layer"] + 3) + 3,
           "clocks": clocks.summary(t_wall0, t_wall1)}
    del model
    torch.cuda.empty_cache()
    return out


def op_inputs():
    """The op-level workload's seeded inputs (fp32 N(0,1) unless stated): GEMV
    matrices 4096 x 4096 and 4096 x 14336 (three copies each, rotated so
    every launch streams its matrix from HBM) with their vectors; residual
    add + RMSNorm over 4096 with weights N(1, 0.1); half-split RoPE on 32 q
    and 8 k heads of 128 at a position drawn uniform in [0, 8192), base 1e4;
    128,256 logits with the maximum planted at 3 random indices; one uniform
    draw for the sampler (temperature 0.8, top_k 50, top_p 0.95)."""
    import torch

    from autoregressive_decode_step_gb300 import synth

    d = {}
    for rows, cols in ((4096, 4096), (4096, 14336)):
        d["gemv", rows, cols] = ([synth.normal((rows * cols,), seed=rows + cols + i) for i in range(3)],
                                 synth.normal((rows,), seed=rows * 3 + 1))
    n = 4096
    d["norm"] = (synth.normal((n,), seed=1), synth.normal((n,), seed=2),
                 synth.normal((n,), seed=3, mean=1.0, std=0.1))
    d["rope"] = (int(torch.randint(0, 8192, (1,), generator=torch.Generator().manual_seed(0))),
                 synth.normal((32 * 128,), seed=10), synth.normal((8 * 128,), seed=20))
    # the output head of the 8B shape (bf16 [128,256][4096], 1.05 GB: larger
    # than L2) and its normalised input
    d["head"] = (synth.normal((128256, 4096), seed=50, std=0.02, dtype=torch.bfloat16), synth.normal((4096,), seed=51))
    # one decode step's attention at 8192 cached positions: 32 q heads over
    # 8 KV heads of 128, bf16 K/V (four caches of 33.6 MB rotated: larger
    # than L2 together)
    d["attn"] = ([(synth.normal((8192, 8 * 128), seed=60 + 2 * i, dtype=torch.bfloat16),
                   synth.normal((8192, 8 * 128), seed=61 + 2 * i, dtype=torch.bfloat16)) for i in range(4)],
                 synth.normal((32 * 128,), seed=70))
    V = 128256
    L = synth.normal((V,), seed=40)
    L[torch.randperm(V, generator=torch.Generator().manual_seed(41))[:3]] = float(L.max()) + 1.0
    d["logits"] = L
    d["u"] = synth.uniform_draws(1, seed=0)
    return d


OP_NAMES = ("gemv_transposed_4096x4096", "gemv_transposed_4096x14336", "gemv_head_128256x4096_bf16",
            "add_rmsnorm_4096", "rope_half_split_32q_8k_x128", "gqa_decode_attn_32q_8kv_x128_ctx8192_bf16",
            "greedy_argmax_128256", "sample_t0.8_k50_p0.95_128256")


def op_bytes():
    V = 128256
    return {"gemv_transposed_4096x4096": 4096 * 4096 * 4 + 4096 * 4 * 2,
            "gemv_transposed_4096x14336": 4096 * 14336 * 4 + (4096 + 14336) * 4,
            "gemv_head_128256x4096_bf16": 128256 * 4096 * 2 + 4096 * 4 + 128256 * 4,
            "gqa_decode_attn_32q_8kv_x128_ctx8192_bf16": 2 * 8192 * 8 * 128 * 2 + 2 * 32 * 128 * 4,
            "add_rmsnorm_4096": 5 * 4096 * 4,
            "rope_half_split_32q_8k_x128": 2 * 40 * 128 * 4,
            "greedy_argmax_128256": V * 4, "sample_t0.8_k50_p0.95_128256": V * 4}


def run_ops(dev, reps=200, warmup=5):
    """The decode glue one op at a time at the pages' op-level sizes, through
    the C ABI: each op's device time per launch, `reps` launches captured in
    a CUDA graph (after `warmup` eager launches) and the replay timed between
    CUDA events on the replaying stream (so the host's per-call cost is not
    in the number), and its algorithmic bytes over that time."""
    import torch

    from autoregressive_decode_step_gb300 import abi as A

    d = op_inputs()
    us = {}

    def gpu_us(fn):
        for i in range(warmup):
            fn(i)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(reps):
                fn(i)
        stream = torch.cuda.current_stream(dev)
        g.replay()
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        del g
        return e0.elapsed_time(e1) * 1e3 / reps

    for rows, cols in ((4096, 4096), (4096, 14336)):
        mats, x = d["gemv", rows, cols]
        mats_d = [m.to(dev) for m in mats]
        xd = x.to(dev)
        y = torch.empty(cols, device=dev)
        ws = A.workspace(A.ds_gemv_workspace_bytes(rows, cols, A.DS_F32), dev)
        us["gemv_transposed_%dx%d" % (rows, cols)] = gpu_us(
            lambda i: A.ds_gemv_transposed(mats_d[i % 3], xd, rows, cols, y, ws))
        del mats_d
        torch.cuda.empty_cache()
    W, x = (t.to(dev) for t in d["head"])
    y = torch.empty(128256, device=dev)
    us["gemv_head_128256x4096_bf16"] = gpu_us(lambda i: A.ds_gemv(W, x, 128256, 4096, y))
    del W
    torch.cuda.empty_cache()
    caches, q = d["attn"]
    caches = [(k.to(dev), v.to(dev)) for k, v in caches]
    q = q.to(dev)
    att = torch.empty(32 * 128, device=dev)
    lens = torch.tensor([8192], dtype=torch.int32, device=dev)
    ws = A.workspace(A.ds_attention_workspace_bytes(1, 32, 8, 128, 8192), dev)
    us["gqa_decode_attn_32q_8kv_x128_ctx8192_bf16"] = gpu_us(
        lambda i: A.ds_gqa_decode_attn(q, caches[i % 4][0], caches[i % 4][1], 8192, None, 512, 16, lens, 1, 32, 8,
                                       128, 1.0 / 128 ** 0.5, att, ws))
    del caches
    torch.cuda.empty_cache()
    r, x, w = (t.to(dev) for t in d["norm"])
    h = torch.empty(4096, device=dev)
    us["add_rmsnorm_4096"] = gpu_us(lambda i: A.ds_add_rmsnorm(r, x, w, 1e-5, h, 4096))
    pos, q, k = d["rope"]
    qd, kd = q.to(dev), k.to(dev)
    us["rope_half_split_32q_8k_x128"] = gpu_us(lambda i: A.ds_rope(qd, kd, pos, 32, 8, 128, 10000.0, 0))
    V = 128256
    Ld = d["logits"].to(dev)
    ids = torch.empty(1, dtype=torch.int32, device=dev)
    mx = torch.empty(1, device=dev)
    ws = A.workspace(A.ds_argmax_workspace_bytes(1, V), dev)
    us["greedy_argmax_128256"] = gpu_us(lambda i: A.ds_greedy_argmax(Ld, 1, V, ids, mx, ws))
    ud = d["u"].to(dev)
    ws = A.workspace(A.ds_sample_workspace_bytes(1, V), dev)
    us["sample_t0.8_k50_p0.95_128256"] = gpu_us(lambda i: A.ds_sample(Ld, 1, V, 0.8, 50, 0.95, ud, ids, ws))
    torch.cuda.synchronize()
    nb = op_bytes()
    return {"ops": {k: {"gpu_us": v, "gpu_gbs": nb[k] / (v * 1e-6) / 1e9, "algorithmic_bytes": nb[k]}
                    for k, v in us.items()},
            "reps": reps, "warmup": warmup,
            "workload": "op-level decode glue, fp32, seeded N(0,1) inputs at the pages' measured sizes; the "
                        "GEMVs rotate three weight copies and the attention four caches (larger than L2 together); "
                        "device time per launch from a replayed CUDA graph of the launches"}


def oracle_op_times(threads=None):
    """The oracle on the host cores (all of them, or `threads`) for the same
    ops and inputs as run_ops: best of at least 3 calls (and 0.2 s) per op,
    in microseconds."""
    import oracle as O

    from autoregressive_decode_step_gb300 import synth

    synth_np = synth.to_numpy_storage
    d = op_inputs()
    out = {}
    before = O.threads()
    if threads:
        O.set_threads(threads)

    def best_us(fn, min_calls=3, min_s=0.2):
        best, t_all, calls = float("inf"), 0.0, 0
        while calls < min_calls or t_all < min_s:
            t0 = time.perf_counter()
            fn()
            dt = time.perf_counter() - t0
            best, t_all, calls = min(best, dt), t_all + dt, calls + 1
        return best * 1e6

    for rows, cols in ((4096, 4096), (4096, 14336)):
        mats, x = d["gemv", rows, cols]
        a_np, x_np = mats[0].numpy(), x.double().numpy()
        out["gemv_transposed_%dx%d" % (rows, cols)] = best_us(
            lambda: O.gemv_transposed(a_np, x_np, rows, cols, O.DT_F32))
    W, x = d["head"]
    w_np, xh = synth_np(W), x.double().numpy()
    out["gemv_head_128256x4096_bf16"] = best_us(lambda: O.gemv(w_np, xh, 128256, 4096, O.DT_BF16), min_calls=1)
    caches, q = d["attn"]
    k_np, v_np, q_np = synth_np(caches[0][0]), synth_np(caches[0][1]), q.double().numpy()
    out["gqa_decode_attn_32q_8kv_x128_ctx8192_bf16"] = best_us(
        lambda: O.gqa_attention(q_np, k_np, v_np, O.DT_BF16, 8192, 32, 8, 128, 1.0 / 128 ** 0.5), min_calls=1)
    r, x, w = (t.numpy() for t in d["norm"])
    out["add_rmsnorm_4096"] = best_us(lambda: O.add_rmsnorm(r, x, w, 1e-5, O.DT_F32))
    pos, q, k = d["rope"]
    qn, kn = q.double().numpy(), k.double().numpy()
    out["rope_half_split_32q_8k_x128"] = best_us(
        lambda: (O.rope(qn, 32, 128, pos, 10000.0, 0), O.rope(kn, 8, 128, pos, 10000.0, 0)))
    Ln = d["logits"].numpy()
    out["greedy_argmax_128256"] = best_us(lambda: O.argmax(Ln))
    u0 = float(d["u"][0])
    out["sample_t0.8_k50_p0.95_128256"] = best_us(lambda: O.sample(Ln, 0.8, 50, 0.95, u0))
    if threads:
        O.set_threads(before)
    return out


def run_ours(args, rank, world, local):
    import torch

    from autoregressive_decode_step_gb300 import build as B
    B.build()
    from autoregressive_decode_step_gb300 import configs as C
    from autoregressive_decode_step_gb300 import synth
    from autoregressive_decode_step_gb300.model import DecodeModel

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.ops_only:
        if rank == 0:
            print(json.dumps({"ops": run_ops(dev, reps=args.ops_reps, warmup=min(5, args.ops_reps))}), flush=True)
        return 0
    cfg = dict(C.LLAMA3_8B)
    if args.layers is not None:
        cfg["n_layer"] = args.layers
    K, Wm = args.steps, args.warmup
    cap = args.ctx + max(Wm, K) + 8
    W = synth.model_weights(cfg, seed=0, device=dev)
    if args.batched_only or args.prompt_only:
        props = torch.cuda.get_device_properties(dev)
        bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), getattr(props, "pci_bus_id", 0),
                                    getattr(props, "pci_device_id", 0))
        line = {"metric": METRIC, "n_gpus": world, "data": "synthetic"}
        if args.batched_only:
            line["batched"] = run_batched(cfg, W, dev, rank, clocks_cls=ClockSampler, bus=bus,
                                          steps=args.batched_steps)
        if args.prompt_only:
            line["prompt_chunks"] = run_step_seq(cfg, W, dev, rank, clocks_cls=ClockSampler, bus=bus)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return 0
    model = DecodeModel(cfg, W, capacity=cap, device=dev, block_tokens=16)
    if args.kv_fill == "prefill":
        prompt = synth.prompt_ids(cfg, args.ctx, seed=rank)
        model.prefill(prompt)
        first = int(model.next_ids[0])
    else:
        ks, vs = synth.synthetic_kv(cfg, args.ctx, seed=rank + 1, device=dev)
        for l in range(cfg["n_layer"]):
            model.k_cache[l][:args.ctx].copy_(ks[l])
            model.v_cache[l][:args.ctx].copy_(vs[l])
        del ks, vs
        first = synth.prompt_ids(cfg, 1, seed=rank)[0]

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        replay = model.graph(advance=True, write_logits=False, stream=stream)

    def reset():
        model.set_state([first], [args.ctx])
        torch.cuda.synchronize()

    # ---------------- device-timed region: K graph replays
    reset()
    for _ in range(Wm):
        replay(stream)
    stream.synchronize()
    reset()
    props = torch.cuda.get_device_properties(dev)
    bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), getattr(props, "pci_bus_id", 0),
                                getattr(props, "pci_device_id", 0))
    clocks = ClockSampler(bus)
    clocks.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    chunks = []
    if args.chunk > 1:  # K steps as launches of up to `chunk` steps each
        left = K
        while left > 0:
            chunks.append(min(args.chunk, left))
            left -= chunks[-1]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    e0.record(stream)
    if chunks:
        for n in chunks:
            model.steps(n, stream=stream)
    else:
        for _ in range(K):
            replay(stream)
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.perf_counter()
    ms = e0.elapsed_time(e1)
    time.sleep(0.2)
    clocks.stop()
    err = model.error_word()
    if err:
        raise RuntimeError("device error word %d during the timed region" % err)
    ms_max = max_over_ranks(ms, world)
    step_ms = ms_max / K
    value = world * K / (ms_max / 1000.0)

    # ---------------- end to end: host token in, id out, every step
    tok_host = torch.empty(1, dtype=torch.int32, pin_memory=True)
    id_host = torch.empty(1, dtype=torch.int32, pin_memory=True)
    reset()
    tok_host[0] = first
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(K):
            model.tokens[:1].copy_(tok_host, non_blocking=True)
            replay(stream)
            id_host.copy_(model.next_ids[:1], non_blocking=True)
            stream.synchronize()
            tok_host[0] = id_host[0]
    t1 = time.perf_counter()
    e2e_s = max_over_ranks(t1 - t0, world)
    e2e_value = world * K / e2e_s

    # ---------------- per-op breakdown inside the step kernel: device
    # timestamps (globaltimer) at every phase boundary, a few untimed steps
    reset()
    names = []
    acc = {}
    n_pt = 8
    with torch.cuda.stream(stream):
        for _ in range(n_pt):
            model.step(advance=True, stream=stream, phase_times=True)
            for name, t in model.phase_times_us(stream=stream):
                if name not in acc:
                    names.append(name)
                    acc[name] = []
                acc[name].append(t)
    per_step = {k: sum(acc[k]) / n_pt for k in names}
    per_launch = {k: per_step[k] / (1 if k in ("embed", "head") else cfg["n_layer"]) for k in names}

    # the dominant (and only) kernel of the timed region is the persistent
    # step kernel: launches = chunks (or one per step), so its mean launch
    # duration is the CUDA-event time over the launches
    peak, peak_kind = peaks()
    n_launch = len(chunks) if chunks else K
    step_bytes = [C.step_bytes(cfg, args.ctx + i + 1) for i in range(K)]
    alg_bytes = sum(step_bytes) / n_launch
    launch_us = ms * 1000.0 / n_launch
    achieved = alg_bytes / (launch_us / 1e6) / 1e9
    ratio = traffic_ratio(kernel_source_sha()) if args.layers is None else None
    traffic = ratio * alg_bytes if ratio is not None else None
    per_launch_steps = sorted(set(chunks)) if chunks else [1]
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic,
                "kernel": "step_kernel: persistent cooperative decode step (all layers + head + argmax); %s greedy "
                          "step(s) per launch, %d launch(es), picks handed over on the device"
                          % ("/".join(str(c) for c in per_launch_steps), n_launch),
                "peak_source": peak_kind + " (MEASURED_PEAKS hbm_gbs copy)" if peak_kind == "measured" else peak_kind,
                "algorithmic_bytes_per_launch": alg_bytes,
                "algorithmic_bytes": "every weight byte once + K/V of every attended position",
                "traffic_source": "dram__bytes_read.sum + dram__bytes_write.sum over algorithmic bytes from "
                                  "profiles/step_kernel_llama3_8b.json, times this launch's algorithmic bytes"
                                  if traffic is not None else "no ncu record on the current kernel source",
                "mean_launch_us": launch_us}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": Wm,
            "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (random-init weights N(0,0.02), random prompt)",
            "config": dict(workload_config(args, cfg), kv_fill=args.kv_fill),
            "roofline": roofline,
            "frac_of_nominal_7900": achieved / NOMINAL_HBM_GBS,
            "per_op_us_per_launch": per_launch, "per_op_us_per_step": per_step,
            "per_op_source": "device phase timestamps inside the step kernel, mean of %d steps" % n_pt,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 4},
            "gpu_launches": n_launch,
            "clocks": clocks.summary(t_wall0, t_wall1)}
    del model
    torch.cuda.empty_cache()
    if args.layers is None and not args.no_batched:
        line["batched"] = run_batched(cfg, W, dev, rank, clocks_cls=ClockSampler, bus=bus,
                                      steps=args.batched_steps)
        try:
            line["prompt_chunks"] = run_step_seq(cfg, W, dev, rank, clocks_cls=ClockSampler, bus=bus)
        except Exception as e:  # reported in the line, never fatal to the step's numbers
            line["prompt_chunks"] = {"error": "%s: %s" % (type(e).__name__, e)}
    if args.layers is None and not args.no_legs:
        legs = {}
        for c in (4096, 8192):
            try:
                legs[str(c)] = run_batch1_leg(cfg, W, dev, c, K, Wm, args.chunk, kv_seed=rank + 11 + c)
                legs[str(c)]["workload"] = ("llama3-8b shape, batch-1 greedy decode, synthetic %d-position context "
                                            "(seeded N(0,1) K/V), %d decoded" % (c, K))
            except Exception as e:
                legs[str(c)] = {"error": "%s: %s" % (type(e).__name__, e)}
        line["context_legs"] = legs
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.layers is None:
        # the oracle as it stands, whole decode steps of the same model
        od = OracleDecoder(cfg, W, args.ctx, args.ctx + 8, seed=1)
        import oracle as O
        times = [od.step() for _ in range(3)]
        del od
        line["cpu_baseline"] = {"value": len(times) / sum(times), "unit": "tokens/s", "cores": O.threads(),
                                "kind": "oracle", "step_s": times,
                                "sample": "3 whole decode steps of the oracle (32 layers + head, greedy) at positions "
                                          "%d..%d over a synthetic %d-position context, on the same weights"
                                          % (args.ctx, args.ctx + 2, args.ctx)}
    del W
    torch.cuda.empty_cache()
    if args.layers is None and not args.no_legs:
        try:
            Q = C.QWEN3_0_6B
            Wq = synth.model_weights(Q, seed=0, device=dev)
            leg = run_batch1_leg(Q, Wq, dev, 512, 256, 32, 32, kv_seed=rank + 21,
                                 prompt=synth.prompt_ids(Q, 512, seed=rank + 22))
            leg["workload"] = ("qwen3-0.6b shape (28 layers, d 1024, 16q/8kv x 128, ff 3072, tied 151,936 head, bf16 "
                               "weights, fp32 K/V), batch-1 greedy decode, 512-token random prompt prefilled through "
                               "the decode step, 256 decoded")
            line["qwen3_0_6b"] = leg
            del Wq
            torch.cuda.empty_cache()
        except Exception as e:
            line["qwen3_0_6b"] = {"error": "%s: %s" % (type(e).__name__, e)}
        try:
            line["toy"] = run_toy_leg(dev)
        except Exception as e:
            line["toy"] = {"error": "%s: %s" % (type(e).__name__, e)}
    if args.layers is None and not args.no_ops:
        try:
            line["ops"] = run_ops(dev, reps=args.ops_reps)
        except Exception as e:  # reported in the line, never fatal to the step's numbers
            line["ops"] = {"error": "%s: %s" % (type(e).__name__, e)}
        if rank == 0 and world == 1 and not args.no_cpu_baseline and "ops" in line["ops"]:
            per_op = oracle_op_times()
            line.setdefault("cpu_baseline", {})["per_op_us"] = per_op
            line["cpu_baseline"]["per_op_us_one_core"] = oracle_op_times(threads=1)
            for k, v in line["ops"]["ops"].items():
                v["oracle_us"] = per_op[k]
                v["oracle_over_gpu"] = per_op[k] / v["gpu_us"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    rank, world, local = dist_init()
    if args.impl == "reference":
        rc = run_reference(args, rank, world)
    else:
        rc = run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
