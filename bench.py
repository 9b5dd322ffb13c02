#!/usr/bin/env python
"""Benchmark of one full-size MoE decode layer on GB300 (one JSON line).

Headline: microseconds per layer for the full-size layer at B = 1 (d=7168,
f=1536, 896 MXFP4 experts, top-16, bf16 shared expert, residual + RMSNorm
tail), event-timed on the device (by default with L2 not flushed between
steps: each step streams 360 MB of weights, 2.8x L2; --l2 flush flushes it,
and the line reports the other mode too), plus the achieved HBM bandwidth
against the bytes the layer must touch.  B = 8 and
B = 64 are reported in the same line under "batches".

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the plain fp64 statement of the layer)
on the host cores instead: that is this project's reference arm.
Multi-GPU (torchrun, one rank per GPU): independent replicas, no collective on
the data path; the reported time is the max over ranks.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "µs per MoE decode layer at B=1/8/64; achieved HBM TB/s vs GB300 peak"
DTYPE = "mxfp4(e2m1,e8m0) x f16 -> f32 routed; bf16 x bf16 -> f32 router/shared"
DATA = "synthetic: seeded Philox4x32-10 normal draws (no trained weights, no dataset)"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="full_b1")
    p.add_argument("--no-batches", action="store_true",
                   help="skip the B=8 / B=64 and four-layer chain extras")
    p.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline")
    p.add_argument("--profile-case", choices=sorted(PROFILE_CASES), default=None,
                   help="run --warmup untimed forwards of a profiling workload (--l2 between "
                        "them) and exit; for ncu captures, prints no JSON line")
    p.add_argument("--l2", choices=["none", "flush"], default="none",
                   help="between timed steps: none (every step streams its 360 MB of weights, "
                        "2.8x L2, so no weight byte is an L2 hit; code and the small "
                        "activations stay warm as in a decode loop over layers) or flush "
                        "(write 2x L2 first: code and activations cold too); the line "
                        "reports the B = 1 value in both modes")
    p.add_argument("--expert-path", type=int, choices=[0, 1, 2], default=0,
                   help="profiling workload only: 0 both expert paths (by batch), 1 mma.sync, "
                        "2 tcgen05")
    return p.parse_args()


# Profiling workloads.  "full_b1_e128" is the full_b1 layer with 128 experts
# held instead of 896 (2.2 GB of expert weights instead of 15.7 GB): at B = 1
# the 16 selected experts make its FC1 and FC2 launches the same size as
# full_b1's, while the device holds a few GB, as a many-pass capture needs.
PROFILE_CASES = {"full_b1": ("full_b1", None), "full_b1_e128": ("full_b1", 128),
                 "full_b8_e128": ("full_b8", 128), "full_b64_e128": ("full_b64", 128)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value, world, device=None):
    """Max of a float over ranks (identity at world size 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value, world, device=None):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def bytes_touched(cfg, n_distinct, B):
    """Algorithmic HBM bytes of one layer: touched experts + router + shared
    expert + gamma + activations (x read, residual read+write, out write)."""
    return (n_distinct * cfg.expert_bytes() + cfg.n_experts * cfg.d * 2 + 4 * cfg.n_experts
            + 3 * cfg.d * cfg.f_shared * 2 + 2 * cfg.d + 8 * B * cfg.d)


def fc1_bytes(cfg, n_distinct, B):
    """Algorithmic bytes of one FC1 launch: the shared expert's bf16 gate/up
    rows, the gate/up nibbles and scales of the touched experts, x read, and
    h_s and h written."""
    per_expert = 2 * cfg.f * cfg.d // 2 + 2 * cfg.f * cfg.d // 32
    shared = 2 * cfg.f_shared * cfg.d * 2
    return (shared + n_distinct * per_expert + 2 * B * cfg.d + 4 * B * cfg.f_shared
            + 4 * B * cfg.top_k * cfg.f)


def fc2_bytes(cfg, n_distinct, B):
    """Algorithmic bytes of FC2: the shared expert's bf16 down rows, the down
    nibbles and scales of the touched experts, h_s and h read, y_s and the
    per-pair outputs written."""
    per_expert = cfg.d * cfg.f // 2 + cfg.d * cfg.f // 32
    shared = cfg.d * cfg.f_shared * 2
    return (shared + n_distinct * per_expert + 4 * B * cfg.f_shared + 4 * B * cfg.top_k * cfg.f
            + 4 * B * cfg.d + 4 * B * cfg.top_k * cfg.d)


KERNEL_SOURCES = ("common.cuh", "stream.cuh", "moe_decode.cu")
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "roofline_traffic.json")


def kernel_source_sha256():
    """sha256 over the dominant B = 1 kernel's sources (helpers, the streaming
    kernel and its launch plan), concatenated in that order."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "moe_decode_step_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def traffic_from_profile():
    """DRAM bytes (read + write) per launch of the dominant kernel from the ncu
    record in profiles/roofline_traffic.json, scaled to the timed workload's
    distinct experts; None when missing or taken on other kernel sources."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha256") != kernel_source_sha256():
        return None
    return rec


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((num(r[3]) or 0.0) for r in rows)}


# ---------------------------------------------------------------------------
class L2Flush:
    """Evict L2 between timed steps: write a buffer of 2x L2, then read a second
    one, so no dirty lines from the flush are written back inside the timed
    region."""

    def __init__(self, device):
        import torch
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        self.w = torch.empty(2 * l2, dtype=torch.uint8, device=device)
        self.r = torch.ones(2 * l2 // 4, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)
        self.i = 0

    def __call__(self):
        import torch
        self.i += 1
        self.w.fill_(self.i & 0xFF)
        torch.sum(self.r, dim=0, out=self.sink)


L2_MODES = {"none": "not flushed: inputs larger than L2 (each step streams 360 MB of weights "
                    "at B = 1, 2.8x the 129 MB L2, so no weight byte survives in L2 to the next "
                    "step; per-step DRAM bytes from ncu in profiles/)",
            "flush": "flushed between timed steps (write of 2x L2 size)"}

SLEEP_CYCLES = 1_000_000   # ~0.5 ms head start so the host enqueues a whole forward
                           # (or graph launch) before the GPU reaches the start event


def time_layer(layer, x, res0, steps, warmup, flush, graph=True, timing=True):
    """Device time of one forward per step (CUDA events on the launching stream),
    flush() before every step.  graph=True replays a captured CUDA graph of
    the forward (the production mode: no host launch gaps); graph=False runs the
    eager forward.  Either way a sleep kernel runs before the start event, so
    that the host has submitted the whole step before the GPU reaches the event
    and the host's submission latency stays outside the device time.  Returns
    (us per step, per-phase us per step)."""
    import torch
    res = res0.clone()
    out = torch.empty_like(x)
    cur = torch.cuda.current_stream()
    layer.set_timing(timing)
    if graph:
        side = torch.cuda.Stream()
        side.wait_stream(cur)
        with torch.cuda.stream(side):
            layer.forward(x, res, out)
        cur.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            layer.forward(x, res, out)
        run = g.replay
    else:
        def run():
            layer.forward(x, res, out)
    for _ in range(warmup):
        res.copy_(res0)
        flush()
        run()
    torch.cuda.synchronize()
    times, phases = [], []
    for _ in range(steps):
        res.copy_(res0)
        flush()
        torch.cuda._sleep(SLEEP_CYCLES)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(cur)
        run()
        b.record(cur)
        b.synchronize()
        times.append(a.elapsed_time(b) * 1000.0)
        if timing:
            phases.append(layer.get_timing())
    layer.set_timing(False)
    if graph:
        del g
    return times, phases


def time_steps(layer, x, res0, steps, warmup):
    """Device time per step of `steps` forwards captured back to back in one
    CUDA graph, as the layer runs inside a decode step's graph (one graph
    launch for all of them, each forward chained to the next by programmatic
    dependent launch), timed once with CUDA events around the replay behind a
    sleep kernel; `warmup` single-forward replays run before it.  x stays, the
    residual carries from step to step.  Nothing can be flushed between the
    steps, so this is the L2 mode "none" only (inputs larger than L2)."""
    import torch
    res = res0.clone()
    out = torch.empty_like(x)
    cur = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        layer.forward(x, res, out)
    cur.wait_stream(side)
    torch.cuda.synchronize()
    g1 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g1):
        layer.forward(x, res, out)
    gk = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gk):
        for _ in range(steps):
            layer.forward(x, res, out)
    for _ in range(warmup):
        g1.replay()
    res.copy_(res0)
    torch.cuda.synchronize()
    torch.cuda._sleep(SLEEP_CYCLES)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(cur)
    gk.replay()
    b.record(cur)
    b.synchronize()
    us = a.elapsed_time(b) * 1000.0 / steps
    del gk, g1
    return us


def measure(layer, x, res0, steps, warmup, l2, l2flush):
    """The reported time of one forward in L2 mode `l2`, and the per-step
    times of single-forward graph replays (for the spread).  "none": `steps`
    forwards in one graph (time_steps), the single-forward replays run after
    it, outside the timed steps; "flush": the median of single-forward
    replays, L2 flushed before each."""
    import statistics
    if l2 == "none":
        us = time_steps(layer, x, res0, steps, warmup)
        single, _ = time_layer(layer, x, res0, steps, warmup, lambda: None, graph=True,
                               timing=False)
        return us, single
    single, _ = time_layer(layer, x, res0, steps, warmup, l2flush, graph=True, timing=False)
    return statistics.median(single), single


def time_chain(layers, x0, res0, steps, warmup, flush):
    """Device time of a chain of layers (each layer's out is the next one's x,
    the residual threads through), captured as one CUDA graph; flush() once
    before each chain, then a sleep kernel ahead of the start event (the host
    submits the graph launch meanwhile).  Returns per-chain microseconds."""
    import torch
    x = x0.clone()
    res = res0.clone()
    outs = [torch.empty_like(x0) for _ in layers]

    def chain():
        xi = x
        for L, o in zip(layers, outs):
            L.forward(xi, res, o)
            xi = o

    cur = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(cur)
    with torch.cuda.stream(side):
        chain()
    cur.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for _ in range(warmup):
        res.copy_(res0)
        flush()
        g.replay()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        res.copy_(res0)
        flush()
        torch.cuda._sleep(SLEEP_CYCLES)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(cur)
        g.replay()
        b.record(cur)
        b.synchronize()
        times.append(a.elapsed_time(b) * 1000.0)
    del g
    return times


def trace_layer(layer, x, res0, flush, reps=7):
    """Device timeline of eager forwards: per kernel, the earliest CTA start and
    the latest CTA end (globaltimer, us from the first kernel's start),
    flush() before each forward; the median of each over `reps` forwards."""
    import torch
    res = res0.clone()
    out = torch.empty_like(x)
    layer.set_trace(True)
    runs = []
    for _ in range(reps):
        res.copy_(res0)
        flush()
        torch.cuda._sleep(SLEEP_CYCLES)
        layer.forward(x, res, out)
        runs.append(layer.get_trace())
    layer.set_trace(False)
    return {k: [round(statistics.median(r[k][0] for r in runs), 2),
                round(statistics.median(r[k][1] for r in runs), 2)] for k in runs[0]}


def percentile(v, q):
    v = sorted(v)
    if not v:
        return None
    i = min(len(v) - 1, max(0, int(round(q / 100.0 * (len(v) - 1)))))
    return v[i]


def time_e2e(layer, cfg, x, res0, steps, warmup, flush):
    """The same layer through the host-buffer entry point: H2D of x and the
    residual, forward, D2H of residual and out, stream sync, per step, on a
    stream of the caller's with pinned buffers (the entry point's graph path)."""
    import torch
    xh = x.cpu().pin_memory()
    r0 = res0.cpu()
    rh = torch.empty_like(r0).pin_memory()
    oh = torch.empty_like(r0).pin_memory()
    st = torch.cuda.Stream()
    for _ in range(warmup):
        rh.copy_(r0)
        flush()
        torch.cuda.synchronize()
        layer.forward_host(xh, rh, oh, stream=st)
    times = []
    for i in range(steps):
        rh.copy_(r0)
        flush()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        layer.forward_host(xh, rh, oh, stream=st)
        times.append((time.perf_counter() - t0) * 1e6)
    nbytes = x.numel() * 2
    return times, 2 * nbytes, 2 * nbytes


def cpu_oracle_sample(cfg_name, repeats=1):
    """Time the CPU oracle on one full layer (layer compute only; drawing and
    MXFP4 packing of the weights are excluded)."""
    import gen
    import oracle
    from gen.configs import CONFIGS
    cfg = CONFIGS[cfg_name]
    inp = oracle.LayerInputs(cfg)
    for e in set(oracle.route(inp)[1].ravel().tolist()):
        inp.expert_packed(int(e))
    ts = []
    for _ in range(repeats):
        tm = {}
        oracle.forward(inp, timings=tm)
        ts.append(tm["compute_s"] * 1e6)
    return ts, gen.host_threads()


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from gen.configs import CONFIGS
    cfg = CONFIGS[args.config]
    # warm-up: draws and packing happen here (excluded from the timed steps)
    warm_ts, cores = cpu_oracle_sample(args.config, repeats=max(1, min(args.warmup, 1)))
    t0 = time.perf_counter()
    ts, _ = cpu_oracle_sample(args.config, repeats=args.steps)
    wall = time.perf_counter() - t0
    v = statistics.median(ts)
    sample = (f"{args.config}: one full layer per step (router over {cfg.n_experts} experts, "
              f"{cfg.top_k} MXFP4 experts, shared expert, tail) in fp64; weight draws and "
              "packing excluded")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "us", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1000.0,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": DATA,
            "config": {"workload": args.config, "B": cfg.B, "d": cfg.d, "f": cfg.f,
                       "n_experts": cfg.n_experts, "top_k": cfg.top_k, "f_shared": cfg.f_shared},
            "cpu_baseline": {"value": v, "unit": "us", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": wall}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, rank, world, local):
    import torch
    from gen.configs import CONFIGS
    from moe_decode_step_gb300 import synthetic

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    cfg = CONFIGS[args.config]
    peak, peak_kind = measured_peaks()
    l2flush = L2Flush(dev)
    flush = l2flush if args.l2 == "flush" else (lambda: None)

    layer = synthetic.make_layer(cfg)
    x, res0 = synthetic.make_activations(cfg)
    idx, _ = layer.router_topk(x)
    n_distinct = int(torch.unique(idx).numel())
    torch.cuda.synchronize()

    barrier(world)
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with ClockSampler(local) as clk:
        us_mode, times = measure(layer, x, res0, args.steps, args.warmup, args.l2, l2flush)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - wall0
    # the same forward in the other L2 mode, outside the timed region
    us_alt, _ = measure(layer, x, res0, args.steps, args.warmup,
                        "flush" if args.l2 == "none" else "none", l2flush)
    # per-phase events (graph nodes) on a separate set of replays: the event
    # nodes sit between the chained kernels, so they are kept out of the value
    _, phases = time_layer(layer, x, res0, max(5, args.steps // 2), max(3, args.warmup), flush,
                           graph=True, timing=True)
    # without a graph: the plain forward (no events between its kernels), and
    # separately the per-phase events, which break the programmatic chain
    eager_times, _ = time_layer(layer, x, res0, max(5, args.steps // 2), max(3, args.warmup),
                                flush, graph=False, timing=False)
    _, eager_phases = time_layer(layer, x, res0, max(5, args.steps // 2), max(3, args.warmup),
                                 flush, graph=False)

    us = reduce_max(us_mode, world, dev)
    us_alt = reduce_max(us_alt, world, dev)
    us_single = reduce_max(statistics.median(times), world, dev)
    btouch = bytes_touched(cfg, n_distinct, cfg.B)
    # one row on the mma.sync path runs FC1 and FC2 as one launch (four per
    # forward): that launch is the dominant kernel, with both steps' bytes
    fused = layer.launches_per_forward(cfg.B) == 4
    fc1_us = statistics.median(p[1] for p in phases)
    fc1_b = fc1_bytes(cfg, n_distinct, cfg.B)
    if fused:
        fc1_b += fc2_bytes(cfg, n_distinct, cfg.B)
    rec = traffic_from_profile()
    traffic = None
    if rec is not None:
        # the capture's launch moves the same bytes per touched expert
        traffic = (rec["dram_bytes_per_launch"] - rec["fixed_bytes"]) * n_distinct \
            / rec["n_distinct_experts"] + rec["fixed_bytes"]
    trace = trace_layer(layer, x, res0, flush)
    phase_names = ["router_topk", "fc1", "fc2", "unused", "tail", "layer"]
    phase_med = {n: statistics.median(p[i] for p in phases) for i, n in enumerate(phase_names)}

    e2e_times, h2d, d2h = time_e2e(layer, cfg, x, res0, max(5, args.steps // 2),
                                   max(3, args.warmup), flush)
    # f1: the routed experts on MXFP8 activations (the pages' FP4 x MXFP8
    # products), same layer and timing (the batches below report theirs)
    f1 = None
    if cfg.B == 1 and fused:
        layer.set_act_format(1)
        f1_mode, f1_times = measure(layer, x, res0, args.steps, args.warmup, args.l2, l2flush)
        layer.set_act_format(0)
        f1_us = reduce_max(f1_mode, world, dev)
        f1 = {"us": f1_us, "single_forward_us": statistics.median(f1_times),
              "p10_us": percentile(f1_times, 10), "steps": args.steps,
              "frac_of_peak": btouch / f1_us / 1e3 / peak,
              "activations": "x and h rounded to MXFP8 (E4M3, one E8M0 scale per 32) before "
                             "the MXFP4 products; parity against the oracle's mxfp8 mode"}
    e2e_us = reduce_max(statistics.median(e2e_times), world, dev)
    launches = layer.launches_per_forward(cfg.B) * args.steps
    layer.close()
    del layer

    batches = {}
    chain = None
    if not args.no_batches and args.config == "full_b1":
        for name in ("full_b8", "verify_b16", "full_b64"):
            c2 = CONFIGS[name]
            L2 = synthetic.make_layer(c2)
            x2, r2 = synthetic.make_activations(c2)
            i2, _ = L2.router_topk(x2)
            nd2 = int(torch.unique(i2).numel())
            st2 = max(5, args.steps)
            v2m, t2 = measure(L2, x2, r2, st2, max(3, args.warmup), args.l2, l2flush)
            _, p2 = time_layer(L2, x2, r2, 5, 3, flush, graph=True, timing=True)
            v2 = reduce_max(v2m, world, dev)
            b2 = bytes_touched(c2, nd2, c2.B)
            f2_us = statistics.median(p[1] for p in p2)
            f2_b = fc1_bytes(c2, nd2, c2.B)
            tr2 = trace_layer(L2, x2, r2, flush)
            # f1 on the same layer: the activation planes hold the MXFP8
            # roundings of x and h
            L2.set_act_format(1)
            f1m, f1t = measure(L2, x2, r2, st2, max(3, args.warmup), args.l2, l2flush)
            _, f1p = time_layer(L2, x2, r2, 5, 3, flush, graph=True, timing=True)
            L2.set_act_format(0)
            f1v = reduce_max(f1m, world, dev)
            f1_fc1 = statistics.median(p[1] for p in f1p)
            key = str(c2.B) if c2.drafts == 0 else (f"{c2.B} (rows in correlated groups of "
                                                       f"{1 + c2.drafts}, rho {c2.corr})")
            batches[key] = {
                "us": v2, "single_forward_us": statistics.median(t2), "steps": st2,
                "n_distinct_experts": nd2, "bytes_touched": b2,
                "hbm_tbs": b2 / v2 / 1e6, "frac_of_peak": b2 / v2 / 1e3 / peak,
                "expert_path": "tcgen05 block-scaled MXF4 MMA",
                "fc1_roofline": {"kernel": "tc_kernel (FC1: shared gate/up as a bf16 kind::f16 pass, "
                                           "routed gate/up as block-scaled kind::mxf4)", "bound": "hbm",
                                 "achieved": f2_b / f2_us / 1e3, "peak": peak, "unit": "GB/s",
                                 "frac": f2_b / f2_us / 1e3 / peak, "algorithmic_bytes": f2_b,
                                 "launch_us": f2_us, "peak_kind": peak_kind},
                "phases_us": {n: statistics.median(p[i] for p in p2)
                              for i, n in enumerate(phase_names)},
                "trace_us": tr2,
                "f1_mxfp8": {"us": f1v, "single_forward_us": statistics.median(f1t),
                             "frac_of_peak": b2 / f1v / 1e3 / peak,
                             "fc1_frac": f2_b / f1_fc1 / 1e3 / peak, "fc1_launch_us": f1_fc1,
                             "activations": "planes of the MXFP8 roundings of x and h (E4M3, "
                                            "one E8M0 scale per 32); parity against the "
                                            "oracle's mxfp8 mode"}}
            L2.close()
            del L2
            torch.cuda.empty_cache()
        # four chained full-size layers at B = 1 with the next-layer L2 prefetch
        cc = CONFIGS["chain4_b1"]
        chain_layers = [synthetic.make_layer(cc, layer=l) for l in range(cc.n_layers)]
        for l in range(cc.n_layers - 1):
            chain_layers[l].set_prefetch_next(chain_layers[l + 1])
        xc, rc = synthetic.make_activations(cc, layer=0)
        stc = max(5, args.steps)
        tc = time_chain(chain_layers, xc, rc, stc, max(3, args.warmup), flush)
        vc = reduce_max(statistics.median(tc), world, dev)
        # the same chain with the next-layer prefetch switched off
        for l in range(cc.n_layers - 1):
            chain_layers[l].set_prefetch_next(None)
        tc_off = time_chain(chain_layers, xc, rc, stc, max(3, args.warmup), flush)
        vc_off = reduce_max(statistics.median(tc_off), world, dev)
        chain = {"layers": cc.n_layers, "B": cc.B, "us": vc, "us_per_layer": vc / cc.n_layers,
                 "steps": stc, "l2": ("flushed once before each chain" if args.l2 == "flush"
                                      else "not flushed (63 GB of weights per chain)"),
                 "prefetch": "next layer's router weights into L2, issued by this layer's tail",
                 "us_prefetch_off": vc_off, "us_per_layer_prefetch_off": vc_off / cc.n_layers,
                 "prefetch_gain_us_per_layer": (vc_off - vc) / cc.n_layers}
        for L in chain_layers:
            L.close()
        del chain_layers
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        ts, cores = cpu_oracle_sample(args.config, repeats=10)
        cpu = {"value": statistics.median(ts), "unit": "us", "cores": cores, "kind": "oracle",
               "sample": f"{args.config}: one full layer (router, {cfg.top_k} MXFP4 experts, "
                         "shared expert, tail) in fp64; weight draws and packing excluded"}

    agg_tbs = reduce_sum(btouch / us / 1e6, world, dev)
    line = {
        "metric": METRIC, "value": us, "unit": "us", "n_gpus": world, "steps": args.steps,
        "p10_us": percentile(times, 10), "p90_us": percentile(times, 90),
        "single_forward_us": us_single,
        "warmup": args.warmup, "ms_per_step": us / 1000.0, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE, "data": DATA,
        "config": {"workload": f"{args.config}: one MoE decode layer, B={cfg.B}, d={cfg.d}, "
                               f"f={cfg.f}, E={cfg.n_experts}, top-{cfg.top_k}, MXFP4 experts, "
                               f"bf16 shared expert f={cfg.f_shared}, residual+RMSNorm tail",
                   "B": cfg.B, "l2": L2_MODES[args.l2],
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "hbm": {"bytes_touched": btouch, "n_distinct_experts": n_distinct,
                "tbs": btouch / us / 1e6, "frac_of_peak": btouch / us / 1e3 / peak,
                "frac_of_nominal_8tbs": btouch / us / 1e6 / 8.0, "aggregate_tbs": agg_tbs,
                "peak_gbs": peak, "peak_kind": peak_kind},
        "expert_path": "mma.sync with register dequantisation (B = 1)",
        "value_other_l2_mode": {"us": us_alt, "l2": L2_MODES["flush" if args.l2 == "none"
                                                              else "none"]},
        "roofline": {"kernel": ("stream_expert_kernel (FC1 + FC2 in one launch: shared and "
                                "routed gate/up, shared and routed down)") if fused else
                               "stream_dual_kernel (FC1: shared + routed gate/up)",
                     "bound": "hbm",
                     "achieved": fc1_b / fc1_us / 1e3, "peak": peak, "unit": "GB/s",
                     "frac": fc1_b / fc1_us / 1e3 / peak, "traffic": traffic,
                     "traffic_source": None if rec is None else rec.get("source"),
                     "algorithmic_bytes": fc1_b, "launch_us": fc1_us, "peak_kind": peak_kind},
        "phases_us": phase_med,
        "trace_us": trace,
        "timing_mode": (f"value: {args.steps} forwards captured back to back in one CUDA graph "
                        "(as inside a decode step's graph), one replay timed with CUDA events, "
                        "divided by the steps; single_forward_us, p10_us, p90_us: one forward "
                        "per graph replay, each timed alone (a one-kernel graph measures "
                        "~5 us between its events on this GPU)" if args.l2 == "none" else
                        "value: median of single-forward CUDA graph replays, L2 flushed before "
                        "each") + "; per-phase events as graph nodes on separate replays "
                                  "(phases_us)",
        "eager_us": statistics.median(eager_times),
        "eager_phases_us": {n: statistics.median(p[i] for p in eager_phases)
                            for i, n in enumerate(phase_names)},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_us, "unit": "us", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": launches,
        "clocks": clk.summary(),
        "f1_mxfp8": f1,
        "batches": batches,
        "chain": chain,
        "wall_s": wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_profile_case(args):
    import dataclasses
    import torch
    from gen.configs import CONFIGS
    from moe_decode_step_gb300 import synthetic

    base, n_experts = PROFILE_CASES[args.profile_case]
    cfg = CONFIGS[base]
    if n_experts is not None:
        cfg = dataclasses.replace(cfg, name=args.profile_case, n_experts=n_experts)
    dev = torch.device("cuda", 0)
    flush = L2Flush(dev) if args.l2 == "flush" else (lambda: None)
    layer = synthetic.make_layer(cfg, expert_path=args.expert_path)
    x, res0 = synthetic.make_activations(cfg)
    res = res0.clone()
    out = torch.empty_like(x)
    for _ in range(max(1, args.warmup)):
        res.copy_(res0)
        flush()
        layer.forward(x, res, out)
    torch.cuda.synchronize()
    rc = layer.status()
    layer.close()
    print(f"profile case {args.profile_case}: {max(1, args.warmup)} forwards, status {rc}")
    return 0 if rc == 0 else 1


def main():
    args = parse_args()
    if args.profile_case:
        return run_profile_case(args)
    rank, world, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
