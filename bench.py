"""Benchmark of the W12 hot path on one GB300 (or N independent replicas).

A step is one pass of a 27B-class dense decoder layer's six linears (q, k, v,
o, gate_up, down; hidden 5120) through the W12 decode-GEMM at M = 1 tokens,
weights and activations resident in HBM.  The layer's 511 MB of W12 weights
exceed the 129 MB L2, so every step streams them from HBM.  The headline
value is the effective weight-stream rate 1.5 B x K x N summed over the six
GEMMs / step time.  Alongside: the same through the public API with host
buffers (e2e), a sweep at M = 16 / 32 / 128, the fused lm_head verify step,
a cuBLAS BF16 GEMM of the same shapes, the dominant kernel's roofline, and
the CPU oracle on a bounded sample of the same workload.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl w12|reference]
Under torchrun each rank runs its own replica (the layer does not need any
exchange); rank 0 prints one JSON line.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from lossless_bit_weight_w12_gb300 import synth  # noqa: E402

METRIC = "W12 GEMM effective weight GB/s (% of GB300 HBM peak) at M=1/16/32"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e nominal
WORKLOAD = "27B-class dense decoder layer (q 5120->6144, k/v 5120->1024, o 6144->5120, " \
           "gate_up 5120->34816, down 17408->5120), W12 weights, M=1, seed 1"
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
DOMINANT = "gate_up"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _layer_bytes():
    return sum(synth.weight_bytes_w12(K, N) for _, K, N in synth.LAYER_SHAPES)


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while running (median SM clock, reasons)."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, interval_ms=200):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.path = None

    def start(self):
        import threading
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def pump():
            for line in self.proc.stdout:
                self.lines.append(line)
        self.thread = threading.Thread(target=pump, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            c = [x.strip() for x in line.split(",")]
            if len(c) < 9:
                continue
            try:
                sm.append(float(c[1]))
                smax = float(c[2])
            except ValueError:
                continue
            for nm, v in zip(names, c[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- setup

def build_layer(w12, dev, seed=1, M_list=(1,)):
    """Encode the layer's six weights (seed `seed` streams) and draw x per M."""
    import torch
    shapes = synth.LAYER_SHAPES
    rng = synth.streams(seed, len(shapes) + 8)
    layer = []
    for i, (name, K, N) in enumerate(shapes):
        w = synth.weights(rng[i], K, N)
        d, blob = w12.encode(w, w12.LAYOUT_NK)
        layer.append({"name": name, "K": K, "N": N, "desc": d, "blob": w12.upload(blob, dev),
                      "w_bf16": None, "w_np": w})
    xs = {}
    for M in M_list:
        xr = synth.streams(seed * 1000 + M, len(shapes))
        xs[M] = [torch.from_numpy(synth.activations(xr[i], M, K).view(np.int16)).to(dev)
                 for i, (_, K, _) in enumerate(shapes)]
    return layer, xs


def make_bufs(w12, dev, layer, M):
    import torch
    ys = [torch.empty((M, g["N"]), dtype=torch.float32, device=dev) for g in layer]
    wss = [w12.workspace(w12.gemm_workspace_size(g["desc"], M), dev) for g in layer]
    return ys, wss


def run_step(w12, layer, xs, ys, wss, mark=None):
    for i, g in enumerate(layer):
        done = mark(g["name"]) if mark is not None else None
        w12.gemm(g["desc"], g["blob"], xs[i], ys[i], wss[i], path=w12.OPT_EARLY_WEIGHTS)
        if done is not None:
            done()


def step_distribution(torch, fn, nbytes, n=100, seed=0):
    """n single steps, each between its own two events (eager launches):
    the median step time and a bootstrap 95 % interval of the median."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    torch.cuda.synchronize()
    for a, b in evs:
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    t = np.array([a.elapsed_time(b) / 1e3 for a, b in evs])
    med = float(np.median(t))
    boots = np.median(np.random.default_rng(seed).choice(t, size=(2000, n), replace=True), axis=1)
    lo, hi = np.percentile(boots, [2.5, 97.5])
    return {"n": n, "median_us": 1e6 * med, "ci95_us": [1e6 * float(lo), 1e6 * float(hi)],
            "min_us": 1e6 * float(t.min()), "gbs_at_median": nbytes / med / 1e9,
            "how": "single eager launches, each between two events; bootstrap of the median (2000 resamples)"}


def read_probe(torch, dev, gib=2, reps=10):
    """Read-only streaming reference next to the copy peak: a torch sum over
    `gib` GiB of float32 (each byte read once per pass)."""
    buf = torch.ones(gib << 28, dtype=torch.float32, device=dev)
    for _ in range(3):
        buf.sum()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        buf.sum()
    b.record()
    torch.cuda.synchronize()
    t = a.elapsed_time(b) / 1e3 / reps
    nbytes = buf.numel() * 4
    del buf
    return {"gbs": nbytes / t / 1e9, "bytes": nbytes, "kind": f"torch sum over {gib} GiB float32 (read-only stream)"}


def max_over_ranks(torch, seconds, world, device):
    """The slowest rank's time, on every rank (`seconds` itself at N = 1)."""
    if world == 1:
        return seconds
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_step, steps, world, seconds):
    """Whole-job throughput of N replicas: every rank's units over the
    slowest rank's time."""
    return world * units_per_step * steps / seconds


def time_steps(torch, fn, steps, barrier):
    """Eager timing: K calls of fn between two events on the current stream."""
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record()
    for _ in range(steps):
        fn()
    stop.record()
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(stop) / 1000.0  # seconds


def _timing_event(torch):
    """An event whose record becomes a node of a captured CUDA graph."""
    try:
        return torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:  # older torch: no external events
        return None


class GraphSteps:
    """`steps` repetitions of a step captured into one CUDA graph, with an
    event record node before and after every launch the step makes through
    `mark` (when the installed torch supports external events).  Replaying
    the graph once is one timed region of `steps` steps."""

    def __init__(self, torch, step, steps):
        self.torch = torch
        self.marks = []  # per step: list of (name, start event, end event)
        self.ok_events = _timing_event(torch) is not None
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step(lambda name: None)  # one eager pass on the capture stream (plans, attributes)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=s):
            for _ in range(steps):
                marks = []

                def mark(name, marks=marks):
                    if not self.ok_events:
                        return lambda: None
                    a, b = _timing_event(torch), _timing_event(torch)
                    a.record()
                    marks.append((name, a, b))
                    return b.record
                step(mark)
                self.marks.append(marks)

    def run(self, barrier):
        torch = self.torch
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        start.record()
        self.graph.replay()
        stop.record()
        torch.cuda.synchronize()
        barrier()
        return start.elapsed_time(stop) / 1000.0

    def per_launch(self):
        """Mean duration (s) of each marked launch over the replayed steps."""
        out = {}
        for marks in self.marks:
            for name, a, b in marks:
                out.setdefault(name, []).append(a.elapsed_time(b) / 1000.0)
        return {k: statistics.mean(v) for k, v in out.items()}


# The sources the stream kernel (the bench's dominant launch) is compiled
# from: a committed ncu capture counts only while these are unchanged.
STREAM_KERNEL_SOURCES = ("kernels_stream.cu", "stream_device.cuh", "stream_common.h", "async_common.cuh",
                         "gemm_common.cuh", "device_common.cuh", "verify_common.cuh", "w12_internal.h")


def kernel_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lossless_bit_weight_w12_gb300", "csrc")
    for name in sorted(STREAM_KERNEL_SOURCES):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(ROOT, "include", "w12.h"), "rb") as f:
        h.update(b"w12.h" + f.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_key):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            t = json.load(f)
        e = t[kernel_key]
        if e.get("kernel_hash") != kernel_hash():
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ----------------------------------------------------------------- CPU oracle

def oracle_prepare(every, seed=1, M=1, xseed=None, weights=None, parts=1):
    """The oracle's own encoding of every `every`-th column of each of the
    layer's six weights (seed `seed`, or the given [N, K] arrays), split
    into `parts` disjoint column ranges, with M activations drawn from the
    bench's stream for (xseed, M) (set-up, not timed).  Returns one work
    list per part: (desc, blob, x, weight-MACs)."""
    import oracle
    xseed = seed if xseed is None else xseed
    rng = synth.streams(seed, len(synth.LAYER_SHAPES) + 8)
    xr = synth.streams(xseed * 1000 + M, len(synth.LAYER_SHAPES))
    out = [[] for _ in range(parts)]
    for i, (name, K, N) in enumerate(synth.LAYER_SHAPES):
        w = weights[i] if weights is not None else synth.weights(rng[i], K, N)
        x = synth.activations(xr[i], M, K)
        cols = np.arange(0, N, every)
        for p, cp in enumerate(np.array_split(cols, parts)):
            if cp.size == 0:
                continue
            d, blob = oracle.encode(w[cp], oracle.LAYOUT_NK)
            out[p].append(("gemm", (d, blob, x), M * K * len(cp)))
    return out


def oracle_run(work, min_seconds=0.0):
    """Time the oracle over a work list in whole passes until at least
    `min_seconds` have elapsed (one pass at least).  Returns (units, seconds)
    where units are weight-MACs (GEMM items) or verifies."""
    import oracle
    t0 = time.perf_counter()
    n = 0
    while True:
        for kind, args, units in work:
            if kind == "gemm":
                oracle.gemm(*args)
            else:
                oracle.verify_greedy(*args)
            n += units
        dt = time.perf_counter() - t0
        if dt >= min_seconds:
            break
    return n, dt


def _oracle_proc(work, min_seconds, conn, go):
    """One host process of the all-core oracle timing."""
    sys.path.insert(0, ROOT)
    import oracle
    oracle.lib()
    oracle_run(work[:1])  # warm (page in the library and the data)
    conn.send("ready")
    go.wait()
    conn.send(oracle_run(work, min_seconds))
    conn.close()


def oracle_parallel(parts, min_seconds):
    """The oracle, as it stands, on len(parts) host processes at once (each
    on its own disjoint share of the work, started with spawn); the
    timed region runs from the common start to the last process's end.
    Returns (units, seconds)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    go = ctx.Event()
    procs, conns = [], []
    for work in parts:
        a, b = ctx.Pipe(duplex=False)
        p = ctx.Process(target=_oracle_proc, args=(work, min_seconds, b, go), daemon=True)
        p.start()
        procs.append(p)
        conns.append(a)
    for c in conns:
        assert c.recv() == "ready"
    t0 = time.perf_counter()
    go.set()
    res = [c.recv() for c in conns]
    wall = time.perf_counter() - t0
    for p in procs:
        p.join(timeout=30)
    return sum(n for n, _ in res), wall


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline_protocol(layer_w, seconds=2.5):
    """The oracle on the host's cores, 1 thread and all cores, on four
    workloads: config 0 (K = N = 1024, M = 1), a config-1 layer at M = 1
    (every 16th column of the six weights), a config-2 layer at M = 16 (the
    same weights and columns, seed-2 activations: the oracle's time depends
    only on the shapes; every 64th column), and config-4 verify on logits (R = 1, T = 16,
    V = 151936, fp32; all cores: independent verifies, one per process).
    GEMM rates are effective weight GB/s at 1.5 B per weight of the GEMM
    (1.5 K N per pass, whatever M); verify rates are verifies per second."""
    import oracle
    oracle.lib()
    cores = cpu_cores()
    out = {}

    def measure(name, parts_all, unit_scale, unit, what):
        n1, t1 = oracle_run(parts_all[0] if len(parts_all) == 1 else sum(parts_all, []), seconds)
        nall, tall = oracle_parallel(parts_all, seconds)
        out[name] = {"unit": unit, "what": what,
                     "threads_1": {"value": unit_scale(n1, t1), "units": n1, "seconds": t1},
                     "cores_all": {"value": unit_scale(nall, tall), "units": nall, "seconds": tall,
                                   "processes": len(parts_all)}}

    def gbs(M):
        return lambda n, t: 1.5 * n / M / t / 1e9

    # config 0
    r0 = synth.streams(0, 2)
    w0 = synth.weights(r0[0], 1024, 1024)
    x0 = synth.activations(r0[1], 1, 1024)
    parts0 = []
    for cp in np.array_split(np.arange(1024), cores):
        d, blob = oracle.encode(w0[cp], oracle.LAYOUT_NK)
        parts0.append([("gemm", (d, blob, x0), 1024 * len(cp))])
    measure("config0", parts0, gbs(1), "GB/s", "K=N=1024, M=1, every output")
    # config-1 layer, M = 1; config-2 layer, M = 16
    measure("config1_layer_m1", oracle_prepare(16, seed=1, M=1, weights=layer_w, parts=cores), gbs(1), "GB/s",
            "27B-class layer, M=1, every 16th column of each weight")
    measure("config2_layer_m16", oracle_prepare(64, seed=1, M=16, xseed=2, weights=layer_w, parts=cores),
            gbs(16), "GB/s", "27B-class layer, M=16 (seed-2 activations), every 64th column of each weight")
    # config-4 verify on logits
    r4 = synth.streams(4, 3)
    V, R, T = synth.LM_HEAD_SHAPE[2], 1, 16
    lg = synth.logits(r4[0], R * T, V)
    dr = synth.draft_tokens(r4[1], oracle.argmax(lg).reshape(R, T), R, T, V)
    measure("config4_verify_logits", [[("verify", (lg, R, T, dr), 1)] for _ in range(cores)],
            lambda n, t: n / t, "verifies/s", "R=1, T=16, V=151936 fp32 logits")
    return cores, out


# ----------------------------------------------------------------- arms

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    """The oracle as it stands, on all the host's cores (one process per
    core over disjoint column ranges), on a bounded sample of the same
    workload: each step the fp64 oracle GEMM on every 16th column of each of
    the six layer weights at M = 1."""
    world, rank, _ = dist_setup(args)
    if rank != 0:
        return
    from oracle import build as ob
    ob.build()
    every = 16
    cores = cpu_cores()
    parts = oracle_prepare(every, parts=cores)
    # warm-up steps (untimed), then K timed steps, each a bounded sample
    for _ in range(args.warmup):
        oracle_run(parts[0][:1])
    total_w, total_t = 0, 0.0
    for _ in range(args.steps):
        nw, dt = oracle_parallel(parts, 0.0)
        total_w += nw
        total_t += dt
    value = 1.5 * total_w / total_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * total_t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "sample": f"every {every}th column of each GEMM"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"fp64 oracle GEMM on every {every}th column of each of the "
                                   f"six layer weights, M=1, split over {cores} host processes; "
                                   f"{total_w // args.steps} weight-MACs per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_w12(args):
    import torch
    world, rank, local = dist_setup(args)
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")

        def barrier():
            dist.barrier()
    else:
        torch.cuda.set_device(0)

        def barrier():
            pass
    dev = torch.device("cuda", torch.cuda.current_device())
    from lossless_bit_weight_w12_gb300 import build_lib, w12
    build_lib.build()
    w12.lib()
    hbm_peak, peak_kind = _peaks()

    sweep_ms = (4, 16, 32, 64, 128)
    layer, xs = build_layer(w12, dev, seed=1, M_list=(1,) + sweep_ms)
    ys, wss = make_bufs(w12, dev, layer, 1)
    x1 = xs[1]
    nbytes = _layer_bytes()

    # ---- timed region: K steps in one CUDA graph; a step is ONE batched
    # launch over the six linears (stream-K over all their work units).  No
    # event nodes inside the graph: each step is exactly one kernel launch,
    # so the timed region / K is that kernel's mean launch duration (gaps
    # between launches included).
    descs = [g["desc"] for g in layer]
    blobs = [g["blob"] for g in layer]
    ws_b = w12.workspace(w12.gemm_batched_workspace_size(descs, 1), dev)
    # The layer's weights are written once, before the timed region, so the
    # early weight stream (W12_OPT_EARLY_WEIGHTS) is safe here and is what a
    # serving loop over resident weights uses.
    EARLY = w12.OPT_EARLY_WEIGHTS
    batch = w12.GemmBatch(descs, blobs, x1, ys, ws_b, EARLY)

    gsteps = GraphSteps(torch, lambda mark: batch(), args.steps)
    gwarm = GraphSteps(torch, lambda mark: batch(), args.warmup)
    gwarm.run(barrier)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    dt = gsteps.run(barrier)
    clk = clocks.stop()
    t_launch = dt / args.steps
    dt = max_over_ranks(torch, dt, world, dev)
    value = whole_job_rate(nbytes, args.steps, world, dt) / 1e9
    assert w12.get_device_error(ws_b) == 0
    del gsteps, gwarm

    # ---- steady state: the same step 10 000 times (25 replays of a graph of
    # 400 steps, each replay between two events) with the SM clock sampled
    # throughout, beyond the short timed region above
    long_steps, long_reps = 400, max(1, args.steady_steps // 400)
    glong = GraphSteps(torch, lambda mark: batch(), long_steps)
    glong.run(barrier)
    clk_long = ClockSampler(torch.cuda.current_device(), interval_ms=100)
    clk_long.start()
    reps = [glong.run(barrier) for _ in range(long_reps)]
    clk_l = clk_long.stop()
    del glong
    steady = {"steps": long_steps * long_reps, "seconds": sum(reps),
              "us_per_step_median_of_replays": 1e6 * statistics.median(reps) / long_steps,
              "us_per_step_min_max": [1e6 * min(reps) / long_steps, 1e6 * max(reps) / long_steps],
              "gbs": nbytes * long_steps * long_reps / sum(reps) / 1e9, "clocks": clk_l,
              "how": f"{long_reps} replays of a CUDA graph of {long_steps} steps, each between two events; "
                     "nvidia-smi sampled every 100 ms"}

    # ---- per-GEMM view: the six linears as six launches (informational)
    gsep = GraphSteps(torch, lambda mark: run_step(w12, layer, x1, ys, wss, mark), max(3, args.steps // 2))
    gsep.run(barrier)
    t_sep = gsep.run(barrier) / max(3, args.steps // 2)
    per_gemm = gsep.per_launch()
    del gsep
    for wsb in wss:
        assert w12.get_device_error(wsb) == 0

    # ---- e2e: through the public API with host buffers, copies inside.
    # Every step copies its six x from pinned host memory to the device (one
    # copy) and its six y back (one copy).  Two sets of device buffers and
    # three streams pipeline the steps: step i's host->device copy and step
    # i-1's device->host copy run under step i-1's / step i's weight stream;
    # events keep every buffer's reuse ordered.
    xsz = [x.numel() for x in x1]
    ysz = [y.numel() for y in ys]
    pin_x = torch.cat([x.reshape(-1) for x in x1]).cpu().pin_memory()
    pin_y = [torch.empty(sum(ysz), dtype=torch.float32).pin_memory() for _ in range(2)]
    xd_all = [torch.empty_like(pin_x, device=dev) for _ in range(2)]
    yd_all = [torch.empty(sum(ysz), dtype=torch.float32, device=dev) for _ in range(2)]
    yd = [[v.view(y.shape) for v, y in zip(torch.split(yd_all[k], ysz), ys)] for k in range(2)]
    batch_e2e = [w12.GemmBatch(descs, blobs, [v.view(x.shape) for v, x in zip(torch.split(xd_all[k], xsz), x1)],
                               yd[k], ws_b, EARLY) for k in range(2)]
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    x_free = [None, None]   # kernel k done reading xd[k]
    y_free = [None, None]   # copy-out of yd[k] done

    def e2e_steps(n):
        """n pipelined steps; returns after enqueueing (the compute stream
        waits for the last copy-out)."""
        for i in range(n):
            k = i & 1
            with torch.cuda.stream(s_in):
                if x_free[k] is not None:
                    s_in.wait_event(x_free[k])
                xd_all[k].copy_(pin_x, non_blocking=True)
                x_in = ev()
                x_in.record(s_in)
            s_comp.wait_event(x_in)
            if y_free[k] is not None:
                s_comp.wait_event(y_free[k])
            batch_e2e[k](s_comp)
            done = ev()
            done.record(s_comp)
            x_free[k] = done
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                pin_y[k].copy_(yd_all[k], non_blocking=True)
                out = ev()
                out.record(s_out)
            y_free[k] = out
        s_comp.wait_stream(s_out)

    def time_e2e(n):
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        start.record(s_comp)
        s_in.wait_stream(s_comp)
        e2e_steps(n)
        stop.record(s_comp)
        torch.cuda.synchronize()
        barrier()
        return start.elapsed_time(stop) / 1000.0
    e2e_steps(3)
    torch.cuda.synchronize()
    dt_e2e = max_over_ranks(torch, time_e2e(args.steps), world, dev)
    h2d = pin_x.numel() * pin_x.element_size()
    d2h = pin_y[0].numel() * pin_y[0].element_size()
    batch()
    torch.cuda.synchronize()
    last = (args.steps - 1) & 1
    for y_ref, y_e2e in zip(ys, torch.split(pin_y[last], ysz)):
        assert torch.equal(y_ref.cpu().reshape(-1), y_e2e), "e2e result differs from the device-resident run"

    # ---- the same step as single launches: median and its 95 % interval;
    # the bytes the step actually moves (unit blocks with their meta words,
    # escape lists, x, y); a read-only stream for reference
    per_step = step_distribution(torch, batch, nbytes)
    actual_bytes = (sum(int(d.total_bytes) for d in descs) + sum(x.numel() * 2 for x in x1)
                    + sum(y.numel() * 4 for y in ys))
    probe = read_probe(torch, dev) if rank == 0 else None

    # ---- sweep over M (same weights; inputs > L2): the AUTO path, and every
    # path that serves M (GEMV M <= 4, mma.sync, tcgen05), which shows where
    # the tensor-core tiles overtake the GEMV and tcgen05 overtakes mma.sync
    sweep, by_path = {}, {}
    path_names = {1: "gemv", 2: "mma_sync", 3: "tcgen05"}
    n = 40  # launches per graph; the median of three replays

    def time_layer(xsM, ysM, wsBM, path):
        bM = w12.GemmBatch(descs, blobs, xsM, ysM, wsBM, path | EARLY)
        gM = GraphSteps(torch, lambda mark: bM(), n)
        gM.run(barrier)
        t = statistics.median(gM.run(barrier) for _ in range(3))
        assert w12.get_device_error(wsBM) == 0
        return t
    for M in (1,) + sweep_ms:
        ysM = [torch.empty((M, g["N"]), dtype=torch.float32, device=dev) for g in layer]
        wsBM = w12.workspace(w12.gemm_batched_workspace_size(descs, M), dev)
        row = {}
        for path in (1, 2, 3):
            if path == 1 and M > 4:
                continue
            t = time_layer(xs[M], ysM, wsBM, path)
            row[path_names[path]] = round(1e6 * t / n, 2)
        by_path[str(M)] = row
        if M in sweep_ms:
            t = time_layer(xs[M], ysM, wsBM, 0)
            sweep[str(M)] = {"gbs": nbytes * n / t / 1e9, "us_per_layer": 1e6 * t / n,
                             "frac_of_peak": nbytes * n / t / 1e9 / hbm_peak}
        del ysM, wsBM

    # ---- cuBLAS BF16 GEMM on the same shapes (the 16-bit weight stream)
    bf16_rows = {}
    for M in (1, 16):
        wts = [torch.from_numpy(g["w_np"].view(np.int16)).to(dev).view(torch.bfloat16)
               for g in layer]
        xb = [x.view(torch.bfloat16) for x in xs[M]]

        def bf16_step(mark=None):
            for i in range(len(layer)):
                torch.nn.functional.linear(xb[i], wts[i])
        n = max(3, args.steps // 2)
        gb = GraphSteps(torch, bf16_step, n)
        gb.run(barrier)
        t = gb.run(barrier)
        del gb
        bf16_rows[str(M)] = {"us_per_layer": 1e6 * t / n,
                             "bf16_gbs": sum(2.0 * g["K"] * g["N"] for g in layer) * n / t / 1e9,
                             "w12_speedup": (t / n) / (dt / args.steps)}
        del wts

    # ---- fused lm_head verify (R = 1, T = 16) on the 5120 -> 151936 head
    verify = None
    if args.verify:
        verify = bench_lmhead(w12, torch, dev, args, barrier)

    # ---- the device encoder on the layer's largest matrix (gate_up, bf16
    # already in HBM): plan (bases, escape counts, scan, read-back) + pack
    enc = None
    gi = next(i for i, g in enumerate(layer) if g["name"] == "gate_up")
    w_dev = torch.from_numpy(layer[gi]["w_np"].view(np.int16)).to(dev)
    w12.encode_device(w_dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    reps = 3
    for _ in range(reps):
        d_enc, blob_enc = w12.encode_device(w_dev)
    torch.cuda.synchronize()
    t_enc = (time.perf_counter() - t0) / reps
    enc = {"matrix": "gate_up 5120x34816 (bf16 in HBM)", "ms": 1e3 * t_enc,
           "gweights_per_s": layer[gi]["K"] * layer[gi]["N"] / t_enc / 1e9,
           "bytes_equal_host_encoder": bool(torch.equal(blob_enc.cpu(), torch.from_numpy(
               w12.encode(layer[gi]["w_np"], w12.LAYOUT_NK)[1])))}
    codec = bench_codec(w12, torch, dev, layer, gi, d_enc, blob_enc, w_dev, barrier)
    del w_dev, blob_enc

    # ---- config 4 measured: 64 distinct layers + the fused lm_head verify
    stack = bench_stack(w12, torch, dev, args, barrier) if args.stack else None

    # ---- roofline of the dominant kernel: the step's single batched launch
    achieved = nbytes / t_launch / 1e9 if t_launch else None
    roofline = {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                "frac": achieved / hbm_peak if achieved else None,
                "traffic": traffic_for("stream_layer_m1"),
                "kernel": "stream_kernel<1,2,false,1>: the W12 GEMV (bulk-copied unit blocks, "
                          "CUDA-core bf16 FMA, warp-shuffle reduction) over the six layer linears "
                          "(one launch per step)",
                "peak_kind": f"{peak_kind} hbm_gbs (copy)",
                "algorithmic_bytes_per_launch": nbytes}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cores, wl = cpu_baseline_protocol([g["w_np"] for g in layer])
        head = wl["config1_layer_m1"]["cores_all"]
        cpu = {"value": head["value"], "unit": UNIT, "cores": cores, "kind": "oracle",
               "sample": "fp64 oracle GEMM on every 16th column of each of the six layer weights at "
                         f"M=1, {cores} host processes over disjoint column ranges, whole passes for "
                         f">= 2.5 s ({head['units']} weight-MACs in {head['seconds']:.1f} s); the "
                         "workloads below also on one thread",
               "workloads": wl}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "M": 1, "w12_bytes_per_step": nbytes,
                   "l2": "inputs larger than L2 (511 MB of W12 weights streamed per step)",
                   "launch": "W12_OPT_EARLY_WEIGHTS (weights resident, written before the timed region)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "frac_of_peak": value / world / hbm_peak,
        "frac_of_nominal": value / world / NOMINAL_HBM_GBS,
        "actual_bytes": {"per_step": actual_bytes, "gbs": actual_bytes / t_launch / 1e9,
                         "what": "unit blocks (planes + meta words) + escape lists + x + y"},
        "per_step_stats": per_step,
        "steady_state": steady,
        "read_probe": probe,
        "per_gemm_us": {k: 1e6 * v for k, v in per_gemm.items()},
        "unbatched_us_per_layer": 1e6 * t_sep,
        "timing": "K steps replayed from one CUDA graph (no event nodes inside); a step is one "
                  "batched launch; per-GEMM times from a separate unbatched graph with event nodes; "
                  "sweep and per-path rows: graphs of 40 launches, median of three replays",
        "e2e": {"value": whole_job_rate(nbytes, args.steps, world, dt_e2e) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "public API (w12_gemm_batched) with pinned host buffers; per step one host->device "
                       "copy of x and one device->host copy of y inside the timed region, pipelined over two "
                       "buffer sets (copy-in, compute and copy-out streams ordered by events); eager launches"},
        "gpu_launches": args.steps,
        "roofline": roofline,
        "sweep": sweep,
        "us_per_layer_by_path": by_path,
        "cublas_bf16": bf16_rows,
        "lmhead_verify": verify,
        "stack_m16": stack,
        "encode_device": enc,
        "codec_and_verify": codec,
        "cpu_baseline": cpu,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def accept_rule(g, draft):
    """The greedy acceptance rule on per-position target tokens g [R, T]
    and drafts [R, T - 1]: accept_len = the first position whose draft
    differs from g (T - 1 if none), next = g at that position."""
    g = np.asarray(g)
    R, T = g.shape
    miss = np.asarray(draft).reshape(R, T - 1) != g[:, :T - 1]
    acc = np.where(miss.any(axis=1), miss.argmax(axis=1), T - 1) if T > 1 else np.zeros(R, dtype=np.int64)
    return acc, g[np.arange(R), acc]


def bench_codec(w12, torch, dev, layer, gi, d, blob_dev, w_dev, barrier):
    """The other steps of the path, each against the measured copy bandwidth:
    the decode of gate_up's blob back to bf16 (1.5 B read + 2 B written per
    weight; checked equal to the original), the greedy verify on logits
    already in HBM (R = 1 and 8 draft blocks of T = 16 over V = 151936 fp32
    logits: 4 B read per logit), and the host encoder (OpenMP) on a layer
    matrix.  Device timings: graphs of 20 launches, best of three replays."""
    peak = _peaks()[0]
    K, N = layer[gi]["K"], layer[gi]["N"]

    def graph_time(step, n=20):
        g = GraphSteps(torch, lambda mark: step(), n)
        g.run(barrier)
        return min(g.run(barrier) for _ in range(3)) / n

    out = torch.empty((N, K), dtype=torch.int16, device=dev)
    t_dec = graph_time(lambda: w12.decode(d, blob_dev, out, w12.LAYOUT_NK))
    dec_bytes = 3.5 * K * N
    decode = {"matrix": f"gate_up {K}x{N}", "us": 1e6 * t_dec, "gbs": dec_bytes / t_dec / 1e9,
              "frac_of_peak": dec_bytes / t_dec / 1e9 / peak,
              "bytes_per_weight": "1.5 read + 2 written",
              "bit_exact": bool(torch.equal(out, w_dev))}
    del out

    R8, T, V = 8, 16, 151936
    rng = synth.streams(7, 2)
    lg = synth.logits(rng[0], R8 * T, V)
    drafts = synth.draft_tokens(rng[1], np.argmax(lg, axis=1).reshape(R8, T), R8, T, V)
    lg_d = torch.from_numpy(lg).to(dev)
    verify = {}
    for R in (1, R8):
        dr = torch.from_numpy(np.ascontiguousarray(drafts[:R])).to(dev)
        acc = torch.empty(R, dtype=torch.int32, device=dev)
        nxt = torch.empty(R, dtype=torch.int32, device=dev)
        ws = w12.workspace(w12.verify_workspace_size(R, T, V), dev)
        rows = lg_d[:R * T]
        t_v = graph_time(lambda: w12.verify_greedy(rows, R, T, dr, acc, nxt, ws))
        assert w12.get_device_error(ws) == 0
        vbytes = 4.0 * R * T * V
        verify[f"R{R}"] = {"rows": R * T, "us": 1e6 * t_v, "gbs": vbytes / t_v / 1e9,
                           "frac_of_peak": vbytes / t_v / 1e9 / peak}
    del lg_d

    q = next(g for g in layer if g["name"] == "q")
    w12.encode(q["w_np"], w12.LAYOUT_NK)
    t0 = time.perf_counter()
    reps = 3
    for _ in range(reps):
        w12.encode(q["w_np"], w12.LAYOUT_NK)
    t_host = (time.perf_counter() - t0) / reps
    host = {"matrix": f"q {q['K']}x{q['N']} (numpy bf16 bits on the host)", "ms": 1e3 * t_host,
            "gweights_per_s": q["K"] * q["N"] / t_host / 1e9, "threads": os.cpu_count()}
    return {"decode": decode, "verify_logits": verify, "encode_host": host,
            "how": "device rows: CUDA graphs of 20 launches, best of three replays"}


def bench_lmhead(w12, torch, dev, args, barrier):
    """Fused lm_head (5120 -> 151936) + greedy verify, T = 16 and R = 1, 2, 4,
    8 draft blocks (R*T = 16 .. 128 rows: the batched verify)."""
    K, N = synth.LM_HEAD_SHAPE[1], synth.LM_HEAD_SHAPE[2]
    T = 16
    rng = synth.streams(4, 3)
    w = synth.weights(rng[0], K, N)
    d, blob = w12.encode(w, w12.LAYOUT_NK)
    blob_d = w12.upload(blob, dev)
    b = synth.weight_bytes_w12(K, N)
    out = {}
    for R in (1, 2, 4, 8):
        hidden = torch.from_numpy(synth.activations(rng[1], R * T, K).view(np.int16)).to(dev)
        draft = torch.from_numpy(rng[2].integers(0, N, (R, T - 1)).astype(np.int32)).to(dev)
        acc = torch.empty(R, dtype=torch.int32, device=dev)
        nxt = torch.empty(R, dtype=torch.int32, device=dev)
        ws = w12.workspace(w12.verify_lmhead_workspace_size(d, R, T), dev)

        def step(mark=None):
            w12.verify_greedy_lmhead(hidden, d, blob_d, R, T, draft, acc, nxt, ws)
        n = max(5, args.steps)
        gl = GraphSteps(torch, step, n)
        gl.run(barrier)
        t = gl.run(barrier)
        assert w12.get_device_error(ws) == 0
        out[str(R * T)] = {"us": 1e6 * t / n, "gbs": b * n / t / 1e9, "R": R, "T": T}
    res = dict(out["16"])
    res.update({"N": N, "K": K, "by_rows": out})
    return res


def _stack_weight(task):
    """Worker (spawned process): one weight matrix of config 4 from its
    seed-4 stream, left in a shared-memory block for the parent."""
    from multiprocessing import resource_tracker, shared_memory
    sys.path.insert(0, ROOT)
    from lossless_bit_weight_w12_gb300 import synth as sy
    n_streams, idx, K, N = task
    w = sy.weights(sy.streams(4, n_streams)[idx], K, N)
    shm = shared_memory.SharedMemory(create=True, size=max(w.nbytes, 1))
    np.ndarray(w.shape, dtype=np.uint16, buffer=shm.buf)[:] = w
    resource_tracker.unregister(shm._name, "shared_memory")  # the parent unlinks it
    name = shm.name
    shm.close()
    return name, w.shape


def bench_stack(w12, torch, dev, args, barrier):
    """Config 4 measured on its stated data: 64 decoder layers (six W12
    linears each, one batched launch per layer) + the fused lm_head
    (5120 -> 151936) greedy verify, M = R*T = 16, every weight distinct and
    resident in HBM (33.9 GB of W12).  Every tensor is drawn from its seed-4
    stream as the config-4 test draws it (SeedSequence(4).spawn(64*6 + 4):
    layer l linear i -> 6l + i, lm_head -> 384, per-layer activations -> 385
    in order, hidden -> 386, drafts -> 387), the weights in spawned host
    processes and encoded on the device; the drafts follow the argmax of
    the float64 lm_head logits for a geometric(0.7) prefix.  One step = the
    65 launches, captured in a CUDA graph.  The step's (accept_len, next)
    is checked against the acceptance rule applied to the kernel's own
    logits."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    free, _ = torch.cuda.mem_get_info(dev)
    need = 64 * _layer_bytes() * 1.03 + synth.weight_bytes_w12(5120, 151936) * 1.03 + 4e9
    if free < need:
        return {"skipped": f"needs {need / 1e9:.0f} GB of device memory, {free / 1e9:.0f} GB free"}
    L, M, R, T = synth.N_LAYERS_STACK, 16, 1, 16
    shapes = synth.LAYER_SHAPES
    K_lm, N_lm = synth.LM_HEAD_SHAPE[1], synth.LM_HEAD_SHAPE[2]
    n_streams = 6 * L + 4
    tasks = [(n_streams, 6 * l + i, K, N) for l in range(L) for i, (_, K, N) in enumerate(shapes)]
    tasks.append((n_streams, 6 * L, K_lm, N_lm))
    t0 = time.perf_counter()
    encoded, w_lm = [], None
    with mp.get_context("spawn").Pool(max(1, min(cpu_cores(), 32))) as pool:
        for k, (name, shape) in enumerate(pool.imap(_stack_weight, tasks)):
            shm = shared_memory.SharedMemory(name=name)
            try:
                w = np.ndarray(shape, dtype=np.uint16, buffer=shm.buf)
                wd = torch.from_numpy(w.view(np.int16)).to(dev)
                if k == len(tasks) - 1:
                    w_lm = w.copy()
            finally:
                shm.close()
                shm.unlink()
            encoded.append(w12.encode_device(wd))
            del wd
    torch.cuda.synchronize()
    t_build = time.perf_counter() - t0
    layers = [([d for d, _ in encoded[6 * l:6 * l + 6]], [b for _, b in encoded[6 * l:6 * l + 6]])
              for l in range(L)]
    d_lm, b_lm = encoded[-1]
    rngs = synth.streams(4, n_streams)
    xs_l = []
    for l in range(L):
        xs_l.append([torch.from_numpy(synth.activations(rngs[6 * L + 1], M, K).view(np.int16)).to(dev)
                     for _, K, _ in shapes])
    ys = [torch.empty((M, N), dtype=torch.float32, device=dev) for _, _, N in shapes]
    ws = w12.workspace(w12.gemm_batched_workspace_size(layers[0][0], M), dev)
    batches = [w12.GemmBatch(dl, bl, xs_l[l], ys, ws, w12.OPT_EARLY_WEIGHTS) for l, (dl, bl) in enumerate(layers)]
    hidden = synth.activations(rngs[6 * L + 2], R * T, K_lm)
    # drafts: the float64 lm_head logits' argmax, geometric(0.7) prefix
    hf = (hidden.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    y64 = np.empty((R * T, N_lm), dtype=np.float64)
    for c0 in range(0, N_lm, 8192):
        wf = (w_lm[c0:c0 + 8192].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        y64[:, c0:c0 + 8192] = hf @ wf.T
    g64 = np.argmax(y64, axis=1).reshape(R, T)
    draft = synth.draft_tokens(rngs[6 * L + 3], g64, R, T, N_lm)
    del w_lm, y64
    hidden_d = torch.from_numpy(hidden.view(np.int16)).to(dev)
    draft_d = torch.from_numpy(draft).to(dev)
    acc = torch.empty(R, dtype=torch.int32, device=dev)
    nxt = torch.empty(R, dtype=torch.int32, device=dev)
    ws_lm = w12.workspace(w12.verify_lmhead_workspace_size(d_lm, R, T), dev)

    def step(mark=None):
        for bt in batches:
            bt()
        w12.verify_greedy_lmhead(hidden_d, d_lm, b_lm, R, T, draft_d, acc, nxt, ws_lm)
    n = 5
    gw = GraphSteps(torch, step, 2)
    gw.run(barrier)
    del gw
    g = GraphSteps(torch, step, n)
    g.run(barrier)
    t = g.run(barrier) / n
    assert w12.get_device_error(ws) == 0 and w12.get_device_error(ws_lm) == 0
    acc_step, nxt_step = acc.cpu().numpy().tolist(), nxt.cpu().numpy().tolist()
    # the same verify once more with the logits written out: the acceptance
    # rule on those logits (numpy argmax: lowest index of the maximum; the
    # GPU tests compare with the oracle) must give the step's (accept_len, next)
    logits = torch.empty((R * T, N_lm), dtype=torch.float32, device=dev)
    w12.verify_greedy_lmhead(hidden_d, d_lm, b_lm, R, T, draft_d, acc, nxt, ws_lm, logits_out_dev=logits)
    torch.cuda.synchronize()
    g32 = np.argmax(logits.cpu().numpy(), axis=1).reshape(R, T)
    want_acc, want_next = accept_rule(g32, draft)
    assert acc_step == want_acc.tolist() and nxt_step == want_next.tolist(), (acc_step, nxt_step)
    # positions whose argmax on the kernel's fp32 logits differs from the
    # float64 logits' (expected 0 outside near-ties)
    flips = int((g32.reshape(-1) != g64.reshape(-1)).sum())
    planted = int(np.argmax(draft[0] != g64[0, :T - 1])) if (draft[0] != g64[0, :T - 1]).any() else T - 1
    wbytes = 64 * _layer_bytes() + synth.weight_bytes_w12(K_lm, N_lm)
    res = {"us_per_step": 1e6 * t, "tokens_per_s": R * T / t, "gbs": wbytes / t / 1e9,
           "frac_of_peak": wbytes / t / 1e9 / _peaks()[0], "w12_weight_gb": wbytes / 1e9,
           "launches_per_step": 65, "build_s": t_build,
           "accept_len": acc_step, "next_token": nxt_step, "draft_prefix_of_fp64_argmax": planted,
           "argmax_flips_vs_fp64": flips,
           "verify_matches_rule_on_kernel_logits": True,
           "data": "seed-4 synth recipe (config 4 as stated): weights drawn in spawned host processes, "
                   "encoded on the device; drafts from the float64 lm_head argmax, geometric(0.7) prefix",
           "how": "64 batched layer launches + fused lm_head verify in one CUDA graph (W12_OPT_EARLY_WEIGHTS)"}
    del g, batches, layers, b_lm, encoded
    torch.cuda.empty_cache()
    return res


def run_kernel_only(args):
    """One GEMM of the layer (by name), or the whole layer as one batched
    launch ("layer"), at M = args.m with eager launches: the cases the ncu
    captures under profiles/ are taken on."""
    import torch
    from lossless_bit_weight_w12_gb300 import build_lib, w12
    build_lib.build()
    dev = torch.device("cuda", 0)
    if args.kernel_only == "layer":
        layer, xs = build_layer(w12, dev, seed=1, M_list=(args.m,))
        descs = [g["desc"] for g in layer]
        ys = [torch.empty((args.m, g["N"]), dtype=torch.float32, device=dev) for g in layer]
        ws = w12.workspace(w12.gemm_batched_workspace_size(descs, args.m), dev)
        b = w12.GemmBatch(descs, [g["blob"] for g in layer], xs[args.m], ys, ws, args.path | w12.OPT_EARLY_WEIGHTS)
        for _ in range(args.warmup):
            b()
        t = time_steps(torch, b, args.steps, lambda: None)
        assert w12.get_device_error(ws) == 0
        print(json.dumps({"kernel_only": "layer", "M": args.m, "path": args.path, "us": 1e6 * t / args.steps,
                          "gbs": _layer_bytes() * args.steps / t / 1e9}))
        return
    i, (name, K, N) = next((i, t) for i, t in enumerate(synth.LAYER_SHAPES) if t[0] == args.kernel_only)
    rng = synth.streams(1, len(synth.LAYER_SHAPES) + 8)
    d, blob = w12.encode(synth.weights(rng[i], K, N), w12.LAYOUT_NK)
    blob_d = w12.upload(blob, dev)
    xr = synth.streams(1000 + args.m, len(synth.LAYER_SHAPES))
    x = torch.from_numpy(synth.activations(xr[i], args.m, K).view(np.int16)).to(dev)
    y = torch.empty((args.m, N), dtype=torch.float32, device=dev)
    ws = w12.workspace(w12.gemm_workspace_size(d, args.m), dev)
    for _ in range(args.warmup):
        w12.gemm(d, blob_d, x, y, ws, path=args.path)
    t = time_steps(torch, lambda: w12.gemm(d, blob_d, x, y, ws, path=args.path), args.steps, lambda: None)
    print(json.dumps({"kernel_only": name, "K": K, "N": N, "M": args.m, "path": args.path,
                      "us": 1e6 * t / args.steps,
                      "gbs": synth.weight_bytes_w12(K, N) * args.steps / t / 1e9}))


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="w12", choices=["w12", "reference"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--no-verify", dest="verify", action="store_false")
    ap.add_argument("--no-stack", dest="stack", action="store_false",
                    help="skip the measured 64-layer stack (config 4)")
    ap.add_argument("--steady-steps", type=int, default=10000,
                    help="steps of the steady-state measurement (graphs of 400 steps)")
    ap.add_argument("--kernel-only", default=None, help="time one layer GEMM by name, or \"layer\" for the batched layer (for ncu)")
    ap.add_argument("--m", type=int, default=1, help="tokens for --kernel-only")
    ap.add_argument("--path", type=int, default=0,
                    help="--kernel-only: 0 auto, 1 GEMV, 2 mma.sync, 3 tcgen05")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    return args


def main():
    args = parse_args()
    if args.kernel_only:
        run_kernel_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_w12(args)


if __name__ == "__main__":
    main()
