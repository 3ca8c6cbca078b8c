"""Benchmark of the libreduce hot path on GB300.

One step runs every primitive once over its full-size synthetic workload:

  sum_1e9                 reduce_sum_f32   x[1e9]                uniform[0,1)  seed 42
  axis_128x4096x4095_d1   reduce_axis_f32  [128, 4096, 4095] d1  N(0,1)        seed 7
  axis_4096x65536_d1      reduce_axis_f32  [4096, 65536] d1      uniform[-1,1) seed 11
  axis_65536x4096_d0      reduce_axis_f32  [65536, 4096] d0      uniform[-1,1) seed 11
  rcumsum_32768x32768     reverse_cumsum   [32768, 32768]        uniform[0,1)  seed 3
  rcumsum_1x1e9           reverse_cumsum   [1, 1e9] (look-back)  uniform[0,1)  seed 3

The metric is effective HBM bandwidth: algorithmic bytes (every input read
once, every output written once) divided by device time, in GB/s, and as a
fraction of the measured HBM copy bandwidth.  Inputs are resident in HBM and
each is larger than L2 (>= 1 GiB), so no flush is needed between launches;
the small-n sweep of the 1D sum flushes L2 before every timed launch.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
        python bench.py --profile-case NAME [--steps K] [--warmup W]   (small case for ncu)
Under torchrun (N > 1) each rank runs the same step on its own GPU (replicas,
weak scaling); time is the max over ranks.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from reduction_scan_primitives_gb300 import inputs  # noqa: E402

METRIC = "effective HBM GB/s and % of GB300 peak per reduce/scan config (1 GPU)"
STEP_WORKLOADS = ["sum_1e9", "axis_128x4096x4095_d1", "axis_4096x65536_d1", "axis_65536x4096_d0",
                  "rcumsum_32768x32768", "rcumsum_1x1e9"]
# Follow-on forms, timed separately from the step (reported under next_rows).
NEXT_WORKLOADS = ["cumsum_fwd_32768x32768", "cumsum_fwd_excl_1x1e9", "cumsum_128x4096x4095_d1",
                  "cumsum_64x16384x1024_d1", "cumsum_2x8192x4096_d1", "cumsum_1024x8192x64_d1",
                  "sum_16x1000000x12_d1", "rcumsum_1x1e9_rts",
                  "max_1e9", "norm_128x4096x4095_d1", "mean_4096x65536_d1", "min_65536x4096_d0",
                  "rcumsum_1x1e9_ws", "axis_65536x4096_d0_ws", "rcumsum_2000000x100", "sum_4000000x32_d1",
                  "cumsum_100000x100x3_d1", "sum_100000x100x3_d1", "cumsum_4096x4096x2_d1",
                  "cumsum_1x40000000x4_d1", "cumsum_100000x100x16_d1"]
# Small cases of each kernel for ncu captures: larger than L2, a few GB at most.
PROFILE_CASES = {
    "sum_2e8": dict(op="sum", shape=(200_000_000,), dist="uniform01", seed=42),
    "axis_16x4096x4095_d1": dict(op="axis", shape=(16, 4096, 4095), dim=1, dist="normal", seed=7),
    "axis_4096x65536_d1": dict(inputs.WORKLOADS["axis_4096x65536_d1"]),
    "axis_65536x4096_d0": dict(inputs.WORKLOADS["axis_65536x4096_d0"]),
    "rcumsum_4096x32768": dict(op="rcumsum", shape=(4096, 32768), dist="uniform01", seed=3),
    "rcumsum_1x1e8": dict(op="rcumsum", shape=(1, 100_000_000), dist="uniform01", seed=3),
    "cumsum_16x4096x4095_d1": dict(op="cumsum", shape=(16, 4096, 4095), dim=1, reverse=False,
                                   exclusive=False, dist="normal", seed=7),
    "cumsum_16x4096x4096_d1": dict(op="cumsum", shape=(16, 4096, 4096), dim=1, reverse=True,
                                   exclusive=False, dist="uniform01", seed=3),
    "cumsum_256x8192x64_d1": dict(op="cumsum", shape=(256, 8192, 64), dim=1, reverse=False,
                                  exclusive=False, dist="uniform01", seed=13),
    "sum_16x1000000x12_d1": dict(inputs.WORKLOADS["sum_16x1000000x12_d1"]),
    "cumsum_2x8192x4096_d1": dict(inputs.WORKLOADS["cumsum_2x8192x4096_d1"]),
    "rcumsum_2000000x100": dict(inputs.WORKLOADS["rcumsum_2000000x100"]),
    "sum_4000000x32_d1": dict(inputs.WORKLOADS["sum_4000000x32_d1"]),
    "cumsum_100000x100x3_d1": dict(inputs.WORKLOADS["cumsum_100000x100x3_d1"]),
    "sum_100000x100x3_d1": dict(inputs.WORKLOADS["sum_100000x100x3_d1"]),
    "cumsum_4096x4096x2_d1": dict(inputs.WORKLOADS["cumsum_4096x4096x2_d1"]),
    "cumsum_1x40000000x4_d1": dict(inputs.WORKLOADS["cumsum_1x40000000x4_d1"]),
    "cumsum_40000x100x16_d1": dict(op="cumsum", shape=(40_000, 100, 16), dim=1, reverse=False,
                                   exclusive=False, dist="uniform01", seed=13),
    "sum_5000x1000x13_d1": dict(op="reduce", rop="sum", shape=(5000, 1000, 13), dim=1, dist="uniform_pm1", seed=13),
    "cumsum_1x10000000x16_d1": dict(op="cumsum", shape=(1, 10_000_000, 16), dim=1, reverse=False,
                                    exclusive=False, dist="uniform01", seed=13),
    "sum_1e5": dict(op="sum", shape=(100_000,), dist="uniform01", seed=42),
    "cumsum_500000x7x3_d1": dict(op="cumsum", shape=(500_000, 7, 3), dim=1, reverse=False,
                                 exclusive=False, dist="uniform01", seed=13),
    "cumsum_1x50000000x2_d1": dict(op="cumsum", shape=(1, 50_000_000, 2), dim=1, reverse=False,
                                   exclusive=False, dist="uniform01", seed=13),
}
FALLBACK_HBM_GBS = 6800.0
# Context only (another machine): the page's T4 figures for the 1D sum.
PAGES_T4 = {"sum_1e8_ms": 1.4716, "sum_1e9_ms": 14.4983}


# ---------------------------------------------------------------------------
# Distributed plumbing (timing only; no data-path collective).
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (the job time is the slowest rank's)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# Peaks, clocks, profiles.
# ---------------------------------------------------------------------------
def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def source_digest():
    """Digest of the kernel sources' code: comments and whitespace are left
    out, so a comment edit keeps the recorded counters valid."""
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(ROOT, "reduction_scan_primitives_gb300", "csrc", "*"))):
        with open(f, encoding="utf-8") as fh:
            code = fh.read()
        code = re.sub(r"/\*.*?\*/", " ", code, flags=re.S)
        code = re.sub(r"//[^\n]*", " ", code)
        h.update(os.path.basename(f).encode())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch from the committed ncu summary, keyed by workload,
    valid only while the kernel sources are unchanged since the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    if not os.path.exists(path):
        return out
    digest = source_digest()
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if len(parts) >= 3 and parts[2] == digest:
                out[parts[0]] = float(parts[1])
    return out


# ---------------------------------------------------------------------------
# Workloads.
# ---------------------------------------------------------------------------
def workload_spec(name):
    return inputs.WORKLOADS.get(name) or PROFILE_CASES[name]


def make_call(name, x, out):
    from reduction_scan_primitives_gb300 import libreduce as L
    w = workload_spec(name)
    if w["op"] == "sum":
        return lambda: L.reduce_sum_f32(x, out=out)
    if w["op"] == "axis":
        return lambda: L.reduce_axis_f32(x, w["dim"], out=out)
    if w.get("ws"):
        # Caller-provided scratch, sized by the query call and reused every step.
        if w["op"] == "cumsum":
            ws = L.workspace(L.cumsum_ws_f32(x, w["dim"], w["reverse"], w["exclusive"], out=out))
            return lambda: L.cumsum_ws_f32(x, w["dim"], w["reverse"], w["exclusive"], ws=ws, out=out)
        ws = L.workspace(L.reduce_axis_op_ws_f32(x, w["dim"], w["rop"], out=out))
        return lambda: L.reduce_axis_op_ws_f32(x, w["dim"], w["rop"], ws=ws, out=out)
    if w["op"] == "cumsum":
        return lambda: L.cumsum_f32(x, w["dim"], reverse=w["reverse"], exclusive=w["exclusive"], out=out)
    if w.get("strategy"):
        def call():  # the scan strategy is a library option: set for this call only
            L.set_option(L.OPT_SCAN_STRATEGY, w["strategy"])
            try:
                L.reverse_cumsum_f32(x, out=out)
            finally:
                L.set_option(L.OPT_SCAN_STRATEGY, 0)
        return call
    if w["op"] == "reduce":
        if "dim" in w:
            return lambda: L.reduce_axis_op_f32(x, w["dim"], w["rop"], out=out)
        return lambda: L.reduce_f32(x, w["rop"], out=out)
    return lambda: L.reverse_cumsum_f32(x, out=out)


def alloc_workload(name, device):
    w = workload_spec(name)
    x = inputs.make(w["shape"], w["dist"], w["seed"], device=device)
    if w["op"] == "sum" or (w["op"] == "reduce" and "dim" not in w):
        out = torch.empty((), dtype=torch.float32, device=device)
    elif w["op"] in ("axis", "reduce"):
        shp = list(w["shape"])
        del shp[w["dim"]]
        out = torch.empty(shp, dtype=torch.float32, device=device)
    else:
        out = torch.empty_like(x)
    return x, out


def time_next(device, reps=20):
    """The follow-on forms, each timed alone.

    ms_events: the median of CUDA events around single calls (back-to-back
    launches, inputs larger than L2); for calls of tens of microseconds this
    counts part of the host's launch gap.  For workloads of at most 2 GB per
    call, ms is the device time per call from one CUDA graph of calls that
    rotate over enough copies of the input and output (at least 4x L2 of
    traffic between two calls on the same copy), so no call finds its input
    in L2 and no host time is counted; otherwise ms is ms_events."""
    from reduction_scan_primitives_gb300 import libreduce as L
    peak, _ = hbm_peak()
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    res = {}
    for name in NEXT_WORKLOADS:
        x, out = alloc_workload(name, device)
        call = make_call(name, x, out)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in ev:
            a.record()
            call()
            b.record()
        torch.cuda.synchronize()
        L.check(device)
        ms_events = statistics.median(a.elapsed_time(b) for a, b in ev)
        nbytes = inputs.algorithmic_bytes(workload_spec(name))
        entry = {"ms_events": round(ms_events, 5)}
        ms = ms_events
        if nbytes <= 2 * 1024 ** 3:
            copies = max(2, -(-4 * l2 // nbytes))
            pairs = [(x, out)] + [alloc_workload(name, device) for _ in range(copies - 1)]
            calls = [make_call(name, xi, oi) for xi, oi in pairs] * max(1, 24 // copies)
            ms = _graph_per_launch_us(calls, device) * 1e-3
            L.check(device)
            entry.update({"graph_calls": len(calls), "copies": copies})
            del pairs, calls
        gbs = nbytes / (ms * 1e-3) / 1e9
        entry.update({"ms": round(ms, 5), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4), "bytes": nbytes})
        res[name] = entry
        del x, out
    return res


def _graph_per_launch_us(calls, device):
    """Device time per launch of `calls` (one graph, replayed after a warm
    replay), timed with CUDA events around the replay."""
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(side):
        for c in calls[:3]:
            c()
    torch.cuda.current_stream(device).wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for c in calls:
            c()
    g.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        b.synchronize()
        t = a.elapsed_time(b) * 1e3 / len(calls)
        best = t if best is None else min(best, t)
    del g
    return best


def time_sweep(device, reps=10):
    """1D sum sweep n = 1e4 .. 1e9, L2 cold for every launch.

    ms: CUDA events around one launch, after writing and reading a buffer
    larger than L2.  This GPU's event timestamps advance in steps of 2.048 us,
    and two events with nothing between them read about 2 us apart, so below
    ~1e7 elements this is coarse.  us_graph: for n <= 1e8, the same call
    captured K times in one CUDA graph, launch k reading slice k of a pool
    larger than 4x L2 (so no launch finds its input in L2), replayed and timed
    with events: device time per launch, no host cost and no event step.
    Applied up to 1e8 elements (whose single-launch time is still only ~30
    event steps).
    GB/s is taken from us_graph where present."""
    from reduction_scan_primitives_gb300 import libreduce as L
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    pool_floats = (5 * l2) // 4 + (1 << 20)
    res = {}
    peak, _ = hbm_peak()
    for n in inputs.SUM_SWEEP:
        x = inputs.make((n,), "uniform01", 42, device=device)
        out = torch.empty((), dtype=torch.float32, device=device)
        for _ in range(3):
            L.reduce_sum_f32(x, out=out)
        times = []
        for _ in range(reps):
            # Write a buffer larger than L2, then read it back so the dirty lines
            # are written out before the timed launch rather than during it.
            flush.fill_(1.0)
            flush.sum()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            L.reduce_sum_f32(x, out=out)
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        ms = statistics.median(times)
        entry = {"ms": round(ms, 5)}
        seconds = ms * 1e-3
        if n <= 100_000_000:
            k = max(8, -(-pool_floats // n))
            pool = torch.empty(k * n, dtype=torch.float32, device=device)
            pool.uniform_()
            outs = torch.empty(k, dtype=torch.float32, device=device)
            calls = [(lambda i=i: L.reduce_sum_f32(pool[i * n:(i + 1) * n], out=outs[i])) for i in range(k)]
            us = _graph_per_launch_us(calls, device)
            entry.update({"us_graph": round(us, 3), "graph_launches": k})
            seconds = us * 1e-6
            del pool, outs, calls
        gbs = (4 * n + 4) / seconds / 1e9
        entry.update({"GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)})
        res[str(n)] = entry
        del x
    del flush
    L.check(device)
    return res


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample of each workload.
# ---------------------------------------------------------------------------
def oracle_run(name, xs):
    """(callable running the oracle on the whole workload, its algorithmic bytes)."""
    import oracle
    w = workload_spec(name)
    if w["op"] == "sum":
        return (lambda: oracle.sum1d(xs)), 4 * xs.size + 4
    if w["op"] == "axis":
        o, r, i = inputs.canonical_axis(w["shape"], w["dim"])
        return (lambda: oracle.axis_sum(xs, o, r, i)), 4 * xs.size + 4 * o * i
    rows, n = w["shape"]
    return (lambda: oracle.reverse_cumsum(xs, rows, n)), 8 * xs.size


def threaded_run(name, xs):
    """The all-core fp64 baseline (cpu_baseline/) on the whole workload."""
    import cpu_baseline
    w = workload_spec(name)
    if w["op"] == "sum":
        return lambda: cpu_baseline.sum1d(xs)
    if w["op"] == "axis":
        o, r, i = inputs.canonical_axis(w["shape"], w["dim"])
        return lambda: cpu_baseline.axis_sum(xs, o, r, i)
    rows, n = w["shape"]
    return lambda: cpu_baseline.reverse_cumsum(xs, rows, n)


def cpu_baseline(data):
    """Two CPU figures over every workload of one step, once, on this host:
    the oracle (single-threaded fp64, the parity reference) and the all-core
    fp64 baseline (threads over independent outputs or row segments)."""
    import numpy as np

    import cpu_baseline as cb
    cb.build()
    total_bytes, t_oracle, t_threads = 0, 0.0, 0.0
    for name in STEP_WORKLOADS:
        xs = np.ascontiguousarray(data[name][0].cpu().numpy())
        fn, nbytes = oracle_run(name, xs)
        t0 = time.perf_counter()
        fn()
        t_oracle += time.perf_counter() - t0
        del fn
        fn = threaded_run(name, xs)
        t0 = time.perf_counter()
        fn()
        t_threads += time.perf_counter() - t0
        total_bytes += nbytes
        del fn, xs
    model = cb.cpu_model()
    return {"value": round(total_bytes / t_oracle / 1e9, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": "one step: every workload in full, once (host copy of the device inputs)",
            "seconds": round(t_oracle, 2), "cpu_model": model,
            "threaded": {"value": round(total_bytes / t_threads / 1e9, 3), "unit": "GB/s", "cores": cb.cores(),
                         "kind": "fp64 on every core (fp32 in and out; independent outputs or row "
                                 "segments per thread)", "seconds": round(t_threads, 3), "cpu_model": model}}


# ---------------------------------------------------------------------------
# Arms.
# ---------------------------------------------------------------------------
def run_ours(args):
    world, rank, local = dist_env()
    init_dist(world, "nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from reduction_scan_primitives_gb300 import build as lib_build
    from reduction_scan_primitives_gb300 import libreduce as L
    if rank == 0 or not os.path.exists(lib_build.LIB):
        lib_build.build()
    barrier(world)
    L.load()

    data = {name: alloc_workload(name, device) for name in STEP_WORKLOADS}
    calls = {name: make_call(name, *data[name]) for name in STEP_WORKLOADS}
    nbytes = {name: inputs.algorithmic_bytes(inputs.WORKLOADS[name]) for name in STEP_WORKLOADS}
    step_bytes = sum(nbytes.values())
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(device)
    ev = {name: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)] for name in STEP_WORKLOADS}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        for _ in range(args.warmup):
            for name in STEP_WORKLOADS:
                calls[name]()
        torch.cuda.synchronize()
        L.check(device)
        launches0 = L.launch_count()
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(args.steps):
            for name in STEP_WORKLOADS:
                a, b = ev[name][k]
                a.record(stream)
                calls[name]()
                b.record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    launches = L.launch_count() - launches0
    L.check(device)
    elapsed_ms = max_over_ranks(start.elapsed_time(stop), world, device)

    peak, peak_kind = hbm_peak()
    per = {}
    for name in STEP_WORKLOADS:
        t = [a.elapsed_time(b) for a, b in ev[name]]
        mean = sum(t) / len(t)
        gbs = nbytes[name] / (mean * 1e-3) / 1e9
        per[name] = {"ms_mean": round(mean, 5), "ms_median": round(statistics.median(t), 5),
                     "ms_min": round(min(t), 5), "GB/s": round(gbs, 1),
                     "frac": round(gbs / peak, 4), "bytes": nbytes[name]}
    total_kernel_ms = sum(per[n]["ms_mean"] for n in STEP_WORKLOADS)
    for name in STEP_WORKLOADS:
        per[name]["share"] = round(per[name]["ms_mean"] / total_kernel_ms, 4)
    dom = max(STEP_WORKLOADS, key=lambda n: per[n]["ms_mean"])
    traffic = recorded_traffic()
    roofline = {"bound": "hbm", "kernel": dom, "achieved": per[dom]["GB/s"], "peak": peak,
                "unit": "GB/s", "frac": per[dom]["frac"], "peak_kind": f"of {peak_kind}",
                "traffic": traffic.get(dom)}

    ms_per_step = elapsed_ms / args.steps
    value = step_bytes * args.steps * world / (elapsed_ms * 1e-3) / 1e9

    e2e = run_e2e(args, data, nbytes, device, world) if not args.no_e2e else None
    sweep = time_sweep(device) if (rank == 0 and not args.no_sweep) else None
    nxt = time_next(device) if (rank == 0 and not args.no_next) else None
    cpu = cpu_baseline(data) if (rank == 0 and world == 1 and not args.no_cpu) else None

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded torch generators on the device)",
            "config": {"workload": "one pass of: " + ", ".join(STEP_WORKLOADS),
                       "step_bytes": step_bytes, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2 (each >= 1 GiB); sweep flushes L2"},
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks.summary(), "per_config": per, "sum_sweep": sweep, "next_rows": nxt,
            "pages_context_t4": PAGES_T4,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(args, data, nbytes, device, world):
    """Same metric through the public API with host buffers: every step copies
    each input from pinned host memory, runs the call, copies the result back.
    Three streams, as a user would pipeline it: workload k+1's input copy and
    workload k-1's result copy overlap workload k's call (the two copy
    directions run at once); events order every buffer's reuse."""
    from reduction_scan_primitives_gb300 import libreduce as L
    host_in, host_out = {}, {}
    h2d = d2h = 0
    for name in STEP_WORKLOADS:
        x, out = data[name]
        host_in[name] = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        host_in[name].copy_(x)
        host_out[name] = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h2d += x.numel() * 4
        d2h += out.numel() * 4
    s_in, s_run, s_out = (torch.cuda.Stream(device) for _ in range(3))
    ev = {(k, name): torch.cuda.Event() for k in ("in", "run", "out") for name in STEP_WORKLOADS}
    steps = max(1, min(args.steps, 5))
    first = [True]

    def step():
        for name in STEP_WORKLOADS:
            x, out = data[name]
            with torch.cuda.stream(s_in):
                if not first[0]:
                    s_in.wait_event(ev[("run", name)])  # the last call on x is done
                x.copy_(host_in[name], non_blocking=True)
                ev[("in", name)].record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(ev[("in", name)])
                if not first[0]:
                    s_run.wait_event(ev[("out", name)])  # the last result has left
                make_call(name, x, out)()
                ev[("run", name)].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev[("run", name)])
                host_out[name].copy_(out, non_blocking=True)
                ev[("out", name)].record(s_out)
        first[0] = False

    step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(steps):
        step()
    torch.cuda.synchronize()
    ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world, device)
    L.check(device)
    value = sum(nbytes.values()) * steps * world / (ms * 1e-3) / 1e9
    return {"value": round(value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": steps, "ms_per_step": round(ms / steps, 3),
            "timing": "host clock around the steps (three streams: copy in, call, copy out)"}


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on bounded samples."""
    world, rank, local = dist_env()
    if rank != 0:
        return
    import numpy as np  # noqa: F401
    samples = {}
    for name in STEP_WORKLOADS:
        w = inputs.WORKLOADS[name]
        # The same recipe on the CPU generator; the sample is a slice of the
        # workload's leading rows / elements.
        shape = list(w["shape"])
        lead = {"sum": 25_000_000}.get(w["op"])
        if w["op"] == "sum":
            shape = [lead]
        elif w["op"] == "axis":
            o, r, i = inputs.canonical_axis(w["shape"], w["dim"])
            shape = [max(1, o // 128), r, i] if o > 1 and i > 1 else (
                [max(1, o // 64), r, i] if o > 1 else [1, max(1, r // 64), i])
        elif shape[0] >= 128:
            shape = [shape[0] // 128, shape[1]]
        else:
            shape = [shape[0], max(1, shape[1] // 128)]
        samples[name] = inputs.make(tuple(shape), w["dist"], w["seed"]).numpy()
    import oracle

    def one(name):
        w = inputs.WORKLOADS[name]
        x = samples[name]
        if w["op"] == "sum":
            oracle.sum1d(x)
            return 4 * x.size + 4
        if w["op"] == "axis":
            o, r, i = x.shape
            oracle.axis_sum(x, o, r, i)
            return 4 * x.size + 4 * o * i
        rows, n = x.shape
        oracle.reverse_cumsum(x, rows, n)
        return 8 * x.size

    for _ in range(args.warmup):
        for name in STEP_WORKLOADS:
            one(name)
    t0 = time.perf_counter()
    total = 0
    for _ in range(args.steps):
        for name in STEP_WORKLOADS:
            total += one(name)
    dt = time.perf_counter() - t0
    value = total / dt / 1e9
    sample = "; ".join(f"{n}: {list(samples[n].shape)}" for n in STEP_WORKLOADS)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": "one pass of: " + ", ".join(STEP_WORKLOADS) + " (bounded samples)"},
            "cpu_baseline": {"value": round(value, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile_case(args):
    """Run one small case a few times (for an ncu capture of its kernel)."""
    from reduction_scan_primitives_gb300 import build as lib_build
    from reduction_scan_primitives_gb300 import libreduce as L
    lib_build.build()
    L.load()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    x, out = alloc_workload(args.profile_case, device)
    call = make_call(args.profile_case, x, out)
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    L.check(device)
    print(json.dumps({"profile_case": args.profile_case, "launches": args.warmup + args.steps,
                      "bytes": inputs.algorithmic_bytes(workload_spec(args.profile_case))}))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-next", action="store_true", help="skip the follow-on forms")
    ap.add_argument("--profile-case", choices=sorted(PROFILE_CASES))
    args = ap.parse_args(argv)
    if args.profile_case:
        run_profile_case(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        print("bench: --warmup raised to 3 (minimum)", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
