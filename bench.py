#!/usr/bin/env python3
"""Benchmark of the per-row FP32 reduction library on GB300.

One step = one call of the headline operator (RMSNorm, FP32) over one
rows x cols matrix, through the C ABI.  Default workload: RMSNorm 1024x4096,
x ~ N(0,1) with 1% outliers x100, weight ~ 1 + 0.1 N(0,1), eps = 1e-6.

Device timing: exactly K timed steps run back to back on one stream,
replayed from CUDA graphs of captured library calls (so host launch cost is
not in the number), bracketed by CUDA events with a synchronize (and, for
N > 1, a barrier) on both sides.  One untimed replay is enqueued ahead of the
start event, so the host's graph-launch latency is not in the timed region
either.  Consecutive steps cycle through a pool of input / output buffers at
least 4x the L2 size, so no step finds its input in L2.  `value` =
algorithmic bytes moved per step x steps / time, in GB/s (the HBM-bandwidth
form of the metric; `us_per_op` gives the time form).

Output.  The LAST line on stdout is one compact JSON object, the headline
(at most HEADLINE_MAX_BYTES bytes), carrying the keys a reader needs:
value, roofline, e2e (with its host-link ceiling), clocks, the per-round
median, the copy/empty-kernel floor and the CPU baseline.  Everything else
(the sweep over every published shape and operator, the same-buffer "hot"
number, plain launches, PyTorch's own kernels as context) goes to stderr as
a table, and to --details FILE as JSON.

`--impl reference` times the CPU oracle instead, on a bounded row sample of
the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from row_reduction_gb300.timing import (  # noqa: E402
    MAX_ONE_GRAPH_STEPS, CopyProbe, EmptyProbe, ReadProbe, Workload,
    algorithmic_bytes, time_e2e, time_graph_steps, time_link,
    time_plain_steps, time_rounds)

METRIC = ("RMSNorm FP32 µs/op and HBM GB/s (% of GB300 peak), "
          "1×127 … 1024×4096")
FALLBACK_HBM_GBS = 6800.0
DATASHEET_HBM_GBS = 7900.0   # GB300 HBM3e nominal, for context only
HEADLINE_MAX_BYTES = 1536
# Fields the headline gives up, in this order, if it would exceed
# HEADLINE_MAX_BYTES (long plan strings, every throttle reason): all of them
# stay in the --details file.
HEADLINE_OPTIONAL = (("cpu_baseline", "cpu"), ("config", "l2"),
                     ("roofline", "peak_source"), ("rounds_us",),
                     ("floor",), ("e2e", "us_per_step"))
H_OUT_OPS = ("residual_layernorm", "residual_rmsnorm")
# Operators with one input matrix x and one output matrix y of its shape:
# the copy floor moves exactly their matrix bytes.  Operators that read x
# and write one value per row: the read floor.
COPY_FLOOR_OPS = ("rmsnorm", "layernorm", "softmax", "log_softmax")
READ_FLOOR_OPS = ("row_sum", "cross_entropy")
_OUTL = "with 1% x100 outliers"
INPUT_RECIPE = {
    "rmsnorm": f"x~N(0,1) {_OUTL}, weight~1+0.1N(0,1), eps=1e-6",
    "residual_rmsnorm": f"x~N(0,1) {_OUTL}, residual~N(0,1), "
                        "weight~1+0.1N(0,1), eps=1e-6, h_out written",
    "layernorm": f"x~N(0,1) {_OUTL}, gamma~1+0.1N(0,1), beta~0.1N(0,1), "
                 "eps=1e-5",
    "residual_layernorm": f"x~N(0,1) {_OUTL}, residual~N(0,1), "
                          "gamma~1+0.1N(0,1), beta~0.1N(0,1), eps=1e-5, "
                          "h_out written",
    "softmax": f"x~N(0,4) {_OUTL}",
    "log_softmax": f"x~N(0,4) {_OUTL}",
    "row_sum": f"x~N(0,1) {_OUTL}",
    "cross_entropy": f"logits~N(0,4) {_OUTL}, labels uniform in [0, cols), "
                     "per-row loss and mean",
}


# ---------------------------------------------------------------- helpers
def max_over_ranks(elapsed, device):
    """The slowest rank's elapsed seconds (all ranks get the same value)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([elapsed], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_step, steps, elapsed, world):
    """Whole-job GB/s: every rank moves bytes_per_step per step (replicas,
    weak scaling); time is the slowest rank's."""
    return world * bytes_per_step * steps / elapsed / 1e9


def sig(x, digits=6):
    """x rounded to `digits` significant digits (None stays None)."""
    if x is None or x == 0 or not math.isfinite(x):
        return x
    return float(f"{x:.{digits}g}")


def plan_text(op, rows, cols, dtype="f32"):
    import row_reduction_gb300 as mt
    return mt.mt_describe_plan(mt.mt_plan_query_dtype(op, dtype, rows, cols))


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_sources_sha(op="rmsnorm", plan=None, dtype="f32"):
    """Hash of what defines one operator's kernel: the kernel templates, the
    launch code, that operator's translation unit for the storage type and
    its plan."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_reduction_gb300", "csrc")
    for name in ("mt_kernels.cuh", "mt_stage.cuh", "mt_internal.h",
                 "api.cpp", f"ops_{op}_{dtype}.cu"):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    h.update((plan or "").encode())
    return h.hexdigest()


def profiled_traffic(workload_key, op, plan, dtype="f32"):
    """DRAM bytes per launch from the committed ncu summary of this
    workload, if it was taken on the current kernel code and plan."""
    path = os.path.join(ROOT, "profiles", f"{workload_key}.ncu.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    if fields.get("kernel_sources_sha256") != kernel_sources_sha(op, plan,
                                                                 dtype):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, read by a background
    thread while the GPU runs (start() ... stop())."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
             "sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.reader = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}",
                 f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            if line.strip():
                self.lines.append(line)

    def samples(self):
        return [p for p in (self._parse(l) for l in list(self.lines)) if p]

    def has_samples(self, n):
        """At least n samples so far (True at once if nvidia-smi could not
        be started: there is nothing to wait for)."""
        return self.proc is None or len(self.samples()) >= n

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
            self.proc.wait()
        if self.reader is not None:
            self.reader.join(timeout=5)

    def _parse(self, line):
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9:
            return None
        try:
            sm, mx = float(f[1]), float(f[2])
        except ValueError:
            return None
        active = [n for n, v in zip(self.NAMES, f[5:9])
                  if v.lower() == "active"]
        return sm, mx, active

    def summary(self):
        s = self.samples()
        if not s:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": statistics.median(x[0] for x in s),
                "sm_max_mhz": max(x[1] for x in s),
                "reasons": sorted({r for x in s for r in x[2]}),
                "samples": len(s)}


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k = line.split(":")[0].strip().lower()
                if k in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:   # Arm hosts: /proc/cpuinfo has no model name, lscpu does
        out = subprocess.run(["lscpu"], capture_output=True, text=True,
                             timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


def row_slices(d, bounds):
    """The input dict restricted to rows [lo, hi) for each bound pair."""
    return [{k: (v[lo:hi] if isinstance(v, np.ndarray) and
                 k in ("x", "residual", "labels") else v)
             for k, v in d.items()} for lo, hi in bounds]


class OracleRunner:
    """Runs the oracle over the rows of `d` on `threads` threads, each on a
    contiguous block of rows.  The oracle's C code runs through ctypes,
    which releases the interpreter lock, so the blocks run in parallel."""

    def __init__(self, op, d, rows, threads):
        import oracle
        from concurrent.futures import ThreadPoolExecutor
        oracle.build()
        self.oracle, self.op = oracle, op
        threads = max(1, min(threads, rows))
        step = -(-rows // threads)
        bounds = [(lo, min(rows, lo + step)) for lo in range(0, rows, step)]
        self.parts = row_slices(d, bounds)
        self.threads = len(self.parts)
        self.pool = ThreadPoolExecutor(self.threads) if self.threads > 1 \
            else None

    def __call__(self):
        if self.pool is None:
            self.oracle.run(self.op, self.parts[0])
        else:
            list(self.pool.map(lambda p: self.oracle.run(self.op, p),
                               self.parts))

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()


def time_oracle(runner, budget_s):
    reps, t0 = 0, time.perf_counter()
    while True:
        runner()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or el * (reps + 1) / reps > 3 * budget_s:
            return reps, el


def cpu_baseline(op, d, rows, cols, budget_s=10.0, dtype="f32"):
    """The CPU oracle as it stands on the same inputs (`d` in `dtype`
    storage, handed to the oracle as their exact FP32 values), on all host
    cores (row blocks on parallel threads) and on one thread, each repeated
    for about budget_s / 2 seconds."""
    from row_reduction_gb300 import inputs
    d = inputs.widen_all(d, dtype)
    b = algorithmic_bytes(op, rows, cols, op in H_OUT_OPS,
                          op == "cross_entropy", dtype)
    cores = os.cpu_count() or 1
    out = {}
    for name, threads in (("all", cores), ("one", 1)):
        runner = OracleRunner(op, d, rows, threads)
        reps, el = time_oracle(runner, budget_s / 2)
        runner.close()
        out[name] = (runner.threads, reps, el, b * reps / el / 1e9)
    n, reps, el, gbs = out["all"]
    n1, reps1, el1, gbs1 = out["one"]
    return {"value": gbs, "unit": "GB/s", "cores": n, "kind": "oracle",
            "sample": f"full {rows}x{cols} x{reps} in {el:.1f} s, "
                      f"{n} row blocks on {n} threads",
            "cpu": cpu_model(), "us_per_op": el / reps * 1e6,
            "single_thread": {"value": gbs1, "unit": "GB/s", "cores": 1,
                              "us_per_op": el1 / reps1 * 1e6}}


def headline_json(line):
    """The headline as one compact JSON line of at most HEADLINE_MAX_BYTES
    (a reader that keeps only the tail of stdout must still see all of it):
    the HEADLINE_OPTIONAL fields go first, one at a time, while it is too
    long; raises if the line without them is still too long."""
    line = json.loads(json.dumps(line))      # private copy
    text = json.dumps(line, separators=(",", ":"))
    for path in HEADLINE_OPTIONAL:
        if len(text.encode()) <= HEADLINE_MAX_BYTES:
            break
        node = line
        for key in path[:-1]:
            node = node.get(key) if isinstance(node, dict) else None
        if isinstance(node, dict):
            node.pop(path[-1], None)
        text = json.dumps(line, separators=(",", ":"))
    n = len(text.encode())
    if n > HEADLINE_MAX_BYTES:
        raise ValueError(f"headline is {n} bytes, over {HEADLINE_MAX_BYTES}")
    return text


def emit_headline(line):
    sys.stdout.flush()
    sys.stderr.flush()
    print(headline_json(line), flush=True)


# ---------------------------------------------------------------- arms
def run_reference(args, rank, world):
    if rank != 0:
        return 0
    import oracle
    from row_reduction_gb300 import inputs
    oracle.build()
    rows, cols = args.rows, args.cols
    d = inputs.widen_all(
        inputs.as_storage(inputs.make(args.op, rows, cols, inputs.TUNE_SEED,
                                      outliers=True), args.dtype),
        args.dtype)
    cores = os.cpu_count() or 1
    # Size the per-step row sample so the whole run stays near 60 s with
    # the rows split over every host core.
    t0 = time.perf_counter()
    oracle.run(args.op, row_slices(d, [(0, min(rows, 8))])[0])
    per_row = max((time.perf_counter() - t0) / min(rows, 8), 1e-7)
    total_steps = args.steps + args.warmup
    sample_rows = int(max(1, min(rows, 60.0 * cores / total_steps /
                                 per_row)))
    runner = OracleRunner(args.op, row_slices(d, [(0, sample_rows)])[0],
                          sample_rows, cores)
    for _ in range(args.warmup):
        runner()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        runner()
    el = time.perf_counter() - t0
    runner.close()
    b = algorithmic_bytes(args.op, sample_rows, cols, args.op in H_OUT_OPS,
                          args.op == "cross_entropy", args.dtype)
    value = b * args.steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": f"{args.op}_{args.dtype} {rows}x{cols}",
                   "op": args.op, "storage": args.dtype,
                   "rows": rows, "cols": cols,
                   "sample_rows_per_step": sample_rows},
        "cpu_baseline": {"value": value, "unit": "GB/s",
                         "cores": runner.threads, "kind": "oracle",
                         "sample": f"first {sample_rows} of {rows} rows "
                                   f"per step, split into {runner.threads} "
                                   f"row blocks on as many threads",
                         "cpu": cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    emit_headline(line)
    return 0


def quick_us(work, rounds=3, min_round_s=0.01):
    """Median µs per step over a few short graph-replay rounds."""
    return statistics.median(time_rounds(work, rounds=rounds,
                                         min_round_s=min_round_s))


def steps_us(work, steps, reps=5):
    """Median µs per step over `reps` windows of exactly `steps` steps timed
    as the headline is (time_graph_steps: one graph, events on its side
    branch)."""
    return statistics.median(time_graph_steps(work, steps, 5) / steps * 1e6
                             for _ in range(reps))


def best_probe(cls, work, steps):
    """The fastest launch shape of a probe kernel on the workload's pool:
    one wave of resident CTAs or one CTA per row (as the operators'
    one-row-per-CTA plans), with and without the L2 prefetch, found with
    short graph-replay rounds; then that shape timed like the headline
    (windows of `steps` steps).  Returns (µs, shape text)."""
    best = None
    for grid in (0, work.rows):
        for threads in (128, 256, 512, 1024):
            for unroll in (2, 4, 8):
                for flags in (0, 1):
                    us = quick_us(cls(work, threads, unroll, grid, flags))
                    if best is None or us < best[0]:
                        best = (us, threads, unroll, grid, flags)
    us, threads, unroll, grid, flags = best
    us = steps_us(cls(work, threads, unroll, grid, flags), steps)
    return us, (f"{threads} threads, {unroll} in flight, "
                f"grid {grid or 'one wave'}, "
                f"{'L2 prefetch' if flags else 'no prefetch'}")


def measure_floor(work, steps=20):
    """The floor of one step, timed like the steps themselves (dependent
    launches over the same rotating pool, windows of `steps` steps inside
    one graph): the library's plain copy kernel moving the step's matrix
    bytes in and out, or its read kernel reading them (best of a few launch
    shapes each), and its empty kernel, alone and on a full wave."""
    out = {}
    steps = max(1, min(steps, MAX_ONE_GRAPH_STEPS))
    if work.op in COPY_FLOOR_OPS:
        out["copy_us"], out["copy_shape"] = best_probe(CopyProbe, work,
                                                       steps)
        out["copy_bytes"] = CopyProbe(work).bytes
    if work.op in READ_FLOOR_OPS:
        out["read_us"], out["read_shape"] = best_probe(ReadProbe, work,
                                                       steps)
        out["read_bytes"] = ReadProbe(work).bytes
    out["empty_us"] = quick_us(EmptyProbe(32, 1), rounds=5, min_round_s=0.03)
    out["empty_wave_us"] = quick_us(EmptyProbe(512, 0), rounds=5,
                                    min_round_s=0.03)
    return out


def build_headline(f):
    """The headline line from the raw figures of a run (a dict: shape and
    steps, bytes per step, elapsed seconds, peak, plan, traffic, per-round
    µs, floor, e2e and link seconds, clock summary, pool, CPU baseline)."""
    per_step = f["elapsed"] / f["steps"]
    achieved = f["bytes"] / per_step / 1e9
    peak = f["peak"]
    moved = f["h2d"] + f["d2h"]
    e2e_us = f["e2e_el"] / f["e2e_steps"] * 1e6
    link_gbs = moved * f["e2e_steps"] / f["link_el"] / 1e9
    rounds = f["rounds"]
    line = {
        "metric": METRIC,
        "value": sig(f["world"] * achieved), "unit": "GB/s",
        "n_gpus": f["world"], "steps": f["steps"], "warmup": f["warmup"],
        "ms_per_step": sig(per_step * 1e3), "us_per_op": sig(per_step * 1e6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "storage": f["dtype"], "data": "synthetic",
        "config": {
            "workload": f"{f['op']} {f['dtype']} {f['rows']}x{f['cols']}, "
                        f"{INPUT_RECIPE[f['op']]}",
            "op": f["op"], "storage": f["dtype"], "rows": f["rows"],
            "cols": f["cols"], "plan": f["plan"],
            "l2": f"inputs larger than L2: {f['pool_sets']}-set rotating "
                  f"pool, {f['pool_bytes'] / 2**20:.0f} MiB >= 4x L2",
            "parallelism": "replicas" if f["world"] > 1 else "single GPU"},
        "roofline": {"bound": "hbm", "achieved": sig(achieved),
                     "peak": peak, "unit": "GB/s",
                     "frac": sig(sig(achieved) / peak),
                     "traffic": f["traffic"], "peak_source": f["peak_kind"]},
        "rounds_us": {"median": sig(statistics.median(rounds), 4),
                      "min": sig(min(rounds), 4), "max": sig(max(rounds), 4),
                      "n": len(rounds)},
        "e2e": {"value": sig(f["bytes"] / (e2e_us * 1e3)), "unit": "GB/s",
                "h2d_bytes_per_step": f["h2d"],
                "d2h_bytes_per_step": f["d2h"],
                "us_per_step": sig(e2e_us), "link_gbs": sig(link_gbs),
                "frac": sig(moved / (sig(e2e_us) * 1e3) / sig(link_gbs))},
        "gpu_launches": f["steps"] * f["launches_per_step"],
        "clocks": f["clocks"],
    }
    fl = f["floor"]
    line["floor"] = {}
    for kind in ("copy", "read"):
        if f"{kind}_us" in fl:
            us = fl[f"{kind}_us"]
            line["floor"].update({
                f"{kind}_us": sig(us, 4),
                f"{kind}_frac": sig(fl[f"{kind}_bytes"] / us / 1e3 / peak, 4),
                f"frac_of_{kind}": sig(us / (per_step * 1e6), 4)})
    line["floor"]["empty_us"] = sig(fl["empty_us"], 4)
    cb = f.get("cpu")
    if cb:
        line["cpu_baseline"] = {k: (sig(cb[k], 4) if k == "value" else cb[k])
                                for k in ("value", "unit", "cores", "kind",
                                          "sample", "cpu")}
    return line


def run_profile(args):
    """--profile: only the timed steps of the workload (or of a probe's
    chain on the workload's pool), for a profiler to capture; prints one
    short line, not the headline."""
    import torch
    import row_reduction_gb300 as mt
    from row_reduction_gb300 import build as mt_build, inputs
    mt_build.build()
    mt.lib()
    props = torch.cuda.get_device_properties(0)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20)) or (126 << 20)
    work = Workload(args.op, args.rows, args.cols, inputs.TUNE_SEED,
                    outliers=True, l2_bytes=l2, dtype=args.dtype,
                    ce_mean=not args.loss_only)
    if args.probe == "copy":
        work = CopyProbe(work, 512, 8, 0, 1)
    elif args.probe == "read":
        work = ReadProbe(work, 512, 8, 0, 1)
    el = time_graph_steps(work, args.steps, args.warmup)
    print(f"profile run: {args.op} {args.dtype} {args.rows}x{args.cols}"
          f"{' ' + args.probe + ' probe' if args.probe else ''}: "
          f"{el / args.steps * 1e6:.3f} us per step over {args.steps} steps")
    return 0


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    import row_reduction_gb300 as mt
    from row_reduction_gb300 import build as mt_build, inputs

    mt_build.build()
    mt.lib()
    torch.cuda.set_device(local_rank)
    props = torch.cuda.get_device_properties(local_rank)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20)) or (126 << 20)
    barrier = (lambda: dist.barrier()) if world > 1 else None

    work = Workload(args.op, args.rows, args.cols, inputs.TUNE_SEED,
                    outliers=True, l2_bytes=l2, dtype=args.dtype)
    sampler = ClockSampler(local_rank)
    elapsed = time_graph_steps(work, args.steps, args.warmup,
                               barrier=barrier, sampler=sampler)
    if world > 1:
        elapsed = max_over_ranks(elapsed, "cuda")
    if rank != 0:
        return 0

    peak, peak_kind = measured_peak()
    key = f"{args.op}_{args.dtype}_{args.rows}x{args.cols}"
    plan = plan_text(args.op, args.rows, args.cols, args.dtype)
    rounds = time_rounds(work, rounds=5, min_round_s=0.03)
    floor = measure_floor(work, args.steps)
    e2e_steps = max(3, min(args.steps, 200))
    e2e_el, bi, bo = time_e2e(work, e2e_steps, 3, depth=3)
    link_el = time_link(bi, bo, e2e_steps, 3, depth=3)
    fig = {"op": args.op, "dtype": args.dtype, "rows": args.rows,
           "cols": args.cols, "steps": args.steps, "warmup": args.warmup,
           "world": world, "bytes": work.bytes, "elapsed": elapsed,
           "peak": peak, "peak_kind": peak_kind, "plan": plan,
           "traffic": profiled_traffic(key, args.op, plan, args.dtype),
           "rounds": rounds, "floor": floor, "e2e_el": e2e_el,
           "e2e_steps": e2e_steps, "h2d": bi, "d2h": bo, "link_el": link_el,
           "clocks": sampler.summary(), "pool_sets": len(work.sets),
           "pool_bytes": work.pool_bytes,
           "launches_per_step": work.launches_per_step, "cpu": None}
    line = build_headline(fig)
    details = {"headline": line, "floor": floor,
               "rounds_us": rounds, "e2e_serial_us_per_step": None}
    serial_el, _, _ = time_e2e(work, e2e_steps, 3, depth=1)
    details["e2e_serial_us_per_step"] = serial_el / e2e_steps * 1e6
    plain_steps = min(args.steps, 20000)
    plain = time_plain_steps(work, plain_steps, min(args.warmup, 200))
    details["plain_launch"] = {"us_per_op": plain / plain_steps * 1e6,
                               "note": "one Python ctypes call per step"}
    if world == 1:
        details["hot"] = hot_number(args, l2)
        details["torch_context"] = torch_context(work)
    if world == 1 and not args.no_cpu_baseline:
        cb = cpu_baseline(args.op, work.host, args.rows, args.cols,
                          args.cpu_seconds, args.dtype)
        details["cpu_baseline"] = cb
        fig["cpu"] = cb
        line = build_headline(fig)
        details["headline"] = line
    if world == 1 and not args.no_sweep:
        details["sweep"] = run_sweep(l2, peak)
    print_details(details, peak)
    if args.details:
        with open(args.details, "w") as f:
            json.dump(details, f, indent=1)
    emit_headline(line)
    return 0


def print_details(d, peak):
    """A human-readable summary of the details on stderr."""
    err = sys.stderr
    fl = d["floor"]
    print("== floor (same pool, graph replays of dependent launches)",
          file=err)
    for k, v in fl.items():
        print(f"   {k}: {v}", file=err)
    print(f"== e2e serial (one stream): "
          f"{d['e2e_serial_us_per_step']:.2f} us/step", file=err)
    print(f"== plain Python launches: {d['plain_launch']['us_per_op']:.3f} "
          "us/op", file=err)
    for k in ("hot", "torch_context"):
        if d.get(k):
            print(f"== {k}: {json.dumps(d[k])}", file=err)
    if d.get("cpu_baseline"):
        print(f"== cpu_baseline: {json.dumps(d['cpu_baseline'])}", file=err)
    if d.get("sweep"):
        print("== sweep: op dtype rows x cols | us/op | GB/s | % of "
              f"{peak:.0f} | plan", file=err)
        for r in d["sweep"]:
            tag = "" if r.get("mean", True) else " (loss only)"
            print(f"   {r['op']}{tag} {r['dtype']} {r['rows']}x{r['cols']}"
                  f" | {r['us_per_op']:.3f} | {r['gbs']:.0f} | "
                  f"{100 * r['frac_of_peak']:.1f} | {r['plan']}", file=err)
    err.flush()


def hot_number(args, l2):
    """The same step on one buffer set every time (inputs and outputs stay
    in L2 when they fit): a labelled upper bound, not the headline."""
    import torch
    from row_reduction_gb300 import inputs
    hot = Workload(args.op, args.rows, args.cols, inputs.TUNE_SEED,
                   outliers=True, l2_bytes=l2, max_pool_bytes=0,
                   dtype=args.dtype)
    steps = 2000
    el = time_graph_steps(hot, steps, 100)
    out = {"us_per_op": el / steps * 1e6,
           "value": hot.bytes * steps / el / 1e9, "unit": "GB/s",
           "note": "same buffers every step (L2-resident when they fit)"}
    del hot
    torch.cuda.empty_cache()
    return out


def torch_context(work):
    """PyTorch's own kernel for the operator on the same buffer pool, timed
    the same way (CUDA graphs, events): context from another library, not
    a target and not part of this library."""
    import torch
    import torch.nn.functional as F
    op = work.op
    if op == "cross_entropy":
        long_labels = {id(s): s["labels"].long() for s in work.sets}
    fns = {
        "rmsnorm": lambda s: F.rms_norm(s["x"], (work.cols,), s["weight"],
                                        work.eps),
        "layernorm": lambda s: F.layer_norm(s["x"], (work.cols,), s["gamma"],
                                            s["beta"], work.eps),
        "softmax": lambda s: torch.softmax(s["x"], dim=1),
        "log_softmax": lambda s: torch.log_softmax(s["x"], dim=1),
        "row_sum": lambda s: s["x"].sum(dim=1),
        "cross_entropy": lambda s: F.cross_entropy(s["x"],
                                                   long_labels[id(s)]),
    }
    if op not in fns or not hasattr(F, "rms_norm"):
        return None
    f = fns[op]
    n = len(work.sets)
    stream = torch.cuda.Stream()
    try:
        with torch.cuda.stream(stream):
            for i in range(3):
                f(work.sets[i % n])
        stream.synchronize()
        G = n * max(1, math.ceil(64 / n))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(G):
                f(work.sets[i % n])
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            g.replay()
            start.record(stream)
            for _ in range(20):
                g.replay()
            end.record(stream)
        end.synchronize()
    except Exception as e:  # context only: report why it is missing
        return {"unavailable": str(e)[:200]}
    us = start.elapsed_time(end) * 1e3 / (20 * G)
    del g
    return {"system": f"torch {torch.__version__}", "us_per_op": us,
            "value": work.bytes / us / 1e3, "unit": "GB/s",
            "note": "PyTorch's own kernel on the same pool; context only"}


def sweep_cases():
    """Every published shape: RMSNorm shapes and bandwidth sweep, then the
    operator family (cross-entropy with its mean and with the per-row losses
    alone); then the same RMSNorm sweep and the family at 1024x4096 with
    BF16 and FP16 storage.  Entries: (op, rows, cols, outliers, dtype,
    with the CE mean)."""
    from row_reduction_gb300 import inputs
    cases = [("rmsnorm", r, c, False, "f32", True)
             for r, c in inputs.RMSNORM_SHAPES]
    cases += [("rmsnorm", r, c, True, "f32", True)
              for r, c in inputs.RMSNORM_SWEEP]
    cases += [(op, r, c, False, "f32", True) for op in inputs.ALL_OPS
              if op != "rmsnorm" for r, c in inputs.FAMILY_SHAPES]
    cases.append(("cross_entropy", 1024, 4096, False, "f32", False))
    for dt in ("bf16", "f16"):
        cases += [("rmsnorm", r, c, True, dt, True)
                  for r, c in inputs.RMSNORM_SWEEP]
        cases += [(op, 1024, 4096, False, dt, True) for op in inputs.ALL_OPS
                  if op != "rmsnorm"]
        cases.append(("cross_entropy", 1024, 4096, False, dt, False))
    return cases


def run_sweep(l2, peak):
    import torch
    from row_reduction_gb300 import inputs
    out = []
    for op, r, c, outl, dt, mean in sweep_cases():
        work = Workload(op, r, c, inputs.TUNE_SEED, outliers=outl,
                        l2_bytes=l2, max_pool_bytes=8 << 30, dtype=dt,
                        ce_mean=mean)
        # about 0.25 s of timed work, at least 64 steps
        probe = time_graph_steps(work, 64, 16)
        steps = int(max(64, min(200000, 0.25 / max(probe / 64, 1e-7))))
        el = time_graph_steps(work, steps, max(16, steps // 20))
        us = el / steps * 1e6
        gbs = work.bytes / (el / steps) / 1e9
        out.append({"op": op, "dtype": dt, "rows": r, "cols": c,
                    "outliers": outl, "mean": mean, "us_per_op": us,
                    "gbs": gbs, "frac_of_peak": gbs / peak,
                    "plan": plan_text(op, r, c, dt),
                    "pool_sets": len(work.sets),
                    "l2_resident": work.l2_resident, "steps": steps})
        del work
        torch.cuda.empty_cache()
    return out


def verify_line(line):
    """Audits one headline JSON line of this benchmark: the reported figures
    recomputed from the raw ones (steps, time, bytes), and the recorded plan
    against the planner's current choice.  Returns a list of problems
    (empty when the line is consistent).  Figures in the line carry six
    significant digits, so they are compared to within 1e-5."""
    bad = []

    def close(a, b, what, rel=1e-5):
        if a is None or b is None or abs(a - b) > rel * max(abs(b), 1e-30):
            bad.append(f"{what}: {a} vs {b}")

    if line.get("impl") == "reference":
        close(line["cpu_baseline"]["value"], line["value"], "cpu_baseline")
        return bad
    cfg = line["config"]
    dtype = cfg.get("storage", "f32")
    op, rows, cols = cfg["op"], cfg["rows"], cfg["cols"]
    b = algorithmic_bytes(op, rows, cols, op in H_OUT_OPS,
                          op == "cross_entropy", dtype)
    per_step = line["ms_per_step"] / 1e3
    close(line["value"], line["n_gpus"] * b / per_step / 1e9, "value")
    close(line["us_per_op"], line["ms_per_step"] * 1e3, "us_per_op")
    roof = line["roofline"]
    close(roof["achieved"], b / per_step / 1e9, "roofline.achieved")
    close(roof["frac"], roof["achieved"] / roof["peak"], "roofline.frac")
    r = line.get("rounds_us")
    if r and not r["min"] <= r["median"] <= r["max"]:
        bad.append(f"rounds_us: median {r['median']} outside "
                   f"[{r['min']}, {r['max']}]")
    e = line.get("e2e")
    if e and "link_gbs" in e:
        moved = e["h2d_bytes_per_step"] + e["d2h_bytes_per_step"]
        close(e["frac"], moved / (e["us_per_step"] * 1e3) / e["link_gbs"],
              "e2e.frac", rel=1e-4)
        close(e["value"], b / (e["us_per_step"] * 1e3), "e2e.value",
              rel=1e-4)
    if cfg["plan"] != plan_text(op, rows, cols, dtype):
        bad.append(f"plan: recorded {cfg['plan']!r}, planner now "
                   f"{plan_text(op, rows, cols, dtype)!r}")
    return bad


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=2000)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", default="rmsnorm")
    ap.add_argument("--rows", type=int, default=1024)
    ap.add_argument("--cols", type=int, default=4096)
    ap.add_argument("--dtype", choices=["f32", "f16", "bf16"], default="f32",
                    help="storage type of matrices and parameter vectors "
                         "(arithmetic is FP32 for all)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", action="store_true",
                    help="only run the timed steps (for a profiler); print "
                         "one short line instead of the headline")
    ap.add_argument("--probe", choices=["copy", "read"], default=None,
                    help="with --profile: run the library's copy or read "
                         "probe over the workload's buffers instead")
    ap.add_argument("--loss-only", action="store_true",
                    help="cross-entropy without the batch mean "
                         "(mean_loss = NULL); with --profile")
    ap.add_argument("--details", metavar="FILE", default=None,
                    help="also write every figure (sweep, floor, hot, "
                         "context) to FILE as JSON")
    ap.add_argument("--verify", metavar="FILE", default=None,
                    help="audit the JSON line(s) in FILE instead of timing")
    args = ap.parse_args()
    if args.verify:
        problems = []
        for ln in open(args.verify):
            if ln.startswith("{"):
                problems += verify_line(json.loads(ln))
        for p in problems:
            print(p)
        print("consistent" if not problems else f"{len(problems)} problems")
        return 1 if problems else 0
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.profile:
        return run_profile(args)
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        return run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
