"""Measured launch-plan search; writes the planner's table.

For each (operator, storage type, rows, cols) the tuner enumerates the legal
plans (V in {1, 2, 4} for FP32 and {2, 4, 8} for FP16/BF16; W a power of
two; the smallest register chunk count that holds the row; rows per CTA B so
that a CTA has 32..1024 threads; the loop path and the staged path for wide
rows; clusters of 2, 4, 8 or 16 CTAs per row for few or very wide rows; the
launch flags),
then, in a second stage, the four fastest again on persistent grids of one
to three CTAs per SM.  For each plan it:

1. runs it once on the tuning-seed inputs and validates the complete output
   against the reference plan's output (|a-b| <= 1e-5*(1+|b|)); a plan that
   fails or errors is rejected and logged, never timed;
2. times it: median over rounds of graph-replayed back-to-back calls over a
   rotating buffer pool larger than 4x L2 (row_reduction_gb300.timing).

The three fastest are re-measured with more rounds; the winner is then
validated on held-out-seed inputs.  This follows the pages' protocol: a
finite GPU-objective search in which every timed candidate's complete output
is validated and every winner is re-measured ("Consecutive-worker reduction
layout checkpoint", §Evidence and what remains and §Measurement contract),
and tuning on one input seed with validation on another ("Thread Ownership
and Software Staging", §Bounded tiling: prior register baseline).

Usage (on a GPU):
    python -m row_reduction_gb300.tune --shapes published \
        --json out.json --table row_reduction_gb300/csrc/plan_table.inc
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import time

from . import _binding as B
from . import inputs
from .timing import Workload, time_rounds

CHUNKS = (1, 2, 4, 8, 16)
STAGE_OPS = ("rmsnorm", "layernorm", "softmax", "log_softmax",
             "cross_entropy", "row_sum")
VALUES = {"f32": (4, 2, 1), "f16": (8, 4, 2), "bf16": (8, 4, 2)}
FLAG_SETS = (B.MT_PLAN_PDL, B.MT_PLAN_PDL | B.MT_PLAN_PREFETCH_NEXT, 0)


def pow2ceil(v):
    p = 1
    while p < v:
        p <<= 1
    return p


def candidates(op, rows, cols, dtype="f32"):
    """Legal plans worth timing for one shape."""
    out = []
    op_id = B.OP_IDS[op]
    for V in VALUES[dtype]:
        W = V if V > 1 else 1
        while W <= 1024:
            if W * V <= 2 * pow2ceil(cols) or W <= 32:
                K = next((k for k in CHUNKS if W * V * k >= cols), None)
                for threads in (32, 64, 128, 256, 512, 1024):
                    if threads < W or threads % W:
                        continue
                    Bk = threads // W
                    if Bk > 1 and Bk > pow2ceil(rows):
                        continue
                    for fl in FLAG_SETS:
                        if K is not None:
                            out.append(B.make_plan(W, V, K, Bk, flags=fl))
                            # Exact tiling: the unguarded whole-tile kernel
                            # too (with the dependent-launch prologue).
                            if (fl and W * V * K == cols and rows % Bk == 0
                                    and (V > 1 or dtype == "f32")):
                                out.append(B.make_plan(
                                    W, V, K, Bk,
                                    flags=fl | B.MT_PLAN_WHOLE_TILES))
                        if cols >= 8192:
                            out.append(B.make_plan(W, V, 0, Bk,
                                                   B.MT_PATH_LOOP, flags=fl))
            W *= 2
    # Split rows (clusters of CTAs per row): when rows are too few to give
    # every SM work, and when a row is wider than one CTA can hold in
    # registers (16384 values), so that the cluster holds it instead of the
    # loop path reading it twice.  16-byte packs, one row per CTA.
    vmax = VALUES[dtype][0]
    if (rows < 304 and cols >= 1024) or cols > 16384:
        for C in ((2, 4, 8, 16) if rows <= 19 else (2, 4, 8)):
            for W in (128, 256, 512, 1024):
                K = next((k for k in CHUNKS if C * W * vmax * k >= cols),
                         None)
                for fl in FLAG_SETS:
                    if K is not None:
                        out.append(B.make_plan(W, vmax, K, 1, flags=fl,
                                               cluster=C))
                    if cols >= 8192:
                        out.append(B.make_plan(W, vmax, 0, 1, B.MT_PATH_LOOP,
                                               flags=fl, cluster=C))
    # Staged rows (shared memory filled by bulk copies): wide rows, one row
    # per CTA or per cluster.
    if cols >= 8192 and op in STAGE_OPS:
        for C in ((1, 2, 4, 8, 16) if rows <= 19 else (1, 2, 4, 8)):
            for W in (256, 512, 1024):
                for pieces in (2, 4):
                    for fl in (B.MT_PLAN_PDL,
                               B.MT_PLAN_PDL | B.MT_PLAN_PREFETCH_NEXT):
                        out.append(B.make_plan(W, vmax, pieces, 1,
                                               B.MT_PATH_STAGE, flags=fl,
                                               cluster=C if C > 1 else 0))
    seen, legal = set(), []
    for p in out:
        key = tuple(p.as_dict().values())
        if key in seen:
            continue
        seen.add(key)
        if B.mt_plan_check_dtype(op_id, dtype, cols, p) == B.MT_OK:
            legal.append(p)
    return legal


def grid_variants(rows, plans, sms):
    """Second-stage candidates: the given plans again with persistent grids
    of one to three CTAs per SM (fewer CTAs than row groups, so each loops
    over several), with and without the next-group prefetch."""
    flag_sets = (B.MT_PLAN_PDL, B.MT_PLAN_PDL | B.MT_PLAN_PREFETCH_NEXT)
    out = []
    for p in plans:
        d = p.as_dict()
        C = max(1, d.get("cluster", 0))
        ngroups = -(-rows // d["rows_per_block"])
        for mult in (1, 2, 3):
            G = sms * mult
            if G % C or G // C >= ngroups:
                continue
            keep = d.get("flags", 0) & B.MT_PLAN_WHOLE_TILES
            for fl in flag_sets:
                out.append(B.MtPlan(**dict(d, grid=G, flags=fl | keep)))
    return out


def _outputs(work, plan):
    import torch
    stream = torch.cuda.current_stream()
    work.call_fn(0, stream.cuda_stream, plan)()
    torch.cuda.synchronize()
    return {k: v.clone() for k, v in work.outputs(0).items()}


def _agrees(a, b, dtype="f32"):
    """Two plans' outputs agree: within the FP32 tolerance, plus one unit of
    the storage type's last place for 16-bit outputs (each plan rounds its
    own FP32 result once)."""
    import torch
    rel = {"f32": 0.0, "f16": 2.0 ** -10, "bf16": 2.0 ** -7}[dtype]
    for k in b:
        x, y = a[k].double(), b[k].double()
        nan = torch.isnan(x) & torch.isnan(y)
        r = rel if a[k].dtype != torch.float32 else 0.0
        ok = ((x - y).abs() <= 1e-5 * (1 + y.abs()) + r * y.abs()) | nan
        if not bool(ok.all()):
            return False
    return True


def tune_shape(op, rows, cols, l2, rounds=5, log=print, dtype="f32"):
    """Tunes one shape; returns a record with the winner and timings."""
    import torch
    outliers = op == "rmsnorm" and (rows, cols) in inputs.RMSNORM_SWEEP
    work = Workload(op, rows, cols, inputs.TUNE_SEED, outliers=outliers,
                    l2_bytes=l2, max_pool_bytes=8 << 30, dtype=dtype)
    default = B.mt_plan_query_dtype(op, dtype, rows, cols)
    ref = _outputs(work, default)
    cands = candidates(op, rows, cols, dtype)
    timed = []
    rejected = 0
    seen = set()

    def run_stage(plans):
        nonlocal rejected
        for p in plans:
            key = tuple(p.as_dict().values())
            if key in seen:
                continue
            seen.add(key)
            try:
                got = _outputs(work, p)
            except B.MTError as e:
                log(f"  reject {B.mt_describe_plan(p)}: {e}")
                rejected += 1
                continue
            if not _agrees(got, ref, dtype):
                log(f"  reject {B.mt_describe_plan(p)}: output differs")
                rejected += 1
                continue
            us = statistics.median(time_rounds(work, p, rounds=rounds,
                                               min_round_s=0.004))
            timed.append((us, p))
        timed.sort(key=lambda t: t[0])

    run_stage(cands)
    # Second stage: persistent grids and prefetch depth for the best plans.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    stage2 = grid_variants(rows, [p for _, p in timed[:4]], sms)
    stage2 = [p for p in stage2 if B.mt_plan_check_dtype(
        B.OP_IDS[op], dtype, cols, p) == B.MT_OK]
    run_stage(stage2)
    cands = cands + stage2
    # Re-measure the three fastest (and the default) with more rounds.
    finals = []
    for us, p in timed[:3]:
        r = time_rounds(work, p, rounds=2 * rounds + 1, min_round_s=0.01)
        finals.append((statistics.median(r), p, r))
    finals.sort(key=lambda t: t[0])
    best_us, best, best_rounds = finals[0]
    d_rounds = time_rounds(work, default, rounds=2 * rounds + 1,
                           min_round_s=0.01)
    del work
    torch.cuda.empty_cache()
    # Held-out validation of the winner.
    hold = Workload(op, rows, cols, inputs.HOLDOUT_SEED, outliers=outliers,
                    l2_bytes=0, max_pool_bytes=0, dtype=dtype)
    ok = _agrees(_outputs(hold, best), _outputs(hold, default), dtype)
    del hold
    torch.cuda.empty_cache()
    if not ok:
        raise RuntimeError(f"{op} {rows}x{cols}: winner fails held-out "
                           "validation")
    rec = {"op": op, "dtype": dtype, "rows": rows, "cols": cols,
           "winner": best.as_dict(), "winner_text": B.mt_describe_plan(best),
           "winner_us": best_us, "winner_rounds_us": best_rounds,
           "default": default.as_dict(),
           "default_us": statistics.median(d_rounds),
           "candidates": len(cands), "rejected": rejected,
           "top": [{"plan": p.as_dict(), "us": us} for us, p in timed[:8]]}
    log(f"{op} {dtype} {rows}x{cols}: {len(cands)} plans, winner "
        f"{rec['winner_text']} {best_us:.3f} us (default "
        f"{rec['default_us']:.3f} us)")
    return rec


def evaluate(records, l2, rounds=7, log=print):
    """Regret of the planner's own choice on tuned shapes: times the plan
    mt_plan_query_dtype returns and compares it with each record's measured
    winner.  Used on held-out shapes (records not in the table) to check
    the fallback of the planner."""
    import torch
    out = []
    for r in records:
        dt = r.get("dtype", "f32")
        outliers = r["op"] == "rmsnorm" and \
            (r["rows"], r["cols"]) in inputs.RMSNORM_SWEEP
        work = Workload(r["op"], r["rows"], r["cols"], inputs.TUNE_SEED,
                        outliers=outliers, l2_bytes=l2,
                        max_pool_bytes=8 << 30, dtype=dt)
        p = B.mt_plan_query_dtype(r["op"], dt, r["rows"], r["cols"])
        us = statistics.median(time_rounds(work, p, rounds=rounds,
                                           min_round_s=0.01))
        best = statistics.median(time_rounds(work, B.MtPlan(**r["winner"]),
                                             rounds=rounds, min_round_s=0.01))
        rec = {"op": r["op"], "dtype": dt, "rows": r["rows"],
               "cols": r["cols"], "plan": B.mt_describe_plan(p),
               "plan_us": us, "best_us": best, "regret": us / best - 1.0}
        log(f"{r['op']} {dt} {r['rows']}x{r['cols']}: planner {us:.3f} us "
            f"vs best {best:.3f} us (regret {100 * rec['regret']:.1f}%) "
            f"[{rec['plan']}]")
        out.append(rec)
        del work
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------ the table
ROWS_REACH = 16   # a measured plan serves row counts within this factor


def _rows_ranges(rows_list):
    """Splits the row counts between the tuned ones at geometric midpoints,
    each range at most a factor ROWS_REACH from its tuned row count (the
    planner re-fits or falls back beyond that)."""
    rows_list = sorted(rows_list)
    out = []
    for i, r in enumerate(rows_list):
        lo = 0 if i == 0 else int(math.floor(math.sqrt(
            rows_list[i - 1] * r))) + 1
        hi = (2 ** 62 if i == len(rows_list) - 1 else
              int(math.floor(math.sqrt(r * rows_list[i + 1]))))
        lo = max(lo, r // ROWS_REACH)
        hi = min(hi, r * ROWS_REACH)
        out.append((r, lo, hi))
    return out


def write_table(records, path):
    lines = [
        "// plan_table.inc -- measured plan winners, written by the "
        "package's tuner",
        "// (row_reduction_gb300/tune.py) from timings on the GPU; do not "
        "edit by",
        "// hand.  Entry: {op, dtype, cols_min, cols_max, rows_min, rows_max,",
        "// rows tuned, {W, V, chunks, rows_per_block, path, grid, flags,",
        "// cluster}}.  The last entry (op -1) only terminates the list.",
        "static const PlanEntry kPlanTable[] = {",
    ]
    by = {}
    for r in records:
        by.setdefault((r["op"], r.get("dtype", "f32"), r["cols"]),
                      []).append(r)
    for (op, dt, cols), recs in sorted(
            by.items(), key=lambda kv: (B.OP_IDS[kv[0][0]],
                                        B.DTYPE_IDS[kv[0][1]], kv[0][2])):
        ranges = dict((r, (lo, hi)) for r, lo, hi in
                      _rows_ranges([x["rows"] for x in recs]))
        for r in sorted(recs, key=lambda x: x["rows"]):
            lo, hi = ranges[r["rows"]]
            w = r["winner"]
            lines.append(
                f"    {{{B.OP_IDS[op]}, {B.DTYPE_IDS[dt]}, {cols}, {cols}, "
                f"{lo}, {hi}, {r['rows']}, "
                f"{{{w['threads_per_row']}, {w['values_per_thread']}, "
                f"{w['chunks']}, {w['rows_per_block']}, {w['path']}, "
                f"{w['grid']}, {w.get('flags', 0)}, {w.get('cluster', 0)}"
                f"}}}},  "
                f"// {op} {dt} {r['rows']}x{cols}: "
                f"{r['winner_us']:.3f} us")
    lines.append("    {-1, 0, 0, 0, 0, 0, 0, {0, 0, 0, 0, 0, 0, 0, 0}},")
    lines.append("};")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


def published_shapes(ops):
    """RMSNorm: the published shapes and bandwidth sweep; every other
    operator (the fused variants included): the family shapes."""
    shapes = []
    for op in ops:
        if op == "rmsnorm":
            shapes += [(op, r, c) for r, c in
                       inputs.RMSNORM_SHAPES + inputs.RMSNORM_SWEEP]
        else:
            shapes += [(op, r, c) for r, c in inputs.FAMILY_SHAPES]
    return shapes


# Held-out shapes for the planner's regret: every operator and storage type,
# row lengths outside the measured table (so the planner re-fits or falls
# back), from short rows to rows wider than one CTA's registers.  They are
# tuned to find each shape's own optimum, never written into the table.
HELDOUT_CASES = (
    "rmsnorm:f32:512x2048", "rmsnorm:f32:2048x5120", "rmsnorm:f32:300x3000",
    "rmsnorm:f32:1x30000", "rmsnorm:f32:32x32768", "rmsnorm:f32:4096x12288",
    "rmsnorm:bf16:3000x768", "rmsnorm:f16:777x5000",
    "layernorm:f32:2048x1024", "layernorm:f32:100x8192",
    "layernorm:bf16:4096x2560", "layernorm:f16:512x768",
    "residual_layernorm:f32:1500x2048", "residual_layernorm:bf16:8192x1024",
    "residual_layernorm:f16:64x12288",
    "softmax:f32:4096x1000", "softmax:bf16:4096x1000",
    "softmax:bf16:128x50257", "softmax:f16:2000x2000",
    "log_softmax:f32:333x7777", "log_softmax:bf16:1024x32768",
    "log_softmax:f16:64x100000",
    "row_sum:f32:5000x1000", "row_sum:f32:16x50000",
    "row_sum:bf16:2048x4000", "row_sum:f16:700x300",
    "cross_entropy:f32:4096x1000", "cross_entropy:f32:2048x50257",
    "cross_entropy:bf16:4096x1000", "cross_entropy:bf16:128x50257",
    "cross_entropy:f16:1000x151936",
    "residual_rmsnorm:f32:2048x3072", "residual_rmsnorm:bf16:4096x5120",
    "residual_rmsnorm:f16:100x6000",
)


# A second held-out set, for the shape-derived plans' out-of-sample check:
# shapes that neither the table nor the constants of those rules saw.
VALIDATION_CASES = (
    "rmsnorm:f32:1536x2304", "rmsnorm:bf16:6000x1536",
    "layernorm:f32:768x3072", "layernorm:bf16:12000x512",
    "layernorm:f16:48x40000", "residual_layernorm:bf16:2500x4096",
    "residual_rmsnorm:f32:5000x768", "softmax:f32:256x20000",
    "softmax:bf16:9000x1000", "log_softmax:f16:3000x2500",
    "row_sum:bf16:200x60000", "row_sum:f32:10000x640",
    "cross_entropy:f32:512x32768", "cross_entropy:bf16:60x128000",
)


def parse_case(text):
    """'op:dtype:RxC' -> (dtype, op, rows, cols)."""
    op, dt, shape = text.split(":")
    if op not in B.OP_IDS or dt not in B.DTYPE_IDS:
        raise ValueError(f"bad case {text!r}")
    r, c = shape.split("x")
    return dt, op, int(r), int(c)


def main(argv=None):
    ap = argparse.ArgumentParser(description="measured plan search")
    ap.add_argument("--ops", default=",".join(inputs.ALL_OPS))
    ap.add_argument("--shapes", default="published",
                    help="'published' or a list like 1024x4096,64x4096")
    ap.add_argument("--json", required=True)
    ap.add_argument("--table", default=None)
    ap.add_argument("--rounds", type=int, default=5)
    ap.add_argument("--dtypes", default="f32",
                    help="storage types, e.g. f32,bf16,f16")
    ap.add_argument("--evaluate", default=None,
                    help="tuning records (JSON) to measure the planner's "
                         "regret on, instead of tuning")
    ap.add_argument("--cases", default=None,
                    help="explicit (operator, storage type, shape) cases "
                         "instead of --ops/--dtypes/--shapes, e.g. "
                         "rmsnorm:f32:512x2048,softmax:bf16:128x50257, "
                         "or 'heldout' / 'validation' for HELDOUT_CASES / "
                         "VALIDATION_CASES")
    args = ap.parse_args(argv)
    import torch
    from . import build
    build.build()
    if args.evaluate:
        props = torch.cuda.get_device_properties(0)
        l2 = int(getattr(props, "L2_cache_size", 126 << 20)) or (126 << 20)
        recs = json.load(open(args.evaluate))["records"]
        res = evaluate(recs, l2, log=lambda s: print(s, flush=True))
        with open(args.json, "w") as f:
            json.dump({"device": torch.cuda.get_device_name(0),
                       "evaluation": res}, f, indent=1)
        return 0
    ops = [o for o in args.ops.split(",") if o]
    if args.shapes == "published":
        shapes = published_shapes(ops)
    else:
        shapes = [(op, int(s.split("x")[0]), int(s.split("x")[1]))
                  for op in ops for s in args.shapes.split(",")]
    work = [(dt, op, r, c) for dt in args.dtypes.split(",") if dt
            for op, r, c in shapes]
    if args.cases:
        cases = (HELDOUT_CASES if args.cases == "heldout"
                 else VALIDATION_CASES if args.cases == "validation"
                 else args.cases.split(","))
        work = [parse_case(c) for c in cases if c]
    props = torch.cuda.get_device_properties(0)
    l2 = int(getattr(props, "L2_cache_size", 126 << 20)) or (126 << 20)
    records = []
    if os.path.exists(args.json):          # resume an interrupted run
        records = json.load(open(args.json))["records"]
    done = {(r["op"], r.get("dtype", "f32"), r["rows"], r["cols"])
            for r in records}
    t0 = time.time()
    for dt, op, rows, cols in work:
        if (op, dt, rows, cols) in done:
            continue
        records.append(tune_shape(op, rows, cols, l2, args.rounds,
                                  log=lambda s: print(s, flush=True),
                                  dtype=dt))
        with open(args.json, "w") as f:
            json.dump({"device": torch.cuda.get_device_name(0),
                       "records": records}, f, indent=1)
    print(f"tuned {len(records)} shapes in {time.time() - t0:.0f} s")
    if args.table:
        write_table(records, args.table)
    return 0


if __name__ == "__main__":
    sys.exit(main())
