"""Device timing of library calls, shared by the tuner and the benchmark.

A :class:`Workload` holds a pool of input/output buffer sets for one
(operator, rows, cols); consecutive steps cycle through the pool, which is
sized to at least 4x the L2 cache (capped at 256 sets), so no step finds its
input in L2 unless the whole pool fits there (tiny, launch-bound shapes;
``l2_resident`` says so).  Steps are captured into CUDA graphs of whole pool
cycles and replayed back to back on one stream; CUDA events on that stream
bracket the timed replays.  The timing method follows the pages' contract of
batched GPU intervals divided by the batch size ("Consecutive-worker
reduction layout checkpoint", §Measurement contract).
"""
from __future__ import annotations

import ctypes
import math

from . import _binding as B
from . import inputs

MAX_SETS = 256


ELEM_BYTES = {"f32": 4, "f16": 2, "bf16": 2}


def algorithmic_bytes(op, rows, cols, h_out=False, mean=False, dtype="f32"):
    """Bytes the operator must move once: every input element read once,
    every output written once, parameter vectors counted once.  Matrices
    and parameter vectors take the storage type's size e; per-row outputs
    and labels are 4 bytes."""
    rc = rows * cols
    e = ELEM_BYTES[dtype]
    if op == "rmsnorm":
        return 2 * e * rc + e * cols
    if op == "layernorm":
        return 2 * e * rc + 2 * e * cols
    if op == "residual_layernorm":
        return 3 * e * rc + 2 * e * cols + (e * rc if h_out else 0)
    if op == "softmax":
        return 2 * e * rc
    if op == "row_sum":
        return e * rc + 4 * rows
    if op == "cross_entropy":
        return e * rc + 8 * rows + (4 if mean else 0)
    if op == "residual_rmsnorm":
        return 3 * e * rc + e * cols + (e * rc if h_out else 0)
    if op == "log_softmax":
        return 2 * e * rc
    raise ValueError(op)


def _device(a, dtype):
    import numpy as np
    import torch
    if dtype == "bf16" and a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


class Workload:
    """Buffer pool plus prepared raw C-ABI calls for one shape."""

    def __init__(self, op, rows, cols, seed, outliers=False,
                 l2_bytes=126 << 20, max_pool_bytes=16 << 30, data=None,
                 dtype="f32"):
        import torch
        self.op, self.rows, self.cols, self.dtype = op, rows, cols, dtype
        d = data if data is not None else inputs.make(op, rows, cols, seed,
                                                      outliers=outliers)
        d = inputs.as_storage(d, dtype)
        self.host = d
        self.eps = float(d.get("eps", 0.0))
        self.mean = op == "cross_entropy"
        self.h_out = op in ("residual_layernorm", "residual_rmsnorm")
        self.bytes = algorithmic_bytes(op, rows, cols, self.h_out, self.mean,
                                       dtype)
        params = {k: _device(d[k], dtype) for k in
                  ("weight", "gamma", "beta") if k in d}
        set_bytes = max(self.bytes, 1)
        n = max(1, math.ceil(4 * l2_bytes / set_bytes))
        n = max(1, min(n, max_pool_bytes // set_bytes, MAX_SETS))
        x0 = _device(d["x"], dtype)
        self.sets = []
        for _ in range(n):
            s = dict(params)
            s["x"] = x0.clone()
            if "residual" in d:
                s["residual"] = _device(d["residual"], dtype)
            if "labels" in d:
                s["labels"] = torch.from_numpy(d["labels"]).cuda()
            if op in ("rmsnorm", "layernorm", "softmax", "log_softmax",
                      "residual_layernorm", "residual_rmsnorm"):
                s["y"] = torch.empty_like(x0)
            if self.h_out:
                s["h_out"] = torch.empty_like(x0)
            if op == "row_sum":
                s["out"] = torch.empty(rows, device="cuda")
            if op == "cross_entropy":
                s["loss"] = torch.empty(rows, device="cuda")
                s["mean_loss"] = torch.empty(1, device="cuda")
            self.sets.append(s)
        del x0
        self.pool_bytes = n * set_bytes
        self.l2_resident = self.pool_bytes < 4 * l2_bytes
        self.launches_per_step = 2 if self.mean else 1

    def outputs(self, i=0):
        s = self.sets[i % len(self.sets)]
        return {k: s[k] for k in ("y", "h_out", "out", "loss", "mean_loss")
                if k in s}

    def call_fn(self, i, stream_handle, plan=None):
        """A zero-argument callable issuing step i's C-ABI call (the plain
        entry point, or the *_with_plan one when `plan` is given)."""
        L = B.lib()
        s = self.sets[i % len(self.sets)]

        def P(k):
            return s[k].data_ptr() if k in s else None
        R, C, eps = self.rows, self.cols, ctypes.c_float(self.eps)
        st = stream_handle
        names = {"rmsnorm": (("x", "weight", "y"), True),
                 "layernorm": (("x", "gamma", "beta", "y"), True),
                 "residual_layernorm": (("x", "residual", "gamma", "beta",
                                         "y", "h_out"), True),
                 "softmax": (("x", "y"), False),
                 "row_sum": (("x", "out"), False),
                 "cross_entropy": (("x", "labels", "loss", "mean_loss"),
                                   False),
                 "residual_rmsnorm": (("x", "residual", "weight", "y",
                                       "h_out"), True),
                 "log_softmax": (("x", "y"), False)}
        keys, has_eps = names[self.op]
        if plan is not None:
            self._plan_ref = plan if isinstance(plan, B.MtPlan) else \
                B.MtPlan(**plan)
        if plan is not None and self.dtype != "f32":
            # op, dtype, x, residual, weight, beta, labels, y, h_out, out,
            # mean_loss, rows, cols, eps, stream, plan
            fname = "mt_row_reduce_with_plan"
            args = (B.OP_IDS[self.op], B.DTYPE_IDS[self.dtype], P("x"),
                    P("residual"), P("weight") or P("gamma"), P("beta"),
                    P("labels"), B.MT_NO_IGNORE_INDEX, P("y"), P("h_out"),
                    P("out") or P("loss"), P("mean_loss"), R, C, eps, st,
                    ctypes.byref(self._plan_ref))
        else:
            args = [P(k) for k in keys] + [R, C] + ([eps] if has_eps else [])
            args.append(st)
            fname = f"mt_{self.op}_{self.dtype}"
            if plan is not None:
                fname += "_with_plan"
                args.append(ctypes.byref(self._plan_ref))
            args = tuple(args)
        f = getattr(L, fname)

        def go():
            rc = f(*args)
            if rc != 0:
                raise B.MTError(rc, fname)
        return go


def _graph_of(work, count, stream, plan=None):
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        h = torch.cuda.current_stream().cuda_stream
        for i in range(count):
            work.call_fn(i, h, plan)()
    return g


def graph_size(work, per_graph=64):
    n = len(work.sets)
    return n * max(1, math.ceil(per_graph / n))


def time_graph_steps(work, steps, warmup, plan=None, per_graph=64,
                     barrier=None, sampler=None):
    """Device seconds for exactly `steps` steps (after `warmup` steps),
    replayed from CUDA graphs.  `sampler` (a context manager) runs around
    the timed region; `barrier` is called before and after it."""
    import torch
    stream = torch.cuda.Stream()
    h = stream.cuda_stream
    with torch.cuda.stream(stream):
        for i in range(3):              # fill the library's per-device caches
            work.call_fn(i, h, plan)()
    stream.synchronize()
    G = min(graph_size(work, per_graph), max(1, steps))
    full = _graph_of(work, G, stream, plan)
    rem = steps % G
    tail = _graph_of(work, rem, stream, plan) if rem else None
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / G))):
            full.replay()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(steps // G):
                full.replay()
            if tail is not None:
                tail.replay()
            end.record(stream)
        end.synchronize()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return start.elapsed_time(end) / 1e3


def time_rounds(work, plan=None, rounds=5, min_round_s=0.01, per_graph=64):
    """Per-round µs/op of `rounds` timed rounds (graph replays), each at
    least `min_round_s` long; returns the list."""
    import torch
    stream = torch.cuda.Stream()
    h = stream.cuda_stream
    with torch.cuda.stream(stream):
        for i in range(3):
            work.call_fn(i, h, plan)()
    stream.synchronize()
    G = graph_size(work, per_graph)
    g = _graph_of(work, G, stream, plan)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        g.replay()
        start.record(stream)
        g.replay()
        end.record(stream)
    end.synchronize()
    one = max(start.elapsed_time(end) / 1e3, 1e-6)
    reps = max(1, math.ceil(min_round_s / one))
    out = []
    for _ in range(rounds):
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(reps):
                g.replay()
            end.record(stream)
        end.synchronize()
        out.append(start.elapsed_time(end) * 1e3 / (reps * G))
    del g
    return out


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def time_plain_steps(work, steps, warmup):
    """The same steps, each launched from Python (host launch cost in)."""
    import torch
    stream = torch.cuda.Stream()
    h = stream.cuda_stream
    fns = [work.call_fn(i, h) for i in range(len(work.sets))]
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fns[i % len(fns)]()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for i in range(steps):
            fns[i % len(fns)]()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / 1e3


def _e2e_host_buffers(work):
    import torch
    hx = work.host["x"]
    x_host = (torch.from_numpy(hx.view("int16")).view(torch.bfloat16)
              if work.dtype == "bf16" else torch.from_numpy(hx)).pin_memory()
    out_key = {"row_sum": "out", "cross_entropy": "loss"}.get(work.op, "y")
    return x_host, out_key


def time_e2e(work, steps, warmup, depth=1):
    """Each step copies x from pinned host memory, calls the library and
    copies the result back to pinned host memory.  Returns (seconds,
    host-to-device bytes per step, device-to-host bytes per step).

    depth = 1 runs the steps one after another on one stream.  depth > 1
    rotates that many device buffer sets, pinned result buffers and streams,
    so one step's upload overlaps earlier steps' kernels and downloads (the
    two copy directions use separate copy engines); each step still moves
    its own input and result inside the timed region."""
    import torch
    depth = max(1, min(depth, len(work.sets)))
    x_host, out_key = _e2e_host_buffers(work)
    s0 = work.sets[0]
    outs = [torch.empty(s0[out_key].shape, dtype=s0[out_key].dtype,
                        pin_memory=True) for _ in range(depth)]
    streams = [torch.cuda.Stream() for _ in range(depth)]
    fns = [work.call_fn(b, streams[b].cuda_stream) for b in range(depth)]

    def step(k):
        b = k % depth
        s = work.sets[b]
        with torch.cuda.stream(streams[b]):
            s["x"].copy_(x_host, non_blocking=True)
            fns[b]()
            outs[b].copy_(s[out_key], non_blocking=True)

    for k in range(max(warmup, depth)):
        step(k)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    done = [torch.cuda.Event() for _ in range(depth)]
    start.record(streams[0])
    for st in streams[1:]:
        st.wait_event(start)
    for k in range(steps):
        step(k)
    for b in range(1, depth):
        done[b].record(streams[b])
        streams[0].wait_event(done[b])
    end.record(streams[0])
    end.synchronize()
    return (start.elapsed_time(end) / 1e3,
            x_host.numel() * x_host.element_size(),
            outs[0].numel() * outs[0].element_size())
