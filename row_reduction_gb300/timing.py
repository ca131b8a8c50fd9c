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
                 dtype="f32", ce_mean=True):
        import torch
        self.op, self.rows, self.cols, self.dtype = op, rows, cols, dtype
        d = data if data is not None else inputs.make(op, rows, cols, seed,
                                                      outliers=outliers)
        d = inputs.as_storage(d, dtype)
        self.host = d
        self.eps = float(d.get("eps", 0.0))
        # Cross-entropy: with the batch mean (a second, one-CTA kernel) or
        # the per-row losses alone (mean_loss = NULL).
        self.mean = op == "cross_entropy" and ce_mean
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
                if self.mean:
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


def _replay_for(graph, stream, seconds, until=None, max_seconds=5.0):
    """Replays `graph` on `stream` for about `seconds` (and, when `until` is
    given, until it returns True or `max_seconds` have passed)."""
    import time
    import torch
    t0 = time.perf_counter()
    while True:
        with torch.cuda.stream(stream):
            graph.replay()
        stream.synchronize()
        el = time.perf_counter() - t0
        if el >= max_seconds:
            return
        if el >= seconds and (until is None or until()):
            return


# Largest K timed as one graph (spacer, K steps and both timing events in a
# single CUDA graph); longer runs replay graphs of whole pool cycles.
MAX_ONE_GRAPH_STEPS = 4096


def _graph_with_events(work, spacer, steps, stream, start, end, plan=None):
    """One CUDA graph: `spacer` untimed steps, then `steps` timed steps,
    with the timing events as graph nodes.  The start event hangs off a
    side branch that depends on the last untimed step, so the chain of
    programmatic dependent launches through the timed steps is never broken
    by it: the window runs from the completion of the last untimed step to
    the completion of the last timed step, which is `steps` steps of the
    steady chain."""
    import torch
    side = torch.cuda.Stream()
    fork = torch.cuda.Event()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        cur = torch.cuda.current_stream()
        h = cur.cuda_stream
        for i in range(spacer):
            work.call_fn(i, h, plan)()
        fork.record(cur)
        side.wait_event(fork)
        start.record(side)
        for i in range(steps):
            work.call_fn(spacer + i, h, plan)()
        end.record(cur)
        cur.wait_stream(side)
    return g


def time_graph_steps(work, steps, warmup, plan=None, per_graph=64,
                     barrier=None, sampler=None, load_s=0.3):
    """Device seconds for exactly `steps` steps (after at least `warmup`
    steps), replayed from CUDA graphs.

    The timed region is bracketed by a synchronize (and `barrier`, when
    given) on both sides.  Up to MAX_ONE_GRAPH_STEPS steps are timed inside
    one graph that first runs a pool cycle of untimed steps
    (_graph_with_events), so the timed steps follow a busy GPU and their
    launch chain is unbroken.  Longer runs record the start event after an
    untimed graph (a spacer) and replay graphs of whole pool cycles.  With
    `sampler` (an object with start(), stop() and has_samples(n)), the GPU
    also runs the same steps for `load_s` seconds before and after the
    timed region (before: until the sampler holds at least two samples),
    so clock samples are taken under the timed load."""
    import torch
    stream = torch.cuda.Stream()
    h = stream.cuda_stream
    with torch.cuda.stream(stream):
        for i in range(3):              # fill the library's per-device caches
            work.call_fn(i, h, plan)()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True, external=True)
    end = torch.cuda.Event(enable_timing=True, external=True)
    G = min(graph_size(work, per_graph), max(1, steps))
    spacer = _graph_of(work, graph_size(work, per_graph), stream, plan)
    one = None
    full = tail = None
    if steps <= MAX_ONE_GRAPH_STEPS:
        one = _graph_with_events(work, graph_size(work, per_graph), steps,
                                 stream, start, end, plan)
    else:
        full = _graph_of(work, G, stream, plan)
        rem = steps % G
        tail = _graph_of(work, rem, stream, plan) if rem else None
    warm = full if full is not None else spacer
    with torch.cuda.stream(stream):
        for _ in range(max(1, math.ceil(warmup / graph_size(work,
                                                            per_graph)))):
            warm.replay()
        spacer.replay()
    stream.synchronize()
    if sampler is not None:
        sampler.start()
        _replay_for(spacer, stream, load_s,
                    until=lambda: sampler.has_samples(2))
    torch.cuda.synchronize()
    if barrier:
        barrier()
    with torch.cuda.stream(stream):
        if one is not None:
            one.replay()
        else:
            spacer.replay()             # untimed
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
    if sampler is not None:
        _replay_for(spacer, stream, load_s)
        sampler.stop()
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


class CopyProbe:
    """The library's plain copy kernel (mt_probe_copy) over a workload's own
    buffer pool: step i copies set i's x to its y, the same bytes in and out
    as one RMSNorm or softmax step (without the parameter vector).  Timed
    like a workload, it is the floor of a launch that moves those bytes."""

    def __init__(self, work, threads=512, unroll=4, grid=0, flags=0):
        self.work, self.sets = work, work.sets
        self.threads, self.unroll, self.grid = threads, unroll, grid
        self.flags = flags
        x0 = work.sets[0]["x"]
        self.nbytes = x0.numel() * x0.element_size()
        self.bytes = 2 * self.nbytes

    def call_fn(self, i, stream_handle, plan=None):
        L = B.lib()
        s = self.sets[i % len(self.sets)]
        args = (s["x"].data_ptr(), s["y"].data_ptr(), self.nbytes,
                self.threads, self.unroll, self.grid, self.flags,
                stream_handle)

        def go():
            rc = L.mt_probe_copy(*args)
            if rc != 0:
                raise B.MTError(rc, "mt_probe_copy")
        return go


class ReadProbe:
    """The library's read kernel (mt_probe_read) over a workload's own
    buffer pool: step i reads set i's x, the same bytes in as one row-sum
    or cross-entropy step, and writes one word per CTA.  The floor of a
    launch that reads those bytes."""

    def __init__(self, work, threads=512, unroll=4, grid=0, flags=0):
        import torch
        self.work, self.sets = work, work.sets
        self.threads, self.unroll, self.grid = threads, unroll, grid
        self.flags = flags
        x0 = work.sets[0]["x"]
        self.nbytes = x0.numel() * x0.element_size()
        self.bytes = self.nbytes
        self.words = max(grid, 152 * 64, 1)
        self.out = [torch.empty(self.words, dtype=torch.int32, device="cuda")
                    for _ in range(len(work.sets))]

    def call_fn(self, i, stream_handle, plan=None):
        L = B.lib()
        s = self.sets[i % len(self.sets)]
        args = (s["x"].data_ptr(), self.nbytes,
                self.out[i % len(self.sets)].data_ptr(), self.words,
                self.threads, self.unroll, self.grid, self.flags,
                stream_handle)

        def go():
            rc = L.mt_probe_read(*args)
            if rc != 0:
                raise B.MTError(rc, "mt_probe_read")
        return go


class EmptyProbe:
    """The library's empty kernel (mt_probe_empty): a chain of dependent
    launches that move nothing, the fixed cost of one step."""

    def __init__(self, threads=32, grid=1):
        self.sets = [None]
        self.threads, self.grid = threads, grid
        self.bytes = 0

    def call_fn(self, i, stream_handle, plan=None):
        L = B.lib()
        args = (self.threads, self.grid, stream_handle)

        def go():
            rc = L.mt_probe_empty(*args)
            if rc != 0:
                raise B.MTError(rc, "mt_probe_empty")
        return go


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


def time_link(h2d_bytes, d2h_bytes, steps, warmup, depth=3):
    """The host link alone: each step copies `h2d_bytes` from pinned host
    memory to the device and `d2h_bytes` from the device to pinned host
    memory, with the same rotation over `depth` streams and buffers as
    :func:`time_e2e` (so the two directions overlap on their copy engines).
    Returns seconds for `steps` steps: the ceiling an end-to-end step that
    moves those bytes can reach."""
    import torch
    depth = max(1, depth)
    n_in, n_out = max(1, h2d_bytes), max(1, d2h_bytes)
    h_in = torch.empty(n_in, dtype=torch.uint8, pin_memory=True)
    h_out = [torch.empty(n_out, dtype=torch.uint8, pin_memory=True)
             for _ in range(depth)]
    d_in = [torch.empty(n_in, dtype=torch.uint8, device="cuda")
            for _ in range(depth)]
    d_out = [torch.empty(n_out, dtype=torch.uint8, device="cuda")
             for _ in range(depth)]
    streams = [torch.cuda.Stream() for _ in range(depth)]

    def step(k):
        b = k % depth
        with torch.cuda.stream(streams[b]):
            d_in[b].copy_(h_in, non_blocking=True)
            h_out[b].copy_(d_out[b], non_blocking=True)

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
    return start.elapsed_time(end) / 1e3
