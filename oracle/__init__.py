"""CPU oracle for the per-row FP32 reduction operators.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` import this package.  The product library
(``row_reduction_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, double accumulation, one row at
a time); this module compiles it with gcc and wraps it for NumPy arrays.
Every function returns float64 arrays: the value before the single FP32
rounding the GPU path applies at its store.

Definitions, per row of n = cols entries (see the header of ``oracle.c``):

* ``rmsnorm``  y = x / sqrt(sum(x^2)/n + eps) * w  -- the ``rmsnorm_register``
  kernel (Thread Ownership and Software Staging, §Register-tiled reductions).
* ``layernorm`` / ``residual_layernorm`` / ``softmax`` / ``row_sum`` /
  ``cross_entropy`` -- the operator coverage list of "Consecutive-worker
  reduction layout checkpoint", §Evidence and what remains; the pages name
  them without formulas, so the textbook definitions are used.
* ``residual_rmsnorm``, ``log_softmax``, ``cross_entropy_ignore`` -- fused
  variants on the same rows, the plain compositions of those definitions.

Pins: ``tests/test_oracle_pins.py`` checks every function against closed
forms, invariants, exactly-rounded sums and torch float64 library routines;
``tests/test_oracle_mutations.py`` plants slips in a copy of ``oracle.c`` and
checks that the pins catch each one (it points ``ORACLE_LIB`` at the
mutant's library; unset, the module builds and loads ``liboracle.so``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, -O2)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", "-fvisibility=hidden", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ORACLE_LIB")
            if not path:
                path = build()
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int64
            D = ctypes.c_double
            lib.oracle_rmsnorm_f64.argtypes = [P, P, I, I, D, P]
            lib.oracle_layernorm_f64.argtypes = [P, P, P, I, I, D, P, P]
            lib.oracle_residual_layernorm_f64.argtypes = [P, P, P, P, I, I, D,
                                                          P, P, P]
            lib.oracle_softmax_f64.argtypes = [P, I, I, P]
            lib.oracle_row_sum_f64.argtypes = [P, I, I, P]
            lib.oracle_cross_entropy_f64.argtypes = [P, P, I, I, P, P]
            lib.oracle_residual_rmsnorm_f64.argtypes = [P, P, P, I, I, D, P,
                                                        P]
            lib.oracle_log_softmax_f64.argtypes = [P, I, I, P]
            lib.oracle_cross_entropy_ignore_f64.argtypes = [
                P, P, ctypes.c_int32, I, I, P, P]
            for f in (lib.oracle_rmsnorm_f64, lib.oracle_layernorm_f64,
                      lib.oracle_residual_layernorm_f64,
                      lib.oracle_softmax_f64, lib.oracle_row_sum_f64,
                      lib.oracle_cross_entropy_f64,
                      lib.oracle_residual_rmsnorm_f64,
                      lib.oracle_log_softmax_f64,
                      lib.oracle_cross_entropy_ignore_f64):
                f.restype = None
            _lib = lib
    return _lib


def _f32(a, name):
    a = np.ascontiguousarray(a, dtype=np.float32)
    if a.ndim != 2:
        raise ValueError(f"{name} must be 2-D (rows, cols)")
    return a


def _vec(a, cols, name):
    if a is None:
        return None
    a = np.ascontiguousarray(a, dtype=np.float32).reshape(-1)
    if a.shape[0] != cols:
        raise ValueError(f"{name} must have cols={cols} entries")
    return a


def _p(a):
    return None if a is None else a.ctypes.data


def rmsnorm(x, weight=None, eps=1e-6):
    """y = x / sqrt(mean(x^2) + eps) * weight, per row, float64 result."""
    x = _f32(x, "x")
    rows, cols = x.shape
    w = _vec(weight, cols, "weight")
    y = np.empty((rows, cols), dtype=np.float64)
    _load().oracle_rmsnorm_f64(_p(x), _p(w), rows, cols,
                               float(np.float32(eps)), _p(y))
    return y


def layernorm(x, gamma=None, beta=None, eps=1e-5):
    """y = (x - mean) / sqrt(var + eps) * gamma + beta, biased variance."""
    x = _f32(x, "x")
    rows, cols = x.shape
    g = _vec(gamma, cols, "gamma")
    b = _vec(beta, cols, "beta")
    y = np.empty((rows, cols), dtype=np.float64)
    scratch = np.empty(cols, dtype=np.float64)
    _load().oracle_layernorm_f64(_p(x), _p(g), _p(b), rows, cols,
                                 float(np.float32(eps)), _p(y), _p(scratch))
    return y


def residual_layernorm(x, residual, gamma=None, beta=None, eps=1e-5):
    """Returns (y, h_out): y = layernorm(x + residual); h_out = fp32(x + r)."""
    x = _f32(x, "x")
    r = _f32(residual, "residual")
    if r.shape != x.shape:
        raise ValueError("residual must match x")
    rows, cols = x.shape
    g = _vec(gamma, cols, "gamma")
    b = _vec(beta, cols, "beta")
    y = np.empty((rows, cols), dtype=np.float64)
    h = np.empty((rows, cols), dtype=np.float32)
    scratch = np.empty(cols, dtype=np.float64)
    _load().oracle_residual_layernorm_f64(_p(x), _p(r), _p(g), _p(b), rows,
                                          cols, float(np.float32(eps)), _p(y),
                                          _p(h), _p(scratch))
    return y, h


def softmax(x):
    """y = exp(x - max) / sum(exp(x - max)), per row."""
    x = _f32(x, "x")
    rows, cols = x.shape
    y = np.empty((rows, cols), dtype=np.float64)
    _load().oracle_softmax_f64(_p(x), rows, cols, _p(y))
    return y


def row_sum(x):
    """out[r] = sum of row r."""
    x = _f32(x, "x")
    rows, cols = x.shape
    out = np.empty(rows, dtype=np.float64)
    _load().oracle_row_sum_f64(_p(x), rows, cols, _p(out))
    return out


def cross_entropy(logits, labels):
    """Returns (loss, mean): loss[r] = logsumexp(row) - row[label[r]]."""
    x = _f32(logits, "logits")
    rows, cols = x.shape
    lab = np.ascontiguousarray(labels, dtype=np.int32).reshape(-1)
    if lab.shape[0] != rows:
        raise ValueError("labels must have rows entries")
    loss = np.empty(rows, dtype=np.float64)
    mean = np.empty(1, dtype=np.float64)
    _load().oracle_cross_entropy_f64(_p(x), _p(lab), rows, cols, _p(loss),
                                     _p(mean))
    return loss, float(mean[0])


def residual_rmsnorm(x, residual, weight=None, eps=1e-6):
    """Returns (y, h_out): y = rmsnorm(x + residual); h_out = fp32(x + r)."""
    x = _f32(x, "x")
    r = _f32(residual, "residual")
    if r.shape != x.shape:
        raise ValueError("residual must match x")
    rows, cols = x.shape
    w = _vec(weight, cols, "weight")
    y = np.empty((rows, cols), dtype=np.float64)
    h = np.empty((rows, cols), dtype=np.float32)
    _load().oracle_residual_rmsnorm_f64(_p(x), _p(r), _p(w), rows, cols,
                                        float(np.float32(eps)), _p(y), _p(h))
    return y, h


def log_softmax(x):
    """y = (x - max) - log(sum(exp(x - max))), per row."""
    x = _f32(x, "x")
    rows, cols = x.shape
    y = np.empty((rows, cols), dtype=np.float64)
    _load().oracle_log_softmax_f64(_p(x), rows, cols, _p(y))
    return y


def cross_entropy_ignore(logits, labels, ignore_index):
    """(loss, mean) with rows labelled `ignore_index` given loss 0 and left
    out of the mean."""
    x = _f32(logits, "logits")
    rows, cols = x.shape
    lab = np.ascontiguousarray(labels, dtype=np.int32).reshape(-1)
    if lab.shape[0] != rows:
        raise ValueError("labels must have rows entries")
    loss = np.empty(rows, dtype=np.float64)
    mean = np.empty(1, dtype=np.float64)
    _load().oracle_cross_entropy_ignore_f64(_p(x), _p(lab),
                                            int(ignore_index), rows, cols,
                                            _p(loss), _p(mean))
    return loss, float(mean[0])


def run(op: str, inputs: dict):
    """Dispatch by operator name on a dict made by the input generators.

    Returns a dict of float64 reference outputs keyed like the GPU outputs.
    """
    if op == "rmsnorm":
        return {"y": rmsnorm(inputs["x"], inputs.get("weight"),
                             inputs["eps"])}
    if op == "layernorm":
        return {"y": layernorm(inputs["x"], inputs.get("gamma"),
                               inputs.get("beta"), inputs["eps"])}
    if op == "residual_layernorm":
        y, h = residual_layernorm(inputs["x"], inputs["residual"],
                                  inputs.get("gamma"), inputs.get("beta"),
                                  inputs["eps"])
        return {"y": y, "h_out": h}
    if op == "softmax":
        return {"y": softmax(inputs["x"])}
    if op == "row_sum":
        return {"out": row_sum(inputs["x"])}
    if op == "cross_entropy":
        if inputs.get("ignore_index") is not None:
            loss, mean = cross_entropy_ignore(inputs["x"], inputs["labels"],
                                              inputs["ignore_index"])
        else:
            loss, mean = cross_entropy(inputs["x"], inputs["labels"])
        return {"loss": loss, "mean_loss": np.array([mean])}
    if op == "residual_rmsnorm":
        y, h = residual_rmsnorm(inputs["x"], inputs["residual"],
                                inputs.get("weight"), inputs["eps"])
        return {"y": y, "h_out": h}
    if op == "log_softmax":
        return {"y": log_softmax(inputs["x"])}
    raise ValueError(f"unknown op {op!r}")
