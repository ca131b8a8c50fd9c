"""Seeded synthetic inputs for the six per-row operators.

This module only draws random numbers; it holds none of the operators'
arithmetic.  The tests, the benchmark and the smoke check use it to feed the
same inputs to the CUDA library and to the CPU oracle.

Recipe (NumPy ``default_rng(seed)``, PCG64, FP32 draws):

* x ~ N(0, 1); with ``outliers=True`` a mask ``rng.random(shape) < 0.01``
  selects about 1% of the entries, which are scaled by 100.
* softmax and cross-entropy inputs are N(0, 2^2).
* RMSNorm weight and LayerNorm gamma ~ 1 + 0.1 N(0, 1); beta ~ 0.1 N(0, 1).
* residual ~ N(0, 1).
* labels ~ uniform integers in [0, cols), int32.
* eps: 1e-6 for RMSNorm, 1e-5 for LayerNorm and residual LayerNorm.

The tuning seed is ``TUNE_SEED``; held-out validation uses ``HOLDOUT_SEED``.
Workload ``k`` of a list uses ``seed + k``.

For FP16 / BF16 storage the FP32 draws are rounded to the storage type
(round to nearest even) by :func:`as_storage`; :func:`widen` gives back their
exact FP32 values, which is what the oracle receives.
"""
from __future__ import annotations

import numpy as np

TUNE_SEED = 20260905
HOLDOUT_SEED = 20261202

OPS = ("rmsnorm", "layernorm", "residual_layernorm", "softmax", "row_sum",
       "cross_entropy")
# Fused variants built on the same engine.
FUSED_OPS = ("residual_rmsnorm", "log_softmax")
ALL_OPS = OPS + FUSED_OPS

RMS_EPS = 1e-6
LN_EPS = 1e-5

# The published RMSNorm shapes: an odd single row (tail path), short odd rows
# (row packing), few wide rows (cross-warp cooperation), then the bandwidth
# sweep, whose shapes carry 1% outliers.
RMSNORM_SHAPES = [(1, 127), (17, 257), (64, 4096)]
RMSNORM_SWEEP = [(1024, 4096), (16384, 4096), (65536, 4096), (8192, 1024),
                 (8192, 8192), (8192, 16384)]
# The operator-family shapes.
FAMILY_SHAPES = [(1, 127), (17, 257), (64, 4096), (1024, 4096)]


def _normal(rng, shape, scale=1.0):
    a = rng.standard_normal(shape, dtype=np.float32)
    if scale != 1.0:
        a *= np.float32(scale)
    return a


def make(op: str, rows: int, cols: int, seed: int, outliers: bool = False,
         affine: bool = True) -> dict:
    """Inputs for one call of ``op`` on a rows x cols FP32 matrix.

    Returns a dict with NumPy arrays (``x`` and, per op, ``weight``,
    ``gamma``, ``beta``, ``residual``, ``labels``) and the scalar ``eps``.
    ``affine=False`` leaves the weight / gamma / beta out (identity).
    """
    rng = np.random.default_rng(seed)
    shape = (rows, cols)
    if op in ("softmax", "cross_entropy", "log_softmax"):
        x = _normal(rng, shape, 2.0)
    else:
        x = _normal(rng, shape)
    if outliers:
        mask = rng.random(shape, dtype=np.float32) < np.float32(0.01)
        x[mask] *= np.float32(100.0)
    d = {"x": x}
    if op in ("rmsnorm", "residual_rmsnorm"):
        d["eps"] = RMS_EPS
        if op == "residual_rmsnorm":
            d["residual"] = _normal(rng, shape)
        if affine:
            d["weight"] = np.float32(1.0) + _normal(rng, (cols,), 0.1)
    elif op in ("layernorm", "residual_layernorm"):
        d["eps"] = LN_EPS
        if op == "residual_layernorm":
            d["residual"] = _normal(rng, shape)
        if affine:
            d["gamma"] = np.float32(1.0) + _normal(rng, (cols,), 0.1)
            d["beta"] = _normal(rng, (cols,), 0.1)
    elif op == "cross_entropy":
        d["labels"] = rng.integers(0, cols, rows, dtype=np.int32)
    elif op in ("softmax", "row_sum", "log_softmax"):
        pass
    else:
        raise ValueError(f"unknown op {op!r}")
    return d


def integer_valued(rows: int, cols: int, seed: int, lo: int = -8,
                   hi: int = 8) -> np.ndarray:
    """Small integers stored as FP32: every partial sum of a row of up to
    2^20 of them is an exact FP32 integer, whatever the addition order."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, (rows, cols)).astype(np.float32)


STORAGE = ("f32", "f16", "bf16")
_MATRICES = ("x", "residual", "weight", "gamma", "beta")


def _bf16_bits(a: np.ndarray) -> np.ndarray:
    """FP32 -> bfloat16 bit patterns, round to nearest even (NaN kept)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + (((u >> 16) & 1) + 0x7FFF)) >> 16
    r = np.where(np.isnan(a), (u >> 16) | 0x40, r)
    return r.astype(np.uint16)


def as_storage(d: dict, dtype: str) -> dict:
    """The same inputs with matrices and parameter vectors in `dtype`
    storage: float32 arrays for "f32", float16 for "f16", and uint16 bit
    patterns for "bf16".  Labels and eps are unchanged."""
    if dtype == "f32":
        return dict(d)
    out = dict(d)
    for k in _MATRICES:
        if k in d:
            out[k] = (d[k].astype(np.float16) if dtype == "f16"
                      else _bf16_bits(d[k]))
    return out


def widen(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact FP32 values of an array in `dtype` storage."""
    if dtype == "bf16":
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32)


def widen_all(d: dict, dtype: str) -> dict:
    """`widen` applied to every matrix and parameter vector of `d`."""
    out = dict(d)
    for k in _MATRICES:
        if k in d:
            out[k] = widen(d[k], dtype)
    return out
