"""Helpers for the GPU parity tests: guarded device buffers and the
element-wise tolerance check against the oracle.

Tolerance: an FP32 output element passes when |gpu - ref| <= 1e-5*(1+|ref|),
ref being the oracle's double value; NaN must match NaN and an infinity the
same infinity.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

RTOL = 1e-5
PAD = 64  # guard floats on each side of every buffer


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    both_nan = np.isnan(got) & np.isnan(ref)
    with np.errstate(invalid="ignore"):
        err = np.abs(got - ref)
    with np.errstate(over="ignore"):
        tol = RTOL * (1.0 + np.abs(ref))
    # equal values pass, equal infinities included (log-softmax of -inf);
    # an infinite reference admits nothing else (its tolerance would be
    # infinite)
    bad = ~(((err <= tol) & np.isfinite(ref)) | both_nan | (got == ref))
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        with np.errstate(invalid="ignore", divide="ignore"):
            ratio = np.where(bad & np.isfinite(err / tol), err / tol, 0)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside "
            f"1e-5*(1+|ref|); first at {i}: gpu={got[i]!r} ref={ref[i]!r}; "
            f"max finite err/tol={np.max(ratio):.3g}")


class Guarded:
    """A device buffer of n FP32 (or int32) values at a chosen float offset
    inside a larger allocation whose guard region holds a fill pattern.

    Inputs are guarded with NaN so an out-of-bounds read poisons its row;
    outputs with a sentinel so an out-of-bounds write is caught by
    ``check()``."""

    SENTINEL = -12345.678

    def __init__(self, n, offset=0, fill=float("nan"), dtype=torch.float32,
                 data=None):
        self.n, self.offset = n, offset
        self.buf = torch.full((PAD + offset + n + PAD,), fill, dtype=dtype,
                              device="cuda")
        self.fill = fill
        self.view = self.buf[PAD + offset: PAD + offset + n]
        if data is not None:
            self.view.copy_(torch.as_tensor(np.ascontiguousarray(
                data).reshape(-1)))

    @property
    def ptr(self):
        return self.view.data_ptr()

    @staticmethod
    def _host(t):
        if t.dtype in (torch.float16, torch.bfloat16):
            t = t.float()
        return t.cpu().numpy()

    def numpy(self):
        return self._host(self.view)

    def check(self):
        head = self._host(self.buf[:PAD + self.offset])
        tail = self._host(self.buf[PAD + self.offset + self.n:])
        for part in (head, tail):
            if np.isnan(self.fill):
                assert np.isnan(part).all(), "guard region was written"
            else:
                assert (part == np.float32(self.fill)).all(), \
                    "guard region was written"


def to_dev(d):
    """Copies a generator dict to CUDA tensors (scalars pass through)."""
    out = {}
    for k, v in d.items():
        out[k] = torch.from_numpy(v).cuda() if isinstance(v, np.ndarray) \
            else v
    return out


def ulp(v, dt):
    """Unit in the last place of |v| in 16-bit storage type dt ("f16" or
    "bf16"), with the subnormal spacing below the smallest normal."""
    mant, emin = (7, -126) if dt == "bf16" else (10, -14)
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** emin)
    return 2.0 ** (np.floor(np.log2(a)) - mant)


def check_softmax_rows(got, ref, what, dt="f32", log=False):
    """Softmax checks beyond the element-wise tolerance, whose absolute floor
    1e-5*(1+|ref|) would hide errors in small probabilities:

    * every row whose reference holds no NaN sums to 1: |sum(y) - 1| <= 1e-5
      for FP32 storage; for 16-bit storage 1e-5 plus the rows's summed
      half-ulp rounding of the stored outputs;
    * probabilities below 1e-3 (and above 1e-30, far from the exponential's
      flush to zero) match in relative terms: for FP32
      |log y - log ref| <= 1e-5*(1+|log ref|), the log-softmax tolerance;
      for 16-bit |y - ref| <= half an ulp of ref*(1+2^-6) + 1e-5*ref.

    With log=True the outputs are log-probabilities (log-softmax): the sum
    check applies to exp(y) (FP32 only)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.ndim == 1:
        got, ref = got.reshape(1, -1), ref.reshape(1, -1)
    got = got.reshape(ref.shape)
    ok = ~np.isnan(ref).any(axis=1)
    if log:
        if dt == "f32" and ok.any():
            s = np.exp(got[ok]).sum(axis=1)
            bad = np.abs(s - 1.0) > 1e-5
            assert not bad.any(), (f"{what}: sum(exp(log-softmax)) off 1 by "
                                   f"{np.max(np.abs(s - 1.0)):.3g}")
        return
    if ok.any():
        s = got[ok].sum(axis=1)
        bound = 1e-5
        if dt != "f32":
            bound = bound + (0.5 * ulp(got[ok], dt)).sum(axis=1)
        bad = np.abs(s - 1.0) > bound
        assert not bad.any(), (f"{what}: {bad.sum()} rows do not sum to 1 "
                               f"(worst |sum-1| = "
                               f"{np.max(np.abs(s - 1.0)):.3g})")
    small = ok[:, None] & (ref < 1e-3) & (ref > 1e-30)
    if not small.any():
        return
    g, r = got[small], ref[small]
    if dt == "f32":
        assert (g > 0).all(), f"{what}: a small probability came out <= 0"
        err = np.abs(np.log(g) - np.log(r))
        tol = 1e-5 * (1 + np.abs(np.log(r)))
    else:
        err = np.abs(g - r)
        tol = 0.5 * ulp(r * (1 + 2.0 ** -6), dt) + 1e-5 * r
    bad = err > tol
    if bad.any():
        i = int(np.argmax(np.where(bad, err / tol, 0)))
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} small probabilities off in "
            f"relative terms; worst gpu={g[i]!r} ref={r[i]!r}")


def compare_row_blocks(got, ref_fn, check, what, block=2048):
    """Compares a host matrix `got` (rows x cols) with the oracle on every
    row: ref_fn(lo, hi) gives the oracle's rows [lo, hi) and check(g, r,
    label) compares them.  Row blocks run on parallel threads (the oracle's
    C code releases the interpreter lock), so memory stays bounded and a
    full-size matrix takes seconds."""
    rows = got.shape[0]
    bounds = [(lo, min(rows, lo + block)) for lo in range(0, rows, block)]

    def one(b):
        lo, hi = b
        check(got[lo:hi], ref_fn(lo, hi), f"{what} rows {lo}..{hi - 1}")
        return hi - lo

    with ThreadPoolExecutor(max(1, min(16, os.cpu_count() or 1))) as ex:
        done = sum(ex.map(one, bounds))
    assert done == rows
