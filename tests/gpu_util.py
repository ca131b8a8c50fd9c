"""Helpers for the GPU parity tests: guarded device buffers and the
element-wise tolerance check against the oracle.

Tolerance: an FP32 output element passes when |gpu - ref| <= 1e-5*(1+|ref|),
ref being the oracle's double value; NaN must match NaN.
"""
import numpy as np
import torch

RTOL = 1e-5
PAD = 64  # guard floats on each side of every buffer


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    both_nan = np.isnan(got) & np.isnan(ref)
    err = np.abs(got - ref)
    tol = RTOL * (1.0 + np.abs(ref))
    bad = ~((err <= tol) | both_nan)
    if bad.any():
        idx = np.argwhere(bad)
        i = tuple(idx[0])
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements outside "
            f"1e-5*(1+|ref|); first at {i}: gpu={got[i]!r} ref={ref[i]!r}; "
            f"max err/tol={np.nanmax(np.where(bad, err / tol, 0)):.3g}")


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
