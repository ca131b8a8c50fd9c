"""Pins for the CPU oracle: closed forms, invariants, exactly rounded sums and
torch float64 library routines.  None of these re-type the oracle's own
formula; each is chosen so that a plausible slip in ``oracle.c`` (a dropped
eps, eps outside the square root, n-1 instead of n, a missing max shift, a
wrong label index, stats taken from the wrong row) fails at least one.

RMSNorm is the ``rmsnorm_register`` kernel of "Thread Ownership and Software
Staging", §Register-tiled reductions; the other operators are the coverage
list of "Consecutive-worker reduction layout checkpoint", §Evidence and what
remains.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from row_reduction_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def f32(v):
    return float(np.float32(v))


def rows_of(*rows):
    return np.array(rows, dtype=np.float32)


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_hand_case_3_4(oracle_mod):
    eps = f32(1e-6)
    y = oracle_mod.rmsnorm(rows_of([3.0, 4.0]), None, eps)
    d = math.sqrt(12.5 + eps)          # mean of squares over n=2, not n-1
    assert np.allclose(y[0], [3 / d, 4 / d], rtol=1e-15, atol=0)
    assert abs(y[0, 0] - 0.8485281) < 1e-6


def test_rmsnorm_eps_inside_sqrt(oracle_mod):
    # x = [1, 1], eps = 1: 1/sqrt(1 + 1); eps outside would give 1/(1+1).
    y = oracle_mod.rmsnorm(rows_of([1.0, 1.0]), None, 1.0)
    assert np.allclose(y, 1 / math.sqrt(2.0), rtol=1e-15)


def test_rmsnorm_weight_hand_case(oracle_mod):
    eps = f32(1e-6)
    w = np.array([2.0, 0.5, -1.0], dtype=np.float32)
    y = oracle_mod.rmsnorm(rows_of([1.0, 2.0, 2.0]), w, eps)
    d = math.sqrt(3.0 + eps)
    assert np.allclose(y[0], [2 / d, 1 / d, -2 / d], rtol=1e-15)


def test_rmsnorm_single_element(oracle_mod):
    eps = f32(1e-6)
    y = oracle_mod.rmsnorm(rows_of([-0.5]), np.array([3.0], np.float32), eps)
    assert math.isclose(y[0, 0], -0.5 / math.sqrt(0.25 + eps) * 3.0,
                        rel_tol=1e-15)


def test_rmsnorm_unit_weight_mean_square(oracle_mod):
    # With unit weight, mean(y^2) = ms / (ms + eps) exactly (in real numbers).
    d = inputs.make("rmsnorm", 9, 301, seed=11, outliers=True, affine=False)
    eps = f32(1e-3)
    y = oracle_mod.rmsnorm(d["x"], None, eps)
    x = d["x"].astype(np.float64)
    ms = (x * x).mean(axis=1)
    assert np.allclose((y * y).mean(axis=1), ms / (ms + eps), rtol=1e-12)


def test_rmsnorm_matches_torch_f64(oracle_mod):
    d = inputs.make("rmsnorm", 5, 1000, seed=3)
    y = oracle_mod.rmsnorm(d["x"], d["weight"], d["eps"])
    t = F.rms_norm(torch.from_numpy(d["x"]).double(), (1000,),
                   torch.from_numpy(d["weight"]).double(), f32(d["eps"]))
    assert np.allclose(y, t.numpy(), rtol=1e-12, atol=1e-14)


def test_rows_are_independent(oracle_mod):
    d = inputs.make("rmsnorm", 6, 50, seed=5)
    y = oracle_mod.rmsnorm(d["x"], d["weight"], d["eps"])
    for r in range(6):
        yr = oracle_mod.rmsnorm(d["x"][r:r + 1], d["weight"], d["eps"])
        assert np.array_equal(y[r], yr[0])


# ---------------------------------------------------------------- LayerNorm
def test_layernorm_hand_case(oracle_mod):
    eps = f32(1e-5)
    y = oracle_mod.layernorm(rows_of([1.0, 2.0, 3.0]), None, None, eps)
    d = math.sqrt(2.0 / 3.0 + eps)      # biased variance 2/3
    assert np.allclose(y[0], [-1 / d, 0.0, 1 / d], rtol=1e-14, atol=1e-15)


def test_layernorm_affine_hand_case(oracle_mod):
    eps = f32(1e-5)
    g = np.array([2.0, -1.0, 0.5], np.float32)
    b = np.array([1.0, 0.25, -1.0], np.float32)
    y = oracle_mod.layernorm(rows_of([1.0, 2.0, 3.0]), g, b, eps)
    d = math.sqrt(2.0 / 3.0 + eps)
    assert np.allclose(y[0], [-2 / d + 1, 0.25, 0.5 / d - 1], rtol=1e-14)


def test_layernorm_single_element_gives_beta(oracle_mod):
    y = oracle_mod.layernorm(rows_of([7.0]), np.array([3.0], np.float32),
                             np.array([0.125], np.float32), f32(1e-5))
    assert y[0, 0] == 0.125


def test_layernorm_invariants(oracle_mod):
    d = inputs.make("layernorm", 7, 513, seed=9, affine=False)
    eps = f32(1e-2)
    y = oracle_mod.layernorm(d["x"], None, None, eps)
    x = d["x"].astype(np.float64)
    var = x.var(axis=1)
    assert np.allclose(y.mean(axis=1), 0.0, atol=1e-13)
    assert np.allclose(y.var(axis=1), var / (var + eps), rtol=1e-12)


def test_layernorm_matches_torch_f64(oracle_mod):
    d = inputs.make("layernorm", 4, 777, seed=4)
    y = oracle_mod.layernorm(d["x"], d["gamma"], d["beta"], d["eps"])
    t = F.layer_norm(torch.from_numpy(d["x"]).double(), (777,),
                     torch.from_numpy(d["gamma"]).double(),
                     torch.from_numpy(d["beta"]).double(), f32(d["eps"]))
    assert np.allclose(y, t.numpy(), rtol=1e-12, atol=1e-13)


# ------------------------------------------------------- residual LayerNorm
def test_residual_layernorm_is_layernorm_of_sum(oracle_mod):
    d = inputs.make("residual_layernorm", 3, 129, seed=8)
    y, h = oracle_mod.residual_layernorm(d["x"], d["residual"], d["gamma"],
                                         d["beta"], d["eps"])
    hs = torch.from_numpy(d["x"]).double() + torch.from_numpy(
        d["residual"]).double()
    t = F.layer_norm(hs, (129,), torch.from_numpy(d["gamma"]).double(),
                     torch.from_numpy(d["beta"]).double(), f32(d["eps"]))
    assert np.allclose(y, t.numpy(), rtol=1e-12, atol=1e-13)
    # h_out is the correctly rounded FP32 sum (one IEEE single add).
    assert np.array_equal(h.view(np.uint32),
                          (d["x"] + d["residual"]).view(np.uint32))


def test_residual_layernorm_zero_residual(oracle_mod):
    d = inputs.make("layernorm", 2, 64, seed=12)
    y0 = oracle_mod.layernorm(d["x"], d["gamma"], d["beta"], d["eps"])
    y1, h = oracle_mod.residual_layernorm(d["x"], np.zeros_like(d["x"]),
                                          d["gamma"], d["beta"], d["eps"])
    assert np.array_equal(y0, y1)
    assert np.array_equal(h, d["x"])


# ------------------------------------------------------------------ softmax
def test_softmax_hand_case(oracle_mod):
    y = oracle_mod.softmax(rows_of([0.0, f32(math.log(2)), f32(math.log(3))]))
    assert np.allclose(y[0], [1 / 6, 1 / 3, 1 / 2], rtol=1e-7)


def test_softmax_needs_max_shift(oracle_mod):
    # exp(1000) overflows double; only the max-shifted form gives 1/2.
    y = oracle_mod.softmax(rows_of([1000.0, 1000.0], [-1000.0, -1000.0]))
    assert np.array_equal(y, np.full((2, 2), 0.5))


def test_softmax_invariants(oracle_mod):
    d = inputs.make("softmax", 6, 4103, seed=2)
    y = oracle_mod.softmax(d["x"])
    assert np.allclose(y.sum(axis=1), 1.0, atol=1e-12)
    assert (y > 0).all()
    # Shift invariance (the shift is exact in FP32 for these magnitudes).
    y2 = oracle_mod.softmax(d["x"] + np.float32(0.5))
    assert np.allclose(y, y2, rtol=1e-6)
    assert np.allclose(oracle_mod.softmax(np.full((1, 10), 3.0, np.float32)),
                       0.1, rtol=1e-15)
    assert oracle_mod.softmax(rows_of([5.0]))[0, 0] == 1.0


def test_softmax_matches_torch_f64(oracle_mod):
    d = inputs.make("softmax", 5, 300, seed=1)
    y = oracle_mod.softmax(d["x"])
    t = torch.softmax(torch.from_numpy(d["x"]).double(), dim=1)
    assert np.allclose(y, t.numpy(), rtol=1e-12, atol=1e-16)


def test_softmax_nan_row(oracle_mod):
    y = oracle_mod.softmax(rows_of([1.0, float("nan"), 2.0], [1.0, 2.0, 3.0]))
    assert np.isnan(y[0]).all()
    assert np.isfinite(y[1]).all()


# ------------------------------------------------------------------ row sum
def test_row_sum_matches_fsum(oracle_mod):
    d = inputs.make("row_sum", 8, 4096, seed=6)
    s = oracle_mod.row_sum(d["x"])
    for r in range(8):
        exact = math.fsum(float(v) for v in d["x"][r])
        assert abs(s[r] - exact) <= 1e-12 * (1 + abs(exact))


def test_row_sum_integers_exact(oracle_mod):
    x = inputs.integer_valued(5, 1000, seed=3)
    s = oracle_mod.row_sum(x)
    assert np.array_equal(s, x.astype(np.int64).sum(axis=1).astype(np.float64))
    assert oracle_mod.row_sum(np.ones((2, 257), np.float32)).tolist() == [257.0,
                                                                          257.0]


# ------------------------------------------------------------ cross-entropy
def test_cross_entropy_hand_cases(oracle_mod):
    x = rows_of([0.0, f32(math.log(3))], [0.0, f32(math.log(3))])
    loss, mean = oracle_mod.cross_entropy(x, np.array([1, 0], np.int32))
    # softmax([0, ln3]) = [1/4, 3/4]
    assert math.isclose(loss[0], math.log(4 / 3), rel_tol=1e-7)
    assert math.isclose(loss[1], math.log(4), rel_tol=1e-7)
    assert math.isclose(mean, (math.log(4 / 3) + math.log(4)) / 2,
                        rel_tol=1e-7)


def test_cross_entropy_uniform_and_single(oracle_mod):
    loss, _ = oracle_mod.cross_entropy(np.full((3, 50), 2.5, np.float32),
                                       np.array([0, 17, 49], np.int32))
    assert np.allclose(loss, math.log(50), rtol=1e-15)
    loss1, _ = oracle_mod.cross_entropy(rows_of([4.0]),
                                        np.array([0], np.int32))
    assert loss1[0] == 0.0


def test_cross_entropy_needs_max_shift(oracle_mod):
    loss, _ = oracle_mod.cross_entropy(rows_of([1000.0, 0.0]),
                                       np.array([1], np.int32))
    assert math.isclose(loss[0], 1000.0, rel_tol=1e-15)


def test_cross_entropy_matches_torch_f64(oracle_mod):
    d = inputs.make("cross_entropy", 9, 1000, seed=5)
    loss, mean = oracle_mod.cross_entropy(d["x"], d["labels"])
    xt = torch.from_numpy(d["x"]).double()
    lt = torch.from_numpy(d["labels"]).long()
    t = F.cross_entropy(xt, lt, reduction="none")
    assert np.allclose(loss, t.numpy(), rtol=1e-12)
    assert math.isclose(mean, float(t.mean()), rel_tol=1e-12)
    assert (loss >= 0).all()
    # logsumexp minus the label logit
    lse = torch.logsumexp(xt, dim=1) - xt[torch.arange(9), lt]
    assert np.allclose(loss, lse.numpy(), rtol=1e-12)


def test_cross_entropy_bad_label_is_nan(oracle_mod):
    loss, mean = oracle_mod.cross_entropy(rows_of([1.0, 2.0], [1.0, 2.0]),
                                          np.array([2, 1], np.int32))
    assert math.isnan(loss[0]) and not math.isnan(loss[1])
    assert math.isnan(mean)
    loss, _ = oracle_mod.cross_entropy(rows_of([1.0, 2.0]),
                                       np.array([-1], np.int32))
    assert math.isnan(loss[0])


# ----------------------------------------------------------- input recipe
def test_generator_recipe():
    d = inputs.make("rmsnorm", 256, 1024, seed=1, outliers=True)
    x = d["x"]
    assert x.dtype == np.float32 and x.shape == (256, 1024)
    big = np.abs(x) > 20
    assert 0.007 < big.mean() < 0.013          # ~1% outliers scaled by 100
    assert abs(d["weight"].mean() - 1.0) < 0.02
    assert 0.08 < d["weight"].std() < 0.12
    s = inputs.make("softmax", 64, 4096, seed=2)["x"]
    assert 1.95 < s.std() < 2.05
    c = inputs.make("cross_entropy", 4096, 100, seed=3)["labels"]
    assert c.dtype == np.int32 and c.min() == 0 and c.max() == 99
    a = inputs.make("layernorm", 2, 8, seed=4)
    b = inputs.make("layernorm", 2, 8, seed=4)
    assert np.array_equal(a["x"], b["x"]) and np.array_equal(a["beta"],
                                                             b["beta"])


# ------------------------------------------------------ fused variants
def test_residual_rmsnorm_matches_torch_and_reduces_to_rmsnorm(oracle_mod):
    d = inputs.make("residual_rmsnorm", 4, 333, seed=21)
    y, h = oracle_mod.residual_rmsnorm(d["x"], d["residual"], d["weight"],
                                       d["eps"])
    hs = torch.from_numpy(d["x"]).double() + torch.from_numpy(
        d["residual"]).double()
    t = F.rms_norm(hs, (333,), torch.from_numpy(d["weight"]).double(),
                   f32(d["eps"]))
    assert np.allclose(y, t.numpy(), rtol=1e-12, atol=1e-14)
    assert np.array_equal(h.view(np.uint32),
                          (d["x"] + d["residual"]).view(np.uint32))
    y0, h0 = oracle_mod.residual_rmsnorm(d["x"], np.zeros_like(d["x"]),
                                         d["weight"], d["eps"])
    assert np.array_equal(y0, oracle_mod.rmsnorm(d["x"], d["weight"],
                                                 d["eps"]))
    # hand case: x + r = [3, 4]
    yh, _ = oracle_mod.residual_rmsnorm(rows_of([1.0, 5.0]),
                                        rows_of([2.0, -1.0]), None, 0.0)
    assert np.allclose(yh[0], [3 / math.sqrt(12.5), 4 / math.sqrt(12.5)],
                       rtol=1e-15)


def test_log_softmax_hand_cases_and_torch(oracle_mod):
    y = oracle_mod.log_softmax(rows_of([0.0, f32(math.log(2)),
                                        f32(math.log(3))]))
    assert np.allclose(y[0], [math.log(1 / 6), math.log(1 / 3),
                              math.log(1 / 2)], atol=1e-7)
    y = oracle_mod.log_softmax(rows_of([1000.0, 1000.0]))
    assert np.allclose(y, -math.log(2), rtol=1e-15)
    assert oracle_mod.log_softmax(rows_of([7.0]))[0, 0] == 0.0
    d = inputs.make("log_softmax", 6, 500, seed=22)
    y = oracle_mod.log_softmax(d["x"])
    t = torch.log_softmax(torch.from_numpy(d["x"]).double(), dim=1)
    assert np.allclose(y, t.numpy(), rtol=1e-12, atol=1e-12)
    assert np.allclose(np.exp(y).sum(axis=1), 1.0, atol=1e-12)
    assert np.isnan(oracle_mod.log_softmax(rows_of([1.0, np.nan]))).all()


def test_cross_entropy_ignore_index(oracle_mod):
    d = inputs.make("cross_entropy", 12, 300, seed=23)
    lab = d["labels"].copy()
    lab[[1, 4, 5]] = -100
    loss, mean = oracle_mod.cross_entropy_ignore(d["x"], lab, -100)
    xt = torch.from_numpy(d["x"]).double()
    lt = torch.from_numpy(lab).long()
    t = F.cross_entropy(xt, lt, ignore_index=-100, reduction="none")
    assert np.allclose(loss, t.numpy(), rtol=1e-12)
    assert loss[1] == 0.0 and loss[4] == 0.0
    tm = F.cross_entropy(xt, lt, ignore_index=-100, reduction="mean")
    assert math.isclose(mean, float(tm), rel_tol=1e-12)
    # an in-range ignore index; every row ignored gives a NaN mean
    lab2 = np.zeros(12, np.int32)
    loss2, mean2 = oracle_mod.cross_entropy_ignore(d["x"], lab2, 0)
    assert (loss2 == 0).all() and math.isnan(mean2)
    # a label out of range that is not the ignore index is still NaN
    lab3 = d["labels"].copy()
    lab3[0] = 300
    loss3, mean3 = oracle_mod.cross_entropy_ignore(d["x"], lab3, -100)
    assert math.isnan(loss3[0]) and math.isnan(mean3)
