"""The GPU tests' checkers, on the CPU: each accepts a correct result and
rejects a planted error of the kind it exists to catch."""
import numpy as np
import pytest

from gpu_util import assert_close, check_softmax_rows, compare_row_blocks


def softmax64(x):
    e = np.exp(x - x.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def rows():
    rng = np.random.default_rng(3)
    return softmax64(2.0 * rng.standard_normal((8, 32000)))


def test_softmax_checks_accept_float32_rounding():
    ref = rows()
    check_softmax_rows(ref.astype(np.float32), ref, "fp32 rounding")


def test_softmax_checks_catch_small_probabilities_off_by_a_percent():
    ref = rows()
    got = ref.astype(np.float32).astype(np.float64)
    # ten outputs 1% high: each error is below the absolute floor of the
    # element-wise tolerance, and together they move the row's sum by less
    # than 1e-5, so only the relative check sees them
    got[3, 1000:1010] *= 1.01
    assert_close(got, ref, "element-wise floor hides it")
    with pytest.raises(AssertionError, match="relative terms"):
        check_softmax_rows(got, ref, "planted")


def test_softmax_checks_catch_a_row_not_summing_to_one():
    ref = rows()
    got = ref * (1 + 3e-5)
    with pytest.raises(AssertionError, match="sum to 1"):
        check_softmax_rows(got, ref, "planted")


def test_softmax_checks_16_bit_bounds():
    import torch
    ref = rows()
    bf = torch.from_numpy(ref).float().bfloat16().float().double().numpy()
    check_softmax_rows(bf, ref, "bf16 rounding", dt="bf16")
    off = bf.copy()
    off[2, 10:20] *= 1.02          # a 2% error is several BF16 ulps
    with pytest.raises(AssertionError):
        check_softmax_rows(off, ref, "planted", dt="bf16")


def test_log_softmax_sum_check():
    ref = np.log(rows())
    check_softmax_rows(ref.astype(np.float32), ref, "log", log=True)
    with pytest.raises(AssertionError):
        check_softmax_rows(ref + 3e-5, ref, "planted", log=True)


def test_row_blocks_cover_every_row_and_report_the_block():
    ref = rows()
    seen = []

    def check(g, r, what):
        seen.append(len(g))
        assert_close(g, r, what)
    compare_row_blocks(ref.copy(), lambda lo, hi: ref[lo:hi], check, "all",
                       block=3)
    assert sum(seen) == len(ref)
    bad = ref.copy()
    bad[7, 5] += 1e-3
    with pytest.raises(AssertionError, match="rows 6..7"):
        compare_row_blocks(bad, lambda lo, hi: ref[lo:hi], assert_close,
                           "planted", block=3)


def test_element_check_handles_infinities():
    assert_close(np.array([-np.inf, np.inf, 1.0]),
                 np.array([-np.inf, np.inf, 1.0]), "equal infinities")
    for got in ([np.inf], [5.0], [np.nan]):
        with pytest.raises(AssertionError):
            assert_close(np.array(got), np.array([-np.inf]), "planted")
    with pytest.raises(AssertionError):
        assert_close(np.array([-np.inf]), np.array([3.0]), "planted")
