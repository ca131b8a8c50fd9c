"""GPU parity for FP16 / BF16 storage: 16-bit inputs widened to FP32,
FP32 arithmetic, one rounding to the storage type at the store.

The oracle receives the exact FP32 values of the 16-bit inputs.  An output
in 16-bit storage passes when |gpu - ref| <= ulp_T(|ref|(1+2^-6))/2 +
1e-5(1+|ref|): the rounding of the final store plus the FP32 tolerance.
FP32 outputs (row sums, losses, the mean) keep the FP32 tolerance; h_out and
integer row sums are bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import row_reduction_gb300 as mt
from row_reduction_gb300 import inputs
from gpu_util import (Guarded, assert_close, check_softmax_rows,
                      compare_row_blocks, ulp)

pytestmark = pytest.mark.gpu

DTYPES = ["f16", "bf16"]
OPS = list(inputs.ALL_OPS)
SEED = inputs.TUNE_SEED + 100
MATRIX_OUT = {"rmsnorm": ["y"], "layernorm": ["y"], "softmax": ["y"],
              "residual_layernorm": ["y", "h_out"], "row_sum": [],
              "cross_entropy": [], "residual_rmsnorm": ["y", "h_out"],
              "log_softmax": ["y"]}


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_reduction_gb300 import build
    build.build()
    oracle.build()


def assert_close_storage(got, ref, dt, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    with np.errstate(invalid="ignore", over="ignore"):
        tol = (0.5 * ulp(np.abs(ref) * (1 + 2.0 ** -6), dt) +
               1e-5 * (1 + np.abs(ref)))
        err = np.abs(got - ref)
    both_nan = np.isnan(got) & np.isnan(ref)
    # an infinite reference admits only the same infinity
    bad = ~(((err <= tol) & np.isfinite(ref)) | both_nan | (got == ref))
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside; "
                             f"first at {i}: gpu={got[i]!r} ref={ref[i]!r}")


def dev(a, dt):
    """A numpy array in `dt` storage as a CUDA tensor of that type."""
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def to_np(t):
    return t.float().cpu().numpy()


def case(op, rows, cols, dt, seed, **kw):
    d32 = inputs.make(op, rows, cols, seed, **kw)
    st = inputs.as_storage(d32, dt)
    return st, inputs.widen_all(st, dt)


def run(op, st, dt, rows, cols, plan=None, typed=False):
    t = {k: dev(v, dt) for k, v in st.items()
         if isinstance(v, np.ndarray) and k != "labels"}
    if "labels" in st:
        t["labels"] = torch.from_numpy(st["labels"]).cuda()
    eps = st.get("eps", 0.0)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    outs = {}
    if op in ("rmsnorm", "layernorm", "softmax", "residual_layernorm",
              "residual_rmsnorm", "log_softmax"):
        outs["y"] = torch.full((rows, cols), -7.0, dtype=tdt, device="cuda")
    if op in ("residual_layernorm", "residual_rmsnorm"):
        outs["h_out"] = torch.full((rows, cols), -7.0, dtype=tdt,
                                   device="cuda")
    if op == "row_sum":
        outs["out"] = torch.full((rows,), -7.0, device="cuda")
    if op == "cross_entropy":
        outs["loss"] = torch.full((rows,), -7.0, device="cuda")
        outs["mean_loss"] = torch.full((1,), -7.0, device="cuda")
    if typed:
        f = {"rmsnorm": lambda: getattr(mt, f"mt_rmsnorm_{dt}")(
                 t["x"], t.get("weight"), outs["y"], rows, cols, eps),
             "layernorm": lambda: getattr(mt, f"mt_layernorm_{dt}")(
                 t["x"], t.get("gamma"), t.get("beta"), outs["y"], rows,
                 cols, eps),
             "residual_layernorm": lambda: getattr(
                 mt, f"mt_residual_layernorm_{dt}")(
                 t["x"], t["residual"], t.get("gamma"), t.get("beta"),
                 outs["y"], outs["h_out"], rows, cols, eps),
             "softmax": lambda: getattr(mt, f"mt_softmax_{dt}")(
                 t["x"], outs["y"], rows, cols),
             "row_sum": lambda: getattr(mt, f"mt_row_sum_{dt}")(
                 t["x"], outs["out"], rows, cols),
             "cross_entropy": lambda: getattr(mt, f"mt_cross_entropy_{dt}")(
                 t["x"], t["labels"], outs["loss"], outs["mean_loss"], rows,
                 cols),
             "residual_rmsnorm": lambda: getattr(
                 mt, f"mt_residual_rmsnorm_{dt}")(
                 t["x"], t["residual"], t.get("weight"), outs["y"],
                 outs["h_out"], rows, cols, eps),
             "log_softmax": lambda: getattr(mt, f"mt_log_softmax_{dt}")(
                 t["x"], outs["y"], rows, cols)}[op]
        f()
    else:
        mt.mt_row_reduce_with_plan(
            op, dt, t["x"], residual=t.get("residual"),
            weight=t.get("weight", t.get("gamma")), beta=t.get("beta"),
            labels=t.get("labels"), y=outs.get("y"),
            h_out=outs.get("h_out"), out=outs.get("out", outs.get("loss")),
            mean_loss=outs.get("mean_loss"), rows=rows, cols=cols, eps=eps,
            plan=plan)
    torch.cuda.synchronize()
    return outs


def check(op, dt, outs, st, wide, what):
    ref = oracle.run(op, wide)
    for k, r in ref.items():
        if k == "h_out":
            want = (wide["x"] + wide["residual"])
            want = (want.astype(np.float16) if dt == "f16" else
                    inputs.widen(inputs.as_storage({"x": want}, "bf16")["x"],
                                 "bf16"))
            got = to_np(outs["h_out"])
            assert np.array_equal(got.astype(np.float32).view(np.uint32),
                                  want.astype(np.float32).view(np.uint32)), \
                f"{what}: h_out bits"
        elif k in MATRIX_OUT[op]:
            assert_close_storage(to_np(outs[k]), r, dt, f"{what} {k}")
            if op == "softmax":
                check_softmax_rows(to_np(outs[k]), r, f"{what} {k}", dt)
        else:
            got = to_np(outs["loss" if k == "loss" else k])
            assert_close(got.reshape(r.shape), r, f"{what} {k}")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("shape", inputs.FAMILY_SHAPES)
def test_family_shapes_typed_entry_points(dt, op, shape):
    rows, cols = shape
    st, wide = case(op, rows, cols, dt, SEED)
    outs = run(op, st, dt, rows, cols, typed=True)
    check(op, dt, outs, st, wide, f"{op} {dt} {shape}")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", inputs.RMSNORM_SWEEP)
def test_rmsnorm_sweep_shapes(dt, shape):
    """Every full-size sweep shape (1% outliers) with the default plan,
    compared with the oracle on every element."""
    rows, cols = shape
    st, wide = case("rmsnorm", rows, cols, dt, SEED + 1, outliers=True)
    outs = run("rmsnorm", st, dt, rows, cols)
    got = to_np(outs["y"])
    del outs
    compare_row_blocks(
        got, lambda lo, hi: oracle.rmsnorm(wide["x"][lo:hi], wide["weight"],
                                           wide["eps"]),
        lambda g, r, w: assert_close_storage(g, r, dt, w),
        f"rmsnorm {dt} {shape}")


def half_plans(cols):
    plans = []
    for V in (2, 4, 8):
        for W in (2, 4, 8, 32, 64, 256, 1024):
            if W < V:
                continue
            for B in {max(1, 32 // W), max(1, 256 // W)}:
                for K in (1, 2, 4, 8, 16):
                    if W * V * K >= cols:
                        plans.append(mt.make_plan(W, V, K, B))
                        break
                if W <= 512:
                    plans.append(mt.make_plan(W, V, 0, B, mt.MT_PATH_LOOP))
    return [p for p in plans
            if mt.mt_plan_check_dtype(0, "bf16", cols, p) == mt.MT_OK]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("cols", [1, 31, 33, 127, 128, 129, 257, 4103])
def test_mapping_matrix(dt, op, cols):
    rows = 5
    st, wide = case(op, rows, cols, dt, SEED + cols)
    for p in half_plans(cols):
        outs = run(op, st, dt, rows, cols, plan=p)
        check(op, dt, outs, st, wide,
              f"{op} {dt} {rows}x{cols} {mt.mt_describe_plan(p)}")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("cols", [127, 4096, 4103])
@pytest.mark.parametrize("xoff,yoff", [(1, 1), (3, 0), (5, 2), (0, 7)])
def test_unaligned_bases_with_guards(dt, op, cols, xoff, yoff):
    """Bases shifted by 1-7 elements (rows start off the 16-byte grid) with
    NaN guards around inputs and sentinel guards around outputs."""
    rows = 6
    st, wide = case(op, rows, cols, dt, SEED + 7 * xoff + cols)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    bufs = {}
    offs = {"x": xoff, "residual": (xoff + 3) % 8, "weight": 1, "gamma": 5,
            "beta": 2, "y": yoff, "h_out": (yoff + 1) % 8}
    for k, v in st.items():
        if not isinstance(v, np.ndarray):
            continue
        if k == "labels":
            bufs[k] = Guarded(v.size, 1, -7, torch.int32, v)
        else:
            g = Guarded(v.size, offs.get(k, 0), float("nan"), tdt)
            g.view.copy_(dev(v, dt).reshape(-1))
            bufs[k] = g
    if MATRIX_OUT[op]:
        for k in MATRIX_OUT[op]:
            bufs[k] = Guarded(rows * cols, offs[k], -1.0, tdt)
    if op == "row_sum":
        bufs["out"] = Guarded(rows, 0, -1.0)
    if op == "cross_entropy":
        bufs["out"] = Guarded(rows, 0, -1.0)
        bufs["mean_loss"] = Guarded(1, 0, -1.0)
    P = {k: b.ptr for k, b in bufs.items()}
    for plan in (None, mt.make_plan(32, 8, 16, 1),
                 mt.make_plan(64, 2, 0, 1, mt.MT_PATH_LOOP)):
        if plan is not None and mt.mt_plan_check_dtype(
                op, dt, cols, plan) != mt.MT_OK:
            continue
        mt.mt_row_reduce_with_plan(
            op, dt, P["x"], residual=P.get("residual"),
            weight=P.get("weight", P.get("gamma")), beta=P.get("beta"),
            labels=P.get("labels"), y=P.get("y"), h_out=P.get("h_out"),
            out=P.get("out"), mean_loss=P.get("mean_loss"), rows=rows,
            cols=cols, eps=st.get("eps", 0.0), plan=plan)
        torch.cuda.synchronize()
        for b in bufs.values():
            b.check()
        outs = {k: (bufs[k].view.reshape(rows, cols) if k in ("y", "h_out")
                    else bufs[k].view) for k in bufs
                if k in ("y", "h_out", "out", "mean_loss")}
        if "out" in outs and op == "cross_entropy":
            outs["loss"] = outs.pop("out")
        check(op, dt, outs, st, wide, f"{op} {dt} x+{xoff} y+{yoff} {plan}")


@pytest.mark.parametrize("dt", DTYPES)
def test_row_sum_of_small_integers_is_exact(dt):
    x = inputs.integer_valued(64, 4103, SEED)
    st = inputs.as_storage({"x": x}, dt)
    xt = dev(st["x"], dt)
    got = mt.row_sum(xt).cpu().numpy()
    assert np.array_equal(got, x.astype(np.int64).sum(axis=1).astype(
        np.float32))


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("op", ["rmsnorm", "layernorm", "softmax"])
def test_in_place_and_determinism(dt, op):
    rows, cols = 256, 4096
    st, _ = case(op, rows, cols, dt, SEED + 3)
    x = dev(st["x"], dt)
    kw = {}
    if op == "rmsnorm":
        kw = dict(weight=dev(st["weight"], dt), eps=st["eps"])
        f = mt.rmsnorm
    elif op == "layernorm":
        kw = dict(gamma=dev(st["gamma"], dt), beta=dev(st["beta"], dt),
                  eps=st["eps"])
        f = mt.layernorm
    else:
        f = mt.softmax
    a = f(x, **kw)
    b = f(x, **kw)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    f(x, out=x, **kw)
    assert torch.equal(x.view(torch.int16), a.view(torch.int16))


@pytest.mark.parametrize("dt", DTYPES)
def test_cross_entropy_ignore_index_half(dt):
    rows, cols = 512, 1000
    st, wide = case("cross_entropy", rows, cols, dt, SEED + 9)
    lab = st["labels"].copy()
    lab[1::4] = -100
    x = dev(st["x"], dt)
    loss = torch.empty(rows, device="cuda")
    mean = torch.empty(1, device="cuda")
    getattr(mt, f"mt_cross_entropy_ignore_{dt}")(
        x, torch.from_numpy(lab).cuda(), -100, loss, mean, rows, cols)
    ref_loss, ref_mean = oracle.cross_entropy_ignore(wide["x"], lab, -100)
    assert_close(loss.cpu().numpy(), ref_loss, "loss")
    assert_close(mean.cpu().numpy(), np.array([ref_mean]), "mean")


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("op", ["rmsnorm", "layernorm", "softmax",
                                "log_softmax", "cross_entropy", "row_sum"])
def test_staged_rows_half(dt, op):
    """16-bit rows staged in shared memory (single CTAs, clusters, several
    bulk copies per run), against the oracle."""
    for rows, cols in ((3, 32768), (2, 131072), (5, 40008)):
        st, wide = case(op, rows, cols, dt, SEED + 41 + cols)
        for W, C, pieces in ((256, 1, 4), (512, 2, 2), (128, 4, 8),
                             (1024, 8, 1), (256, 16, 4)):
            p = mt.make_plan(W, 8, pieces, 1, mt.MT_PATH_STAGE,
                             cluster=C if C > 1 else 0,
                             flags=mt.MT_PLAN_PDL)
            if mt.mt_plan_check_dtype(op, dt, cols, p) != mt.MT_OK:
                continue
            outs = run(op, st, dt, rows, cols, plan=p)
            check(op, dt, outs, st, wide,
                  f"{op} {dt} {rows}x{cols} {mt.mt_describe_plan(p)}")
    assert mt.mt_stage_wait_timeouts() == 0


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("op", OPS)
def test_cluster_split_rows_half(dt, op):
    rows, cols = 3, 50003
    st, wide = case(op, rows, cols, dt, SEED + 31)
    for p in (mt.make_plan(512, 8, 4, 1, cluster=4),
              mt.make_plan(256, 8, 0, 1, mt.MT_PATH_LOOP, cluster=8),
              mt.make_plan(128, 8, 4, 1, cluster=16),
              mt.make_plan(512, 8, 0, 1, mt.MT_PATH_LOOP, cluster=16)):
        assert mt.mt_plan_check_dtype(op, dt, cols, p) == mt.MT_OK
        outs = run(op, st, dt, rows, cols, plan=p)
        check(op, dt, outs, st, wide, f"{op} {dt} {mt.mt_describe_plan(p)}")
