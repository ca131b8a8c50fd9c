"""GPU parity: the CUDA library against the CPU oracle, element by element,
through the C ABI, on the published shapes and the edge cases of the work
mapping.  Tolerance |gpu - ref| <= 1e-5*(1+|ref|); bit-exact where the result
is exactly representable (integer row sums, the residual sum h_out).

The lane-mapping matrix follows the test the pages describe ("Consecutive-
worker reduction layout checkpoint", §Verification checkpoint: V = 2/4/8
across N = 1/31/33/127/128/129/257/4103, five rows, packed short rows and
eight-subgroup wide rows), widened to every operator and to V = 1/2/4, W from
1 to 1024 and rows-per-block packing.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import row_reduction_gb300 as mt
from row_reduction_gb300 import inputs
from gpu_util import (Guarded, assert_close, check_softmax_rows,
                      compare_row_blocks, to_dev)

pytestmark = pytest.mark.gpu

OPS = list(inputs.ALL_OPS)
SEED = inputs.TUNE_SEED


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_reduction_gb300 import build
    build.build()
    oracle.build()


# ---------------------------------------------------------------- helpers
def call(op, p, rows, cols, eps=None, plan=None, stream=None):
    """Calls the *_with_plan C entry point of `op` with device addresses."""
    if op == "rmsnorm":
        mt.mt_rmsnorm_f32_with_plan(p["x"], p.get("weight"), p["y"], rows,
                                    cols, eps, stream, plan)
    elif op == "layernorm":
        mt.mt_layernorm_f32_with_plan(p["x"], p.get("gamma"), p.get("beta"),
                                      p["y"], rows, cols, eps, stream, plan)
    elif op == "residual_layernorm":
        mt.mt_residual_layernorm_f32_with_plan(
            p["x"], p["residual"], p.get("gamma"), p.get("beta"), p["y"],
            p.get("h_out"), rows, cols, eps, stream, plan)
    elif op == "softmax":
        mt.mt_softmax_f32_with_plan(p["x"], p["y"], rows, cols, stream, plan)
    elif op == "row_sum":
        mt.mt_row_sum_f32_with_plan(p["x"], p["out"], rows, cols, stream,
                                    plan)
    elif op == "cross_entropy":
        mt.mt_cross_entropy_f32_with_plan(p["x"], p["labels"], p["loss"],
                                          p.get("mean_loss"), rows, cols,
                                          stream, plan)
    elif op == "residual_rmsnorm":
        mt.mt_residual_rmsnorm_f32_with_plan(p["x"], p["residual"],
                                             p.get("weight"), p["y"],
                                             p.get("h_out"), rows, cols, eps,
                                             stream, plan)
    elif op == "log_softmax":
        mt.mt_log_softmax_f32_with_plan(p["x"], p["y"], rows, cols, stream,
                                        plan)
    else:
        raise ValueError(op)


def outputs_of(op, rows, cols):
    if op in ("rmsnorm", "layernorm", "softmax", "log_softmax"):
        return {"y": rows * cols}
    if op in ("residual_layernorm", "residual_rmsnorm"):
        return {"y": rows * cols, "h_out": rows * cols}
    if op == "row_sum":
        return {"out": rows}
    return {"loss": rows, "mean_loss": 1}


def run_guarded(op, d, rows, cols, plan=None, offsets=None):
    """Runs `op` on guarded copies of the inputs in `d`; returns numpy
    outputs after checking every guard region."""
    offsets = offsets or {}
    bufs = {}
    for k, v in d.items():
        if isinstance(v, np.ndarray):
            fill = float("nan") if v.dtype == np.float32 else -7
            dt = torch.float32 if v.dtype == np.float32 else torch.int32
            bufs[k] = Guarded(v.size, offsets.get(k, 0), fill, dt, v)
    for k, n in outputs_of(op, rows, cols).items():
        bufs[k] = Guarded(n, offsets.get(k, 0), Guarded.SENTINEL)
    call(op, {k: b.ptr for k, b in bufs.items()}, rows, cols, d.get("eps"),
         plan)
    torch.cuda.synchronize()
    for b in bufs.values():
        b.check()
    res = {}
    for k in outputs_of(op, rows, cols):
        a = bufs[k].numpy()
        res[k] = a.reshape(rows, cols) if a.size == rows * cols and \
            k in ("y", "h_out") else a
    return res


def compare(op, got, ref, what):
    for k, r in ref.items():
        if k == "h_out":
            assert np.array_equal(got[k].view(np.uint32),
                                  r.view(np.uint32)), f"{what}: h_out bits"
        else:
            assert_close(got[k], r, f"{what} {k}")
            if op in ("softmax", "log_softmax"):
                check_softmax_rows(got[k], r, f"{what} {k}",
                                   log=op == "log_softmax")


# --------------------------------------------------- published shapes
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("shape", inputs.FAMILY_SHAPES)
def test_family_shapes_default_plan(op, shape):
    rows, cols = shape
    d = inputs.make(op, rows, cols, SEED)
    got = run_guarded(op, d, rows, cols)
    compare(op, got, oracle.run(op, d), f"{op} {shape}")


@pytest.mark.parametrize("shape", inputs.RMSNORM_SHAPES)
def test_rmsnorm_published_small_shapes(shape):
    d = inputs.make("rmsnorm", *shape, seed=SEED + 1)
    got = run_guarded("rmsnorm", d, *shape)
    compare("rmsnorm", got, oracle.run("rmsnorm", d), f"rmsnorm {shape}")


@pytest.mark.parametrize("shape", inputs.RMSNORM_SWEEP)
def test_rmsnorm_sweep_full_size(shape):
    """Full-size sweep shapes (1% outliers) with the default plan: every
    element against the oracle, and on every row the unit-weight invariant
    mean((y/w)^2) = ms/(ms+eps) recomputed in float64."""
    rows, cols = shape
    d = inputs.make("rmsnorm", rows, cols, SEED + 2, outliers=True)
    t = to_dev(d)
    y = mt.rmsnorm(t["x"], t["weight"], d["eps"])
    torch.cuda.synchronize()
    compare_row_blocks(
        y.cpu().numpy(),
        lambda lo, hi: oracle.rmsnorm(d["x"][lo:hi], d["weight"], d["eps"]),
        assert_close, f"rmsnorm {shape}")
    xd = t["x"].double()
    ms = (xd * xd).mean(dim=1)
    eps = float(np.float32(d["eps"]))
    u = (y.double() / t["weight"].double())
    lhs = (u * u).mean(dim=1)
    rhs = ms / (ms + eps)
    assert torch.allclose(lhs, rhs, rtol=2e-5, atol=0)


@pytest.mark.parametrize("op", ["rmsnorm", "row_sum", "softmax"])
def test_more_than_2_31_elements(op):
    """A matrix of 524291 x 4096 = 2^31 + 12288 elements (8.6 GB of FP32):
    element offsets need 64 bits.  The rows repeat a 64-row block made by
    the input generator, so the oracle's 64 rows give every expected row;
    sampled rows, the last ones past element 2^31 included, are checked."""
    rows, cols, blk = (1 << 19) + 3, 4096, 64
    assert rows * cols > 2 ** 31
    d = inputs.make(op, blk, cols, SEED + 31)
    ref = oracle.run(op, d)
    x = torch.from_numpy(d["x"]).cuda().repeat((rows + blk - 1) // blk, 1)
    x = x[:rows]
    if op == "rmsnorm":
        out = mt.rmsnorm(x, torch.from_numpy(d["weight"]).cuda(), d["eps"])
        want = ref["y"]
    elif op == "row_sum":
        out = mt.row_sum(x)
        want = ref["out"]
    else:
        out = mt.softmax(x)
        want = ref["y"]
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    sample = np.unique(np.concatenate(
        [[0, blk - 1, rows // 2, rows - 2, rows - 1],
         rng.integers(0, rows, 24)]))
    got = out[torch.from_numpy(sample).cuda()].cpu().numpy()
    assert_close(got, want[sample % blk], f"{op} {rows}x{cols} sampled rows")
    del x, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16,
                                   torch.float16])
def test_signed_zeros_keep_their_sign(dtype):
    """RMSNorm scales x by a positive factor (weights > 0), so -0.0 and
    +0.0 come out with their own sign; bit-checked."""
    rows, cols = 33, 4096
    g = torch.Generator().manual_seed(5)
    x = torch.randn(rows, cols, generator=g)
    x[:, ::7] = 0.0
    x[:, 3::7] = -0.0
    w = 1.0 + 0.1 * torch.rand(cols, generator=g)
    xd, wd = x.to(dtype).cuda(), w.to(dtype).cuda()
    y = mt.rmsnorm(xd, wd, 1e-6).cpu()
    neg = torch.signbit(x.to(dtype)) & (x == 0)
    pos = ~torch.signbit(x.to(dtype)) & (x == 0)
    assert bool((y[neg] == 0).all()) and bool(torch.signbit(y[neg]).all())
    assert bool((y[pos] == 0).all()) and not bool(torch.signbit(y[pos]).any())


# ------------------------------------------------ lane-mapping matrix
MAP_N = [1, 31, 33, 127, 128, 129, 257, 4103]


def candidate_plans(cols):
    plans = []
    for V in (1, 2, 4):
        for W in (1, 2, 4, 8, 32, 64, 256, 1024):
            for packed in (False, True):
                B = max(1, 32 // W) if not packed else max(1, 256 // W)
                # register path: smallest instantiated chunk count
                for K in (1, 2, 4, 8, 16):
                    if W * V * K >= cols:
                        plans.append(mt.make_plan(W, V, K, B))
                        break
                if W <= 512:
                    plans.append(mt.make_plan(W, V, 0, B, mt.MT_PATH_LOOP))
    out, seen = [], set()
    for p in plans:
        key = tuple(p.as_dict().values())
        if key not in seen and mt.mt_plan_check(0, cols, p) == mt.MT_OK:
            seen.add(key)
            out.append(p)
    return out


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("cols", MAP_N)
def test_mapping_matrix(op, cols):
    for rows in (5, 17):
        d = inputs.make(op, rows, cols, SEED + cols + rows)
        ref = oracle.run(op, d)
        t = to_dev(d)
        plans = candidate_plans(cols)
        assert plans
        for p in plans:
            outs = {k: torch.full((n,), Guarded.SENTINEL, device="cuda")
                    for k, n in outputs_of(op, rows, cols).items()}
            ptrs = {k: v.data_ptr() for k, v in t.items()
                    if isinstance(v, torch.Tensor)}
            ptrs.update({k: v.data_ptr() for k, v in outs.items()})
            call(op, ptrs, rows, cols, d.get("eps"), p)
            got = {k: (v.cpu().numpy().reshape(rows, cols)
                       if k in ("y", "h_out") else v.cpu().numpy())
                   for k, v in outs.items()}
            compare(op, got, ref, f"{op} {rows}x{cols} "
                    f"{mt.mt_describe_plan(p)}")


# ------------------------------------------------ whole-tile kernels
# Plans with the whole-tile flag whose packs tile every row exactly
# (cols = W*V*K) run, when rows is a multiple of B and every parameter
# vector is present, the unguarded whole-tile kernels; one more row (no
# longer a multiple of B) sends the same plan to the guarded kernel.
# (cols, W, V, K, B):
WHOLE_TILES = [(128, 32, 4, 1, 4), (512, 128, 1, 4, 2), (1024, 64, 4, 4, 2),
               (2048, 256, 2, 4, 2), (4096, 128, 4, 8, 2),
               (4096, 256, 4, 4, 2), (4096, 64, 4, 16, 2),
               (8192, 512, 4, 4, 2)]


def _first_rows(d, n):
    return {k: (v[:n] if isinstance(v, np.ndarray) and k in
                ("x", "residual", "labels") else v) for k, v in d.items()}


@pytest.mark.parametrize("op", OPS)
def test_whole_tile_kernels(op):
    """The whole-tile kernels agree with the oracle, and bit for bit with
    the guarded kernel of the same plan on the same rows."""
    rows = 6
    for cols, W, V, K, B in WHOLE_TILES:
        p = mt.make_plan(W, V, K, B, flags=mt.MT_PLAN_PDL |
                         mt.MT_PLAN_WHOLE_TILES)
        assert mt.mt_plan_check(mt.OP_IDS[op], cols, p) == mt.MT_OK
        d = inputs.make(op, rows + 1, cols, SEED + 7 * cols + W)
        d6 = _first_rows(d, rows)
        what = f"{op} {rows}x{cols} {mt.mt_describe_plan(p)}"
        full = run_guarded(op, d6, rows, cols, plan=p)
        compare(op, full, oracle.run(op, d6), what + " (whole tiles)")
        guarded = run_guarded(op, d, rows + 1, cols, plan=p)
        for k in full:
            if k == "mean_loss":
                continue
            a, b = full[k], guarded[k][:rows]
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), \
                f"{what}: {k} differs from the guarded kernel"


# --------------------------------------- alignment heads and guards
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("cols", [3, 127, 257, 4096, 4103])
@pytest.mark.parametrize("xoff,yoff", [(1, 1), (2, 0), (3, 1), (0, 2)])
def test_unaligned_bases(op, cols, xoff, yoff):
    """Base pointers shifted by 1-3 floats: rows start off the 16-byte grid
    (heads are peeled) and outputs may be out of phase with x (scalar
    stores).  Guards are NaN on inputs and a sentinel on outputs."""
    rows = 9
    d = inputs.make(op, rows, cols, SEED + 3 * cols + xoff)
    offs = {"x": xoff, "y": yoff, "h_out": (yoff + 1) % 4,
            "residual": (xoff + 2) % 4, "weight": 1, "gamma": 3, "beta": 2,
            "out": yoff, "loss": 1, "labels": 1}
    ref = oracle.run(op, d)
    got = run_guarded(op, d, rows, cols, offsets=offs)
    compare(op, got, ref, f"{op} x+{xoff} y+{yoff} cols={cols}")
    for V in (2, 4):
        for W in (4, 32, 128):
            p = mt.make_plan(W, V, 16, max(1, 32 // W))
            if cols > W * V * 16:
                continue
            got = run_guarded(op, d, rows, cols, plan=p, offsets=offs)
            compare(op, got, ref, f"{op} forced {mt.mt_describe_plan(p)}")
            p = mt.make_plan(W, V, 0, max(1, 32 // W), mt.MT_PATH_LOOP)
            got = run_guarded(op, d, rows, cols, plan=p, offsets=offs)
            compare(op, got, ref, f"{op} forced {mt.mt_describe_plan(p)}")


# ------------------------------------------------------ wide rows
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("cols", [16384, 32771, 100003])
def test_wide_rows(op, cols):
    rows = 3
    d = inputs.make(op, rows, cols, SEED + cols)
    got = run_guarded(op, d, rows, cols)
    compare(op, got, oracle.run(op, d), f"{op} {rows}x{cols}")


# --------------------------------------------------- exact results
def test_row_sum_of_integers_is_bit_exact():
    for rows, cols in ((17, 257), (64, 4096), (3, 100003), (1024, 4096)):
        x = inputs.integer_valued(rows, cols, SEED)
        ref = x.astype(np.int64).sum(axis=1).astype(np.float32)
        xt = torch.from_numpy(x).cuda()
        for p in [None] + candidate_plans(cols)[:12]:
            if p is not None and cols > 4103:
                break
            got = mt.row_sum(xt, plan=p).cpu().numpy()
            assert np.array_equal(got, ref), (rows, cols, p)


def test_row_sum_near_zero_rows():
    """Rows whose sum cancels to near zero keep the 1e-5*(1+|ref|)
    tolerance (compensated accumulation)."""
    rows, cols = 64, 4096
    d = inputs.make("row_sum", rows, cols, SEED)
    x = d["x"].copy()
    x[:, cols // 2:] = -x[:, :cols // 2][:, ::-1]   # exact cancellation
    x[:, 0] += np.float32(1e-3)
    ref = oracle.row_sum(x)
    got = mt.row_sum(torch.from_numpy(x).cuda()).cpu().numpy()
    assert_close(got, ref, "near-zero sums")


def test_row_sum_cancelling_pairs():
    """Rows of large values whose exact negatives sit elsewhere in the row
    (magnitudes up to ~4e4), plus a residue of 1e-3: the exact sum is the
    residue, far below the rounding error of a plain FP32 sum of the row.
    Every plan family (register path, loop path, whole tiles) must keep the
    1e-5*(1+|ref|) tolerance."""
    rng = np.random.default_rng(SEED + 99)
    for rows, cols in ((32, 4096), (16, 4098), (4, 100003)):
        x = np.zeros((rows, cols), np.float32)
        for r in range(rows):
            half = (cols - 1) // 2
            big = (rng.standard_normal(half) * 1e4).astype(np.float32)
            perm = rng.permutation(cols)
            x[r, perm[:half]] = big
            x[r, perm[half:2 * half]] = -big
            x[r, perm[-1]] = np.float32(1e-3) * (r + 1)
        ref = oracle.row_sum(x)
        xt = torch.from_numpy(x).cuda()
        plans = [None]
        if cols == 4096:
            plans += [mt.make_plan(128, 4, 8, 1), mt.make_plan(64, 4, 16, 2),
                      mt.make_plan(256, 2, 8, 1), mt.make_plan(1024, 4, 1, 1),
                      mt.make_plan(128, 4, 0, 2, mt.MT_PATH_LOOP)]
        for p in plans:
            got = mt.row_sum(xt, plan=p).cpu().numpy()
            assert_close(got, ref, f"cancelling pairs {rows}x{cols} "
                         f"{mt.mt_describe_plan(p) if p else 'default'}")


def test_residual_h_out_bit_exact_and_aliasing():
    rows, cols = 33, 1000
    d = inputs.make("residual_layernorm", rows, cols, SEED)
    t = to_dev(d)
    y, h = mt.residual_layernorm(t["x"], t["residual"], t["gamma"],
                                 t["beta"], d["eps"], return_h=True)
    assert torch.equal(h, t["x"] + t["residual"])
    ref_y, _ = oracle.residual_layernorm(d["x"], d["residual"], d["gamma"],
                                         d["beta"], d["eps"])
    assert_close(y.cpu().numpy(), ref_y, "resln")
    # y written over x and h over the residual
    x2, r2 = t["x"].clone(), t["residual"].clone()
    mt.mt_residual_layernorm_f32(x2, r2, t["gamma"], t["beta"], x2, r2, rows,
                                 cols, d["eps"])
    assert torch.equal(x2, y) and torch.equal(r2, h)


@pytest.mark.parametrize("op", ["rmsnorm", "layernorm", "softmax"])
def test_in_place(op):
    for rows, cols in ((17, 257), (64, 4096), (2, 40000)):
        d = inputs.make(op, rows, cols, SEED)
        t = to_dev(d)
        ref = mt.run(op, t)["y"]
        x = t["x"]
        if op == "rmsnorm":
            mt.mt_rmsnorm_f32(x, t["weight"], x, rows, cols, d["eps"])
        elif op == "layernorm":
            mt.mt_layernorm_f32(x, t["gamma"], t["beta"], x, rows, cols,
                                d["eps"])
        else:
            mt.mt_softmax_f32(x, x, rows, cols)
        assert torch.equal(x, ref)


@pytest.mark.parametrize("op", ["layernorm", "residual_layernorm"])
def test_layernorm_ill_conditioned_rows(op):
    """Rows fifty standard deviations away from zero (mean 50, std 1) with
    1% outliers of +-5: a one-pass E[x^2] - E[x]^2 in FP32 misses y by about
    five times the tolerance here; the two-pass statistics (the mean removed
    before the squares are summed) stay within about a third of it.  (Rows
    much further off centre, say mean 1e3 and std 1e-2, are beyond FP32
    itself: the FP32 inputs quantise the deviations to 0.6% of the spread,
    and no FP32 y can match the double oracle to 1e-5.)  Every plan family:
    default, register (guarded and whole tiles), loop, cluster and
    staged."""
    rng = np.random.default_rng(SEED + 1234)
    for rows, cols in ((16, 4096), (6, 40000)):
        x = (50.0 + rng.standard_normal((rows, cols))).astype(np.float32)
        mask = rng.random((rows, cols)) < 0.01
        x[mask] += np.where(rng.random(mask.sum()) < 0.5, -5.0,
                            5.0).astype(np.float32)
        d = inputs.make(op, rows, cols, SEED + cols)
        d["x"] = x
        if op == "residual_layernorm":
            d["residual"] = rng.standard_normal((rows, cols)).astype(
                np.float32) * np.float32(0.1)
        ref = oracle.run(op, d)
        plans = [None]
        if cols == 4096:
            plans += [mt.make_plan(256, 4, 4, 1),
                      mt.make_plan(256, 4, 4, 2, flags=mt.MT_PLAN_PDL |
                                   mt.MT_PLAN_WHOLE_TILES),
                      mt.make_plan(128, 4, 0, 2, mt.MT_PATH_LOOP),
                      mt.make_plan(128, 4, 4, 1, cluster=2)]
        else:
            plans += [mt.make_plan(256, 4, 0, 1, mt.MT_PATH_LOOP),
                      mt.make_plan(256, 4, 16, 1, cluster=4)]
            if op == "layernorm":
                plans += [mt.make_plan(512, 4, 2, 1, mt.MT_PATH_STAGE)]
        for p in plans:
            if p is not None:
                assert mt.mt_plan_check(mt.OP_IDS[op], cols, p) == mt.MT_OK
            got = run_guarded(op, d, rows, cols, plan=p)
            compare(op, got, ref, f"{op} ill-conditioned {rows}x{cols} " + (
                "default" if p is None else mt.mt_describe_plan(p)))


def test_softmax_special_rows():
    x = np.array([[1.0, np.nan, 2.0, 3.0], [1000.0, 1000.0, -1000.0, 0.0],
                  [5.0, 5.0, 5.0, 5.0], [-np.inf, 0.0, 0.0, -np.inf]],
                 dtype=np.float32)
    ref = oracle.softmax(x)
    got = mt.softmax(torch.from_numpy(x).cuda()).cpu().numpy()
    assert_close(got, ref, "softmax special rows")
    check_softmax_rows(got, ref, "softmax special rows")


def test_cross_entropy_labels_and_mean():
    rows, cols = 64, 4096
    d = inputs.make("cross_entropy", rows, cols, SEED)
    d["labels"][3] = cols        # out of range -> NaN row
    d["labels"][7] = -1
    t = to_dev(d)
    loss, m = mt.cross_entropy(t["x"], t["labels"])
    ref_loss, ref_mean = oracle.cross_entropy(d["x"], d["labels"])
    assert_close(loss.cpu().numpy(), ref_loss, "loss")
    assert math.isnan(float(m)) and math.isnan(ref_mean)
    d["labels"][3], d["labels"][7] = 0, cols - 1
    t = to_dev(d)
    loss, m = mt.cross_entropy(t["x"], t["labels"])
    ref_loss, ref_mean = oracle.cross_entropy(d["x"], d["labels"])
    assert_close(loss.cpu().numpy(), ref_loss, "loss")
    assert_close(m.cpu().numpy(), np.array([ref_mean]), "mean")
    # Mean over many rows (the mean kernel's strided loop).
    d = inputs.make("cross_entropy", 70000, 33, SEED)
    t = to_dev(d)
    loss, m = mt.cross_entropy(t["x"], t["labels"])
    ref_loss, ref_mean = oracle.cross_entropy(d["x"], d["labels"])
    assert_close(m.cpu().numpy(), np.array([ref_mean]), "mean 70000 rows")


@pytest.mark.parametrize("op", OPS)
def test_determinism(op):
    rows, cols = 1024, 4096
    d = inputs.make(op, rows, cols, SEED)
    t = to_dev(d)
    a = mt.run(op, t)
    b = mt.run(op, t)
    for k in a:
        assert torch.equal(a[k].view(torch.int32), b[k].view(torch.int32))


def test_non_default_stream_and_zero_rows():
    d = inputs.make("rmsnorm", 64, 4096, SEED)
    t = to_dev(d)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        y = mt.rmsnorm(t["x"], t["weight"], d["eps"], stream=s)
    s.synchronize()
    assert_close(y.cpu().numpy(), oracle.rmsnorm(d["x"], d["weight"],
                                                 d["eps"]), "stream")
    e = torch.empty(0, 4096, device="cuda")
    assert mt.rmsnorm(e, t["weight"]).shape == (0, 4096)


def test_forced_plan_errors_on_gpu():
    x = torch.zeros(4, 4096, device="cuda")
    with pytest.raises(mt.MTError) as ei:
        mt.rmsnorm(x, plan=mt.make_plan(256, 4, 2, 1))
    assert ei.value.status == mt.MT_ERR_OUT_OF_RESOURCES
    with pytest.raises(mt.MTError) as ei:
        mt.rmsnorm(x, plan=mt.make_plan(96, 4, 16, 1))
    assert ei.value.status == mt.MT_ERR_INVALID_ARGUMENT
    # explicit grids, including one smaller than the row-group count
    for g in (1, 3, 1000):
        y = mt.rmsnorm(x + 1, plan=mt.make_plan(256, 4, 4, 1, grid=g))
        assert torch.allclose(y, torch.ones_like(y), rtol=1e-5)


# ------------------------------- persistent grids with L2 prefetches
PDL_NEXT = mt.MT_PLAN_PDL | mt.MT_PLAN_PREFETCH_NEXT


@pytest.mark.parametrize("op", OPS)
def test_persistent_grids_with_prefetch(op):
    """Grids smaller than the row-group count (CTAs loop over row groups),
    with the first row group prefetched into L2 before the wait on the
    previous kernel and the next one prefetched during the current one,
    against the oracle, with guards; the second shape is unaligned and
    ragged."""
    for rows, cols, K, offs in ((1000, 4096, 8, {}),
                                (517, 1000, 2, {"x": 1, "y": 1, "h_out": 1,
                                                "residual": 1})):
        d = inputs.make(op, rows, cols, SEED + rows)
        ref = oracle.run(op, d)
        for grid in (7, 152, 304):
            for fl in (mt.MT_PLAN_PDL, PDL_NEXT):
                p = mt.make_plan(128, 4, K, 2, grid=grid, flags=fl)
                got = run_guarded(op, d, rows, cols, plan=p, offsets=offs)
                compare(op, got, ref,
                        f"{op} {rows}x{cols} {mt.mt_describe_plan(p)}")


def test_prefetched_call_reads_the_previous_kernels_output():
    """A call whose input the previous call on the stream writes: the L2
    prefetch issued before the wait must not let it read the old contents
    (here NaN)."""
    rows, cols = 4096, 4096
    x = torch.randn(rows, cols, device="cuda")
    w = torch.ones(cols, device="cuda")
    z = torch.empty_like(x)
    s = torch.empty(rows, device="cuda")
    pa = mt.make_plan(128, 4, 8, 2, grid=152, flags=PDL_NEXT)
    for _ in range(3):
        z.fill_(float("nan"))
        mt.softmax(x, out=z, plan=pa)
        mt.row_sum(z, out=s, plan=pa)
        mt.rmsnorm(z, w, eps=0.0, out=z, plan=pa)
        torch.cuda.synchronize()
        assert torch.allclose(s, torch.ones_like(s), atol=1e-5)
        assert bool(torch.isfinite(z).all())
        ms = (z.double() ** 2).mean(dim=1)
        assert torch.allclose(ms, torch.ones_like(ms), atol=1e-3)


# ------------------------------------------- cross-entropy mean paths
def _ce_case(rows, cols, seed):
    d = inputs.make("cross_entropy", rows, cols, seed)
    t = to_dev(d)
    _, ref_mean = oracle.cross_entropy(d["x"], d["labels"])
    return d, t, ref_mean


def test_cross_entropy_mean_over_many_rows_and_grids():
    """The mean kernel sums per-row losses in a fixed order; the result
    matches the oracle whatever grid the loss kernel used, and the losses
    do not depend on the grid."""
    rows, cols = 70000, 33
    d, t, ref_mean = _ce_case(rows, cols, SEED + 5)
    ref_loss = oracle.cross_entropy(d["x"], d["labels"])[0]
    base = None
    for grid in (0, 1, 7, 8000, 20000):
        p = mt.make_plan(64, 1, 1, 1, grid=grid, flags=mt.MT_PLAN_PDL)
        loss, m = mt.cross_entropy(t["x"], t["labels"], plan=p)
        if base is None:
            base = loss
            assert_close(loss.cpu().numpy(), ref_loss, "losses")
        assert torch.equal(loss, base)
        assert_close(m.cpu().numpy(), np.array([ref_mean]), f"grid {grid}")


def test_cross_entropy_mean_under_graph_capture():
    """The loss kernel and the dependent mean kernel captured into a CUDA
    graph, with and without an eager call on the stream first, replay
    correctly many times."""
    rows, cols = 1024, 4096
    d, t, ref_mean = _ce_case(rows, cols, SEED + 6)
    loss = torch.empty(rows, device="cuda")
    for warm in (False, True):
        s = torch.cuda.Stream()
        means = torch.full((8,), float("nan"), device="cuda")
        if warm:
            with torch.cuda.stream(s):
                mt.mt_cross_entropy_f32(t["x"], t["labels"], loss,
                                        means[0:1], rows, cols, s)
            s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            mt.mt_cross_entropy_f32(t["x"], t["labels"], loss, means[1:2],
                                    rows, cols,
                                    torch.cuda.current_stream())
        for i in range(5):
            means[1] = float("nan")
            g.replay()
            torch.cuda.synchronize()
            assert_close(means[1:2].cpu().numpy(), np.array([ref_mean]),
                         f"graph replay {i} (warm={warm})")


def test_cross_entropy_mean_on_concurrent_streams():
    rows, cols = 4096, 1000
    cases = [_ce_case(rows, cols, SEED + 7 + k) for k in range(2)]
    streams = [torch.cuda.Stream() for _ in range(2)]
    outs = [(torch.empty(rows, device="cuda"),
             torch.empty(20, device="cuda")) for _ in range(2)]
    torch.cuda.synchronize()
    for i in range(20):
        for k in range(2):
            _, t, _ = cases[k]
            with torch.cuda.stream(streams[k]):
                mt.mt_cross_entropy_f32(t["x"], t["labels"], outs[k][0],
                                        outs[k][1][i:i + 1], rows, cols,
                                        streams[k])
    torch.cuda.synchronize()
    for k in range(2):
        ref_mean = cases[k][2]
        got = outs[k][1].cpu().numpy()
        assert_close(got, np.full(20, ref_mean), f"stream {k}")
        assert len(set(got.tolist())) == 1     # deterministic per stream


def test_calls_from_several_host_threads():
    """Eight host threads, each with its own stream, call every operator at
    once; results match a single-threaded run of the same calls bit for
    bit."""
    import threading
    shapes = [(37, 3000), (5, 70001), (300, 129)]
    jobs = []
    for op in OPS:
        for rows, cols in shapes:
            d = inputs.make(op, rows, cols, SEED + rows + cols)
            jobs.append((op, {k: (torch.from_numpy(v).cuda()
                                  if isinstance(v, np.ndarray) else v)
                              for k, v in d.items()}))

    def run_all(results, idx, stream):
        with torch.cuda.stream(stream):
            for j, (op, t) in enumerate(jobs):
                if j % 8 == idx % 8:
                    results[j] = mt.run(op, t, stream=stream)
        stream.synchronize()

    # Threads first, so the library's per-device caches for these shapes'
    # plans fill concurrently; then the same calls from one thread.
    got = {}
    threads = [threading.Thread(target=run_all,
                                args=(got, i, torch.cuda.Stream()))
               for i in range(8)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    ref = {}
    for j in range(8):
        run_all(ref, j, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert set(got) == set(ref) == set(range(len(jobs)))
    for j, (op, _) in enumerate(jobs):
        for k, v in ref[j].items():
            assert torch.equal(got[j][k].view(torch.int32),
                               v.view(torch.int32)), (op, k)


# ------------------------------------------------------ ignore index
@pytest.mark.parametrize("ignore_index", [-100, 0, 7])
def test_cross_entropy_ignore_index(ignore_index):
    rows, cols = 1024, 4096
    d = inputs.make("cross_entropy", rows, cols, SEED + 11)
    lab = d["labels"].copy()
    lab[::3] = ignore_index
    lab[5] = cols + 3                 # out of range, not ignored: NaN
    t = to_dev(d)
    lt = torch.from_numpy(lab).cuda()
    loss = torch.empty(rows, device="cuda")
    mean = torch.empty(1, device="cuda")
    mt.mt_cross_entropy_ignore_f32(t["x"], lt, ignore_index, loss, mean,
                                   rows, cols)
    ref_loss, ref_mean = oracle.cross_entropy_ignore(d["x"], lab,
                                                     ignore_index)
    assert_close(loss.cpu().numpy(), ref_loss, "loss")
    assert np.isnan(mean.item()) and np.isnan(ref_mean)
    lab[5] = 1
    lt = torch.from_numpy(lab).cuda()
    for plan in (None, mt.make_plan(128, 4, 8, 1),
                 mt.make_plan(256, 4, 0, 1, mt.MT_PATH_LOOP)):
        l2, m2 = mt.cross_entropy(t["x"], lt, ignore_index=ignore_index,
                                  plan=plan)
        ref_loss, ref_mean = oracle.cross_entropy_ignore(d["x"], lab,
                                                         ignore_index)
        assert_close(l2.cpu().numpy(), ref_loss, f"loss {plan}")
        assert_close(m2.cpu().numpy(), np.array([ref_mean]), f"mean {plan}")
    # every row ignored: NaN mean, zero losses
    allig = torch.full((rows,), ignore_index, dtype=torch.int32,
                       device="cuda")
    l3, m3 = mt.cross_entropy(t["x"], allig, ignore_index=ignore_index)
    assert (l3 == 0).all() and np.isnan(m3.item())


def test_residual_rmsnorm_aliasing_and_zero_residual():
    rows, cols = 64, 4096
    d = inputs.make("residual_rmsnorm", rows, cols, SEED + 12)
    t = to_dev(d)
    y, h = mt.residual_rmsnorm(t["x"], t["residual"], t["weight"], d["eps"],
                               return_h=True)
    assert torch.equal(h, t["x"] + t["residual"])
    x2, r2 = t["x"].clone(), t["residual"].clone()
    mt.mt_residual_rmsnorm_f32(x2, r2, t["weight"], x2, r2, rows, cols,
                               d["eps"])
    assert torch.equal(x2, y) and torch.equal(r2, h)
    y0 = mt.residual_rmsnorm(t["x"], torch.zeros_like(t["x"]), t["weight"],
                             d["eps"])
    assert_close(y0.cpu().numpy(), oracle.rmsnorm(d["x"], d["weight"],
                                                  d["eps"]), "r = 0")


# ------------------------------------------ split rows (thread-block clusters)
def cluster_plans(cols, V=4):
    plans = []
    for C in (2, 4, 8, 16):
        for W in (32, 128, 512):
            for K in (1, 2, 4, 8, 16):
                p = mt.make_plan(W, V, K, 1, cluster=C,
                                 flags=mt.MT_PLAN_PDL)
                if mt.mt_plan_check(0, cols, p) == mt.MT_OK:
                    plans.append(p)
                    break
            p = mt.make_plan(W, V, 0, 1, mt.MT_PATH_LOOP, cluster=C,
                             flags=mt.MT_PLAN_PDL | mt.MT_PLAN_PREFETCH_NEXT)
            if mt.mt_plan_check(0, cols, p) == mt.MT_OK:
                plans.append(p)
    return plans


@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("shape", [(1, 65536), (3, 100003), (64, 4096),
                                   (5, 33), (7, 4103)])
def test_cluster_split_rows(op, shape):
    """Rows split across a cluster of 2, 4 or 8 CTAs (partials exchanged
    through distributed shared memory), against the oracle, with guards;
    x is shifted by one element on the odd shapes (alignment heads)."""
    rows, cols = shape
    d = inputs.make(op, rows, cols, SEED + cols + 17)
    ref = oracle.run(op, d)
    offs = {"x": 1, "y": 1, "h_out": 1, "residual": 1} if cols % 4 else {}
    plans = cluster_plans(cols)
    assert plans
    for p in plans:
        got = run_guarded(op, d, rows, cols, plan=p, offsets=offs)
        compare(op, got, ref, f"{op} {shape} {mt.mt_describe_plan(p)}")
    # a grid smaller than the row count: clusters loop over rows
    if rows > 2:
        p = mt.make_plan(128, 4, 0, 1, mt.MT_PATH_LOOP, grid=4, cluster=2)
        got = run_guarded(op, d, rows, cols, plan=p, offsets=offs)
        compare(op, got, ref, f"{op} {shape} persistent clusters")


# ------------------------------------------------------ staged rows
STAGE_OPS = ["rmsnorm", "layernorm", "softmax", "log_softmax",
             "cross_entropy", "row_sum"]


def staged_plans(cols):
    """Legal staged plans for FP32 rows of `cols`: threads, cluster sizes,
    bulk-copy pieces and persistent grids."""
    out = []
    for W, C, pieces, grid in ((128, 1, 1, 0), (256, 1, 4, 0),
                               (512, 2, 2, 0), (1024, 4, 8, 0),
                               (256, 8, 4, 0), (64, 16, 2, 0),
                               (256, 2, 4, 4), (128, 1, 2, 3)):
        p = mt.make_plan(W, 4, pieces, 1, mt.MT_PATH_STAGE, grid=grid,
                         cluster=C if C > 1 else 0, flags=mt.MT_PLAN_PDL)
        if mt.mt_plan_check(0, cols, p) == mt.MT_OK:
            out.append(p)
    return out


@pytest.mark.parametrize("op", STAGE_OPS)
@pytest.mark.parametrize("shape", [(3, 8192), (5, 40004), (2, 131072),
                                   (4, 1028)])
def test_staged_rows(op, shape):
    """Rows staged in shared memory by bulk copies (one CTA or a cluster of
    CTAs per row, 1-8 copies per run, persistent grids), against the
    oracle with guard regions; no staged wait gives up."""
    rows, cols = shape
    d = inputs.make(op, rows, cols, SEED + cols + 23)
    ref = oracle.run(op, d)
    plans = staged_plans(cols)
    assert plans
    for p in plans:
        got = run_guarded(op, d, rows, cols, plan=p)
        compare(op, got, ref, f"{op} {shape} {mt.mt_describe_plan(p)}")
    assert mt.mt_stage_wait_timeouts() == 0


def test_staged_plan_needs_aligned_rows():
    """A forced staged plan on rows off the 16-byte grid is refused before
    any launch."""
    rows, cols = 3, 8192
    p = mt.make_plan(256, 4, 2, 1, mt.MT_PATH_STAGE)
    d = inputs.make("softmax", rows, cols, SEED)
    bufs = {"x": Guarded(rows * cols, 1, float("nan"), data=d["x"]),
            "y": Guarded(rows * cols, 0, Guarded.SENTINEL)}
    with pytest.raises(mt.MTError) as e:
        call("softmax", {k: b.ptr for k, b in bufs.items()}, rows, cols,
             plan=p)
    assert e.value.status == mt.MT_ERR_INVALID_ARGUMENT
    torch.cuda.synchronize()
    for b in bufs.values():
        b.check()


# ------------------------------------------------- masked (-inf) runs
def masked_logits(rows, cols, seed):
    """Softmax inputs N(0, 2^2) with runs of -inf covering whole packs and
    more: a row's head, its tail, alternate 16-value blocks, all but one
    value, pack-straddling runs, and one row without any."""
    d = inputs.make("cross_entropy", rows, cols, seed)
    x = d["x"]
    x[0, :min(cols - 1, 64)] = -np.inf
    x[1 % rows, max(1, cols - 100):] = -np.inf
    for lo in range(0, cols - 16, 32):
        x[2 % rows, lo:lo + 16] = -np.inf
    x[3 % rows, 1:] = -np.inf
    x[4 % rows, 3:cols - 5] = -np.inf
    d["labels"] = np.array([int(np.flatnonzero(np.isfinite(r))[k % 7 %
                            max(1, np.isfinite(r).sum())])
                            for k, r in enumerate(x)], dtype=np.int32)
    return d


@pytest.mark.parametrize("op", ["softmax", "log_softmax", "cross_entropy"])
@pytest.mark.parametrize("cols", [257, 4103, 20000])
def test_masked_runs_of_minus_infinity(op, cols):
    """-inf entries contribute exp(-inf) = 0: rows whose packs are wholly
    -inf stay finite on the register, loop and cluster paths (only an
    all -inf row is NaN, in the oracle as on the GPU)."""
    rows = 6
    d = masked_logits(rows, cols, SEED + cols)
    dd = {"x": d["x"]} if op != "cross_entropy" else \
        {"x": d["x"], "labels": d["labels"]}
    ref = oracle.run(op, dd)
    plans = [None] + [p for p in candidate_plans(min(cols, 4103))
                      if cols <= 4103 or p.path == mt.MT_PATH_LOOP][::3]
    if cols >= 4103:
        plans += cluster_plans(cols)
    if cols % 4 == 0:
        plans += staged_plans(cols)
    for p in plans:
        if p is not None and mt.mt_plan_check(mt.OP_IDS[op], cols, p) != 0:
            continue
        got = run_guarded(op, dd, rows, cols, plan=p)
        what = f"{op} masked {rows}x{cols} " + (
            "default" if p is None else mt.mt_describe_plan(p))
        for k, r in ref.items():
            # finite everywhere (log-softmax: wherever x is finite)
            fin = np.isfinite(dd["x"]) if op == "log_softmax" else True
            assert np.isfinite(r[fin]).all(), (what, k)
        compare(op, got, ref, what)
