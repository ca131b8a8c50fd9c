"""Seeded random sweep of the plan space against the oracle: operator,
storage type, shape, plan (path, W, V, chunks, rows per CTA, cluster, grid,
flags) and, for FP32, base-pointer offsets, all drawn at random.  Every drawn
plan passes mt_plan_check before it runs; every guard region is checked."""
import numpy as np
import pytest

import row_reduction_gb300 as mt
from row_reduction_gb300 import inputs
from test_parity_gpu import compare, run_guarded
from test_parity_half_gpu import case, check, run as run16

import oracle

pytestmark = pytest.mark.gpu

CASES = 160
VALUES = {"f32": (1, 2, 4), "f16": (2, 4, 8), "bf16": (2, 4, 8)}


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_reduction_gb300 import build
    build.build()
    oracle.build()


def random_plan(rng, op, dt, cols):
    op_id = mt.OP_IDS[op]
    for _ in range(400):
        V = int(rng.choice(VALUES[dt]))
        W = int(2 ** rng.integers(0, 11))
        path = int(rng.choice([mt.MT_PATH_REGISTERS, mt.MT_PATH_LOOP]))
        cluster = int(rng.choice([0, 0, 0, 2, 4, 8, 16]))
        B = int(2 ** rng.integers(0, 6))
        K = 0
        if path == mt.MT_PATH_REGISTERS:
            C = max(1, cluster)
            K = next((k for k in (1, 2, 4, 8, 16) if C * W * V * k >= cols),
                     None)
            if K is None:
                continue
        grid = int(rng.choice([0, 0, 1, 3, 7, 152, 304]))
        if cluster > 1:
            grid -= grid % cluster
        flags = int(rng.integers(0, 4))
        p = mt.make_plan(W, V, K, B, path, grid=grid, flags=flags,
                         cluster=cluster)
        if mt.mt_plan_check_dtype(op_id, dt, cols, p) == mt.MT_OK:
            return p
    return None


def test_random_plans_shapes_and_offsets():
    rng = np.random.default_rng(inputs.HOLDOUT_SEED)
    ran = 0
    for i in range(CASES):
        op = str(rng.choice(inputs.ALL_OPS))
        dt = str(rng.choice(["f32", "f32", "bf16", "f16"]))
        rows = int(np.exp(rng.uniform(0, np.log(300))))
        cols = int(np.exp(rng.uniform(0, np.log(40000))))
        p = random_plan(rng, op, dt, cols)
        if p is None:
            continue
        what = f"case {i}: {op} {dt} {rows}x{cols} {mt.mt_describe_plan(p)}"
        seed = inputs.HOLDOUT_SEED + i
        if dt == "f32":
            offs = {k: int(rng.integers(0, 4))
                    for k in ("x", "y", "h_out", "residual")}
            d = inputs.make(op, rows, cols, seed)
            got = run_guarded(op, d, rows, cols, plan=p, offsets=offs)
            compare(op, got, oracle.run(op, d), f"{what} offsets {offs}")
        else:
            st, wide = case(op, rows, cols, dt, seed)
            outs = run16(op, st, dt, rows, cols, plan=p)
            check(op, dt, outs, st, wide, what)
        ran += 1
    assert ran >= CASES * 3 // 4
