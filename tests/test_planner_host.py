"""Host-side checks of the planner and the input generator's storage
rounding (no GPU): every measured table entry is a legal plan, and the
documented planning rules hold on the shapes they were measured on."""
import json
import os

import numpy as np
import pytest
import torch

import row_reduction_gb300 as mt
from row_reduction_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "row_reduction_gb300", "csrc", "plan_table.json")


def plan(op, dt, rows, cols):
    return mt.mt_plan_query_dtype(op, dt, rows, cols)


def test_every_table_winner_is_legal_and_served():
    recs = json.load(open(TABLE))["records"]
    assert len(recs) >= 100
    for r in recs:
        dt = r.get("dtype", "f32")
        w = mt.MtPlan(**r["winner"])
        assert mt.mt_plan_check_dtype(mt.OP_IDS[r["op"]], dt, r["cols"],
                                      w) == mt.MT_OK, r["winner_text"]
        # the planner returns the measured winner on its own shape
        got = plan(r["op"], dt, r["rows"], r["cols"]).as_dict()
        assert got == w.as_dict(), (r["op"], dt, r["rows"], r["cols"])


def test_few_wide_rows_split_across_clusters():
    # up to 9 rows: 16 CTAs per row; up to 19: 8; up to 38: 4; more rows
    # of a staged operator: the staged path on the smallest cluster whose
    # runs take at most 160 KiB (300000 FP32 values: 8 CTAs)
    for rows, C in ((1, 16), (9, 16), (10, 8), (19, 8), (20, 4), (38, 4)):
        p = plan("layernorm", "f32", rows, 300000)
        assert p.cluster == C and p.path != mt.MT_PATH_STAGE, (rows,
                                                               p.as_dict())
    for rows in (39, 76, 5000):
        p = plan("layernorm", "f32", rows, 300000)
        assert (p.path, p.cluster) == (mt.MT_PATH_STAGE, 8), (rows,
                                                              p.as_dict())
    # 20 rows of a one-pass operator are staged too: 8 CTAs per run fit
    # 160 KiB, 16 give the rows 1.5 CTAs per SM
    p = plan("row_sum", "f32", 20, 300000)
    assert (p.path, p.cluster) == (mt.MT_PATH_STAGE, 16), p.as_dict()


def test_many_wide_rows_are_staged_or_held_in_registers():
    # The staged operators read many wide rows once through shared memory,
    # on the smallest cluster whose runs take at most 128 KiB.
    p = plan("layernorm", "f32", 8192, 32000)
    assert p.path == mt.MT_PATH_STAGE and p.cluster <= 1
    p = plan("layernorm", "bf16", 8192, 32000)
    assert p.path == mt.MT_PATH_STAGE and p.cluster <= 1
    p = plan("layernorm", "f32", 8192, 65536)
    assert (p.path, p.cluster) == (mt.MT_PATH_STAGE, 2)
    # The residual operators have no staged path: 32000 FP32 values need
    # two CTAs of 256 threads x 16 chunks, wider rows the loop path.
    p = plan("residual_layernorm", "f32", 8192, 32000)
    assert (p.path, p.cluster) == (mt.MT_PATH_REGISTERS, 2)
    assert plan("residual_layernorm", "f32", 8192,
                65536).path == mt.MT_PATH_LOOP
    # Rows that are not a whole number of 16-byte units: the loop path.
    assert plan("softmax", "bf16", 128, 50257).path == mt.MT_PATH_LOOP


def test_staged_plans_need_whole_units():
    p = mt.make_plan(256, 4, 2, 1, mt.MT_PATH_STAGE)
    assert mt.mt_plan_check(mt.OP_IDS["softmax"], 8192, p) == mt.MT_OK
    assert mt.mt_plan_check(mt.OP_IDS["softmax"], 8194,
                            p) == mt.MT_ERR_INVALID_ARGUMENT
    # no staged path for the residual operators
    assert mt.mt_plan_check(mt.OP_IDS["residual_layernorm"], 8192,
                            p) == mt.MT_ERR_INVALID_ARGUMENT
    # a run beyond the shared-memory budget
    assert mt.mt_plan_check(mt.OP_IDS["softmax"], 65536,
                            p) == mt.MT_ERR_OUT_OF_RESOURCES
    q = mt.make_plan(256, 4, 2, 1, mt.MT_PATH_STAGE, cluster=2, grid=0)
    assert mt.mt_plan_check(mt.OP_IDS["softmax"], 65536, q) == mt.MT_OK


def test_shape_plans_avoid_the_spilling_fp32_instance():
    # ptxas holds RMSNorm's FP32 4-value, 2-chunk instance to 32 registers
    # (it spills): rows that would take it use 2-value packs instead
    for rows, cols in ((512, 2048), (300, 3000)):
        p = plan("rmsnorm", "f32", rows, cols)
        assert not (p.values_per_thread == 4 and p.chunks == 2 and
                    p.path == mt.MT_PATH_REGISTERS), (rows, cols)


def test_loop_heuristic_leaves_the_next_group_prefetch_off():
    # wide rows of an operator without a staged path
    p = plan("residual_layernorm", "f32", 2048, 131072)
    assert p.path == mt.MT_PATH_LOOP
    assert not p.flags & mt.MT_PLAN_PREFETCH_NEXT


def test_shape_derived_plans_price_active_groups_and_work_per_sm():
    # Values per thread follow the work per SM (R*cols / (152*512), 8..32)
    # and CTAs keep at least two active groups per SM.
    p = plan("layernorm", "f16", 512, 768)         # little work: 8 values
    assert p.values_per_thread * p.chunks == 8
    assert -(-512 // p.rows_per_block) >= 2 * 152
    p = plan("rmsnorm", "f16", 777, 5000)           # more work: 32 values
    assert (p.threads_per_row, p.values_per_thread, p.chunks) == (256, 8, 4)
    p = plan("rmsnorm", "f32", 300, 3000)           # FP32 at 8: 2-value packs
    assert (p.threads_per_row, p.values_per_thread, p.chunks) == (512, 2, 4)
    p = plan("residual_rmsnorm", "f32", 2048, 3072)  # residual: at most 16
    assert p.values_per_thread * p.chunks <= 16
    p = plan("row_sum", "f16", 700, 300)            # short rows packed, but
    assert -(-700 // p.rows_per_block) >= 2 * 152   # >= 2 groups per SM
    # an exact tiling takes the whole-tile variant
    p = plan("layernorm", "f32", 2048, 1024)
    assert p.threads_per_row * p.values_per_thread * p.chunks == 1024
    assert p.flags & mt.MT_PLAN_WHOLE_TILES


@pytest.mark.parametrize("seed", [1, 2, 3])
def test_bf16_storage_rounding_matches_torch(seed):
    """The generator's BF16 rounding (nearest even, on the bit pattern) is
    torch's; FP16 is NumPy's IEEE conversion; widening is exact."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(4096) *
         10.0 ** rng.integers(-20, 20, 4096)).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]  # ties
    st = inputs.as_storage({"x": x}, "bf16")["x"]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy()
    assert np.array_equal(st.view(np.int16), ref)
    wide = inputs.widen(st, "bf16")
    assert np.array_equal(
        wide, torch.from_numpy(x).to(torch.bfloat16).float().numpy())
    h = inputs.as_storage({"x": np.clip(x, -6e4, 6e4)}, "f16")["x"]
    assert h.dtype == np.float16
    assert np.array_equal(inputs.widen(h, "f16"), h.astype(np.float32))


def test_tuner_candidates_are_legal_and_cover_the_plan_space():
    from row_reduction_gb300 import tune
    for op, rows, cols, dt in (("rmsnorm", 1, 1048576, "f32"),
                               ("softmax", 4096, 32000, "bf16"),
                               ("layernorm", 1024, 4096, "f32"),
                               ("cross_entropy", 17, 257, "f16")):
        cands = tune.candidates(op, rows, cols, dt)
        assert cands
        for p in cands:
            assert mt.mt_plan_check_dtype(mt.OP_IDS[op], dt, cols,
                                          p) == mt.MT_OK
        clusters = {p.cluster for p in cands}
        if cols > 16384 or (rows < 304 and cols >= 1024):
            assert clusters & {2, 4, 8}
        if rows <= 19 and cols >= 1024:
            assert 16 in clusters
        paths = {p.path for p in cands}
        assert mt.MT_PATH_REGISTERS in paths or cols > 16384
        if cols >= 8192:
            assert mt.MT_PATH_LOOP in paths
        # second stage: persistent grids below the row-group count
        extra = tune.grid_variants(rows, cands[:4], 152)
        for p in extra:
            C = max(1, p.cluster)
            assert p.grid % C == 0
            assert p.grid // C < -(-rows // p.rows_per_block)


def _table_entries():
    import re
    path = os.path.join(os.path.dirname(os.path.dirname(
        os.path.abspath(__file__))), "row_reduction_gb300", "csrc",
        "plan_table.inc")
    out = []
    for line in open(path):
        m = re.match(r"\s*\{(\d+), (\d+), (\d+), (\d+), (\d+), (\d+),",
                     line)
        if m:
            out.append(tuple(int(v) for v in m.groups()))
    return out


def test_heldout_cases_cover_every_operator_and_type_outside_the_table():
    """The regret set spans all operators and storage types, and no case is
    served by a table entry (so it measures the re-fit and heuristic)."""
    from row_reduction_gb300 import tune, inputs
    import row_reduction_gb300 as mt
    cases = [tune.parse_case(c) for c in tune.HELDOUT_CASES]
    assert len(cases) >= 30
    assert {c[1] for c in cases} == set(inputs.ALL_OPS)
    assert {c[0] for c in cases} == {"f32", "f16", "bf16"}
    table = _table_entries()
    assert table
    for dt, op, rows, cols in cases:
        for e_op, e_dt, c0, c1, r0, r1 in table:
            hit = (e_op == mt.OP_IDS[op] and e_dt == mt.DTYPE_IDS[dt] and
                   c0 <= cols <= c1 and r0 <= rows <= r1)
            assert not hit, (op, dt, rows, cols)


def test_every_planned_shape_is_legal():
    """The planner's choice (table, shape-derived fallback or heuristic)
    passes the library's own legality check across row lengths from 1 to
    2**21 (aligned and not), row counts from 1 to 2**20, every operator and
    storage type."""
    cols_list = sorted({1, 2, 3, 7, 31, 33, 127, 257, 300, 768, 1000, 1024,
                        2500, 4096, 4103, 5000, 8192, 12288, 16385, 20000,
                        32000, 32768, 50257, 65536, 100003, 131072, 300000,
                        1 << 20, (1 << 21) + 8})
    rows_list = (1, 2, 9, 10, 17, 38, 39, 76, 77, 128, 303, 304, 1000, 4096,
                 65536, 1 << 20)
    for op in mt.OP_IDS:
        for dt in ("f32", "f16", "bf16"):
            for cols in cols_list:
                for rows in rows_list:
                    p = plan(op, dt, rows, cols)
                    st = mt.mt_plan_check_dtype(op, dt, cols, p)
                    assert st == mt.MT_OK, (op, dt, rows, cols, p.as_dict())
