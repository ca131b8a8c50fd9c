"""Host-side checks of the C ABI (no GPU needed): the library builds, loads
and exports every symbol the header declares; the planner's legality rules
and private-slot bound; argument errors that are caught before any CUDA call.

The ownership map is pinned to the example tables the pages print
(tests/golden/): "Consecutive-worker reduction layout checkpoint",
§Implementation and semantics (W=4, V=2), and "Thread Ownership and Software
Staging", §Register-tiled reductions (striped and adjacent 4-register
ownership of a 1024-element tile).
"""
import os
import re

import pytest

import row_reduction_gb300 as mt
from row_reduction_gb300 import build as mt_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module", autouse=True)
def built():
    mt_build.build()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "mt_rowreduce.h")).read()
    return sorted(set(re.findall(r"^MT_API[^(]*?\b(mt_\w+)\s*\(", src,
                                 flags=re.M)))


def test_library_exports_every_declared_symbol():
    declared = header_symbols()
    assert len(declared) == 48
    L = mt.lib()
    for name in declared:
        assert hasattr(L, name), name
    assert sorted(mt.EXPORTS) == declared


# ---------------------------------------------------------------- ownership
def owner(i, W, V):
    """(chunk, worker, element) of logical element i: i = (chunk*W +
    worker)*V + element."""
    return i // (W * V), (i // V) % W, i % V


def logical(chunk, worker, element, W, V):
    return (chunk * W + worker) * V + element


def read_table(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def test_ownership_matches_printed_w4_v2_table():
    for chunk, worker, e0, e1 in read_table("ownership_w4_v2.txt"):
        c, w = int(chunk), int(worker)
        assert [logical(c, w, e, 4, 2) for e in (0, 1)] == [int(e0), int(e1)]
        for e, i in enumerate((int(e0), int(e1))):
            assert owner(i, 4, 2) == (c, w, e)


def test_register_ownership_striped_and_adjacent():
    for layout, t, *slots in read_table("register_ownership_1024x4.txt"):
        t = int(t)
        slots = [int(s) for s in slots]
        if layout == "striped":      # V = 1 with four chunks of W = 256
            got = [logical(k, t, 0, 256, 1) for k in range(4)]
        else:                        # V = 4, one chunk, W = 256
            got = [logical(0, t, e, 256, 4) for e in range(4)]
        assert got == slots, (layout, t)


def test_private_slot_bound_matches_brute_force():
    for W in (1, 2, 4, 8, 32):
        for V in (1, 2, 4, 8):
            for n in list(range(0, 70)) + [127, 128, 129, 257, 4103]:
                counts = [0] * W
                for i in range(n):
                    counts[owner(i, W, V)[1]] += 1
                assert mt.mt_private_slot_bound(n, W, V) == max(counts), \
                    (n, W, V)
    assert mt.mt_private_slot_bound(-1, 4, 4) == -1
    assert mt.mt_private_slot_bound(10, 0, 4) == -1


# ---------------------------------------------------------------- planner
OK, INV, OOR = mt.MT_OK, mt.MT_ERR_INVALID_ARGUMENT, mt.MT_ERR_OUT_OF_RESOURCES
REG, LOOP = mt.MT_PATH_REGISTERS, mt.MT_PATH_LOOP


@pytest.mark.parametrize("plan,cols,want", [
    (dict(W=256, V=4, chunks=4), 4096, OK),
    (dict(W=256, V=4, chunks=2), 4096, OOR),      # row does not fit
    (dict(W=300, V=4, chunks=4), 4096, INV),      # W not a power of two
    (dict(W=2048, V=4, chunks=1), 4096, INV),     # W > 1024
    (dict(W=256, V=3, chunks=4), 4096, INV),      # V not 1/2/4
    (dict(W=256, V=8, chunks=4), 4096, INV),
    (dict(W=256, V=4, chunks=3), 3000, INV),      # chunks not instantiated
    (dict(W=16, V=4, chunks=4, rows_per_block=1), 200, INV),  # half a warp
    (dict(W=2, V=4, chunks=16, rows_per_block=16), 100, INV),  # W < V
    (dict(W=1024, V=4, chunks=16), 65536, OOR),   # over the kernel's threads
    (dict(W=256, V=4, chunks=16), 16384, OK),
    (dict(W=512, V=4, chunks=0, path=LOOP), 10 ** 6, OK),
    (dict(W=1024, V=4, chunks=0, path=LOOP), 10 ** 6, OOR),
    (dict(W=256, V=4, chunks=4, path=7), 4096, INV),
    (dict(W=256, V=4, chunks=4, grid=-1), 4096, INV),
    (dict(W=256, V=4, chunks=4, rows_per_block=0), 4096, INV),
    (dict(W=1, V=1, chunks=1, rows_per_block=32), 1, OK),
])
def test_plan_check(plan, cols, want):
    p = mt.make_plan(plan["W"], plan["V"], plan.get("chunks", 0),
                     plan.get("rows_per_block", 1), plan.get("path", REG),
                     plan.get("grid", 0))
    for op in range(8):
        assert mt.mt_plan_check(op, cols, p) == want


@pytest.mark.parametrize("op", list(mt.OP_IDS))
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_default_plans_are_legal(op, dtype):
    shapes = [(r, c) for r in (0, 1, 5, 17, 64, 1024, 65536)
              for c in (1, 2, 3, 4, 7, 31, 33, 127, 128, 129, 257, 1000,
                        1024, 4096, 4103, 8192, 16384, 32768, 100003)]
    for rows, cols in shapes:
        p = mt.mt_plan_query_dtype(op, dtype, rows, cols)
        assert mt.mt_plan_check_dtype(op, dtype, cols, p) == OK, \
            (rows, cols, p)
        assert p.grid >= 0
        if dtype == "f32":
            assert tuple(p.as_dict().values()) == tuple(
                mt.mt_plan_query(op, rows, cols).as_dict().values())


def test_plan_check_per_storage_type():
    # FP32 packs hold 1, 2 or 4 values; FP16/BF16 packs 2, 4 or 8.
    K = {1: 8, 2: 4, 4: 2, 8: 1}        # 512 * V * K = 4096
    for V, want in ((1, OK), (2, OK), (4, OK), (8, INV)):
        assert mt.mt_plan_check_dtype(0, "f32", 4096,
                                      mt.make_plan(512, V, K[V], 1)) == want
    for dt in ("f16", "bf16"):
        for V, want in ((1, INV), (2, OK), (4, OK), (8, OK)):
            assert mt.mt_plan_check_dtype(
                0, dt, 4096, mt.make_plan(512, V, K[V], 1)) == want
    assert mt.lib().mt_plan_check_dtype(0, 3, 4096, None) == INV
    import ctypes
    p = mt.make_plan(256, 4, 4, 1)
    assert mt.lib().mt_plan_check_dtype(0, 3, 4096, ctypes.byref(p)) == INV
    assert mt.lib().mt_plan_check_dtype(0, -1, 4096, ctypes.byref(p)) == INV


def test_plan_query_errors_and_describe():
    with pytest.raises(mt.MTError):
        mt.mt_plan_query(8, 1, 1)
    with pytest.raises(mt.MTError):
        mt.mt_plan_query(0, -1, 1)
    with pytest.raises(mt.MTError):
        mt.mt_plan_query(0, 1, 0)
    s = mt.mt_describe_plan(mt.make_plan(128, 4, 8, 2))
    assert s == ("path=registers W=128 V=4 chunks=8 rows_per_block=2 "
                 "threads=256 grid=auto")
    assert mt.mt_describe_plan(mt.make_plan(512, 2, 0, 1, LOOP, 304)).endswith(
        "grid=304")
    assert mt.status_string(OOR) == "MT_ERR_OUT_OF_RESOURCES"
    assert mt.status_string(99) == "MT_ERR_UNKNOWN"


def test_plan_flags():
    every = (mt.MT_PLAN_PDL | mt.MT_PLAN_PREFETCH_NEXT |
             mt.MT_PLAN_WHOLE_TILES)
    for fl in range(every + 1):
        p = mt.make_plan(128, 4, 8, 2, grid=152, flags=fl)
        assert mt.mt_plan_check(0, 4096, p) == OK
    for fl in (8, 16, -1, every | 8):
        p = mt.make_plan(128, 4, 8, 2, flags=fl)
        assert mt.mt_plan_check(0, 4096, p) == INV
    both = mt.MT_PLAN_PDL | mt.MT_PLAN_PREFETCH_NEXT
    s = mt.mt_describe_plan(mt.make_plan(128, 4, 8, 2, grid=152, flags=both))
    assert s.endswith("grid=152 pdl prefetch_next")
    s = mt.mt_describe_plan(mt.make_plan(128, 4, 8, 2, flags=every))
    assert s.endswith("pdl prefetch_next whole_tiles")


# ------------------------------------------------------ argument validation
# These return before any CUDA call, so they run without a GPU.  Addresses
# are arbitrary 16-byte aligned integers that are never dereferenced.
A = 1 << 20


def status(fn, *args):
    return getattr(mt.lib(), fn)(*args)


def test_invalid_arguments_are_rejected_before_launch():
    L = mt.lib()
    assert L.mt_rmsnorm_f32(None, None, A, 4, 4, 1e-6, None) == INV
    assert L.mt_rmsnorm_f32(A, None, None, 4, 4, 1e-6, None) == INV
    assert L.mt_rmsnorm_f32(A + 2, None, A, 4, 4, 1e-6, None) == INV
    assert L.mt_rmsnorm_f32(A, A + 1, A, 4, 4, 1e-6, None) == INV
    assert L.mt_rmsnorm_f32(A, None, A, -1, 4, 1e-6, None) == INV
    assert L.mt_rmsnorm_f32(A, None, A, 4, 0, 1e-6, None) == INV
    assert L.mt_rmsnorm_f32(A, None, A, 4, 1 << 31, 1e-6, None) == INV
    assert L.mt_rmsnorm_f32(A, None, A, 1 << 40, 1 << 30, 1e-6, None) == INV
    assert L.mt_layernorm_f32(A, None, A + 3, A, 4, 4, 1e-5, None) == INV
    assert L.mt_residual_layernorm_f32(A, None, None, None, A, None, 4, 4,
                                       1e-5, None) == INV
    assert L.mt_softmax_f32(A, None, 4, 4, None) == INV
    assert L.mt_row_sum_f32(A, None, 4, 4, None) == INV
    assert L.mt_cross_entropy_f32(A, None, A, None, 4, 4, None) == INV
    assert L.mt_cross_entropy_f32(A, A, A, A + 2, 4, 4, None) == INV


def test_probe_arguments_are_rejected_before_launch():
    """The measurement aids check their arguments before any CUDA call."""
    L = mt.lib()
    assert L.mt_probe_copy(A, A + 4096, 4095, 512, 4, 0, 0, None) == INV
    assert L.mt_probe_copy(A, A + 4096, -16, 512, 4, 0, 0, None) == INV
    assert L.mt_probe_copy(A, A + 4096, 4096, 500, 4, 0, 0, None) == INV
    assert L.mt_probe_copy(A, A + 4096, 4096, 2048, 4, 0, 0, None) == INV
    assert L.mt_probe_copy(A, A + 4096, 4096, 512, 3, 0, 0, None) == INV
    assert L.mt_probe_copy(A, A + 4096, 4096, 512, 4, -1, 0, None) == INV
    assert L.mt_probe_copy(A, A + 4096, 4096, 512, 4, 0, 2, None) == INV
    assert L.mt_probe_copy(A + 4, A + 4096, 4096, 512, 4, 0, 0, None) == INV
    assert L.mt_probe_copy(None, A, 4096, 512, 4, 0, 0, None) == INV
    assert L.mt_probe_copy(A, A + 2048, 4096, 512, 4, 0, 0, None) == INV
    assert L.mt_probe_copy(A, A + 4096, 0, 512, 4, 0, 0, None) == OK
    assert L.mt_probe_read(A, 4095, A + 8192, 64, 512, 4, 0, 0, None) == INV
    assert L.mt_probe_read(A, 4096, A + 8192, 64, 512, 3, 0, 0, None) == INV
    assert L.mt_probe_read(A, 4096, A + 8192, 64, 512, 4, 65, 0, None) == INV
    assert L.mt_probe_read(A, 4096, A + 8194, 64, 512, 4, 8, 0, None) == INV
    assert L.mt_probe_read(A + 8, 4096, A + 8192, 64, 512, 4, 8, 0,
                           None) == INV
    assert L.mt_probe_read(A, 4096, None, 64, 512, 4, 8, 0, None) == INV
    assert L.mt_probe_read(A, 4096, A + 8192, 64, 512, 4, 8, 2, None) == INV
    assert L.mt_probe_read(A, 0, A + 8192, 64, 512, 4, 8, 0, None) == OK
    assert L.mt_probe_empty(16, 1, None) == INV
    assert L.mt_probe_empty(32, -1, None) == INV


def test_zero_rows_is_a_no_op():
    L = mt.lib()
    assert L.mt_rmsnorm_f32(A, None, A, 0, 4096, 1e-6, None) == OK
    assert L.mt_softmax_f32(A, A, 0, 7, None) == OK
    assert L.mt_cross_entropy_f32(A, A, A, A, 0, 7, None) == OK


def test_forced_illegal_plan_fails_closed():
    bad = mt.make_plan(256, 4, 2, 1)          # cannot hold 4096 columns
    f = mt.lib().mt_rmsnorm_f32_with_plan
    import ctypes
    assert f(A, None, A, 4, 4096, 1e-6, None, ctypes.byref(bad)) == OOR
    bad = mt.make_plan(100, 4, 16, 1)
    assert f(A, None, A, 4, 4096, 1e-6, None, ctypes.byref(bad)) == INV
    # rows == 0 still validates the plan
    assert f(A, None, A, 0, 4096, 1e-6, None, ctypes.byref(bad)) == INV


def test_generic_and_half_entry_points_validate_before_launch():
    L = mt.lib()
    f = L.mt_row_reduce_with_plan
    # op, dtype, x, res, w, b, labels, y, h, out, mean, rows, cols, eps, s, plan
    NI = mt.MT_NO_IGNORE_INDEX
    assert f(0, 2, A, None, None, None, None, NI, A, None, None, None, 0, 8,
             0.0, None, None) == OK
    # a pointer the operator does not take
    assert f(0, 2, A, None, None, None, None, NI, A, None, A, None, 4, 8,
             0.0, None, None) == INV
    assert f(3, 0, A, None, A, None, None, NI, A, None, None, None, 4, 8,
             0.0, None, None) == INV
    assert f(7, 0, A, A, None, None, None, NI, A, None, None, None, 4, 8,
             0.0, None, None) == INV
    # a missing required pointer / unknown op or dtype
    assert f(4, 1, A, None, None, None, None, NI, None, None, None, None, 4,
             8, 0.0, None, None) == INV
    assert f(6, 0, A, None, None, None, None, NI, A, None, None, None, 4, 8,
             0.0, None, None) == INV      # residual RMSNorm needs residual
    assert f(8, 0, A, None, None, None, None, NI, A, None, None, None, 4, 8,
             0.0, None, None) == INV
    assert f(0, 3, A, None, None, None, None, NI, A, None, None, None, 4, 8,
             0.0, None, None) == INV
    # 16-bit storage needs 2-byte alignment; FP32 outputs need 4
    assert L.mt_rmsnorm_bf16(A + 1, None, A, 4, 8, 1e-6, None) == INV
    assert L.mt_rmsnorm_bf16(A + 2, None, A + 6, 0, 8, 1e-6, None) == OK
    assert L.mt_row_sum_f16(A + 2, A + 2, 4, 8, None) == INV
    assert L.mt_cross_entropy_bf16(A, None, A, None, 4, 8, None) == INV
    assert L.mt_residual_layernorm_f16(A, None, None, None, A, None, 4, 8,
                                       1e-5, None) == INV


def test_cluster_plan_legality():
    ok = dict(W=256, V=4, chunks=4, rows_per_block=1)
    def chk(cols, dtype="f32", **kw):
        d = dict(ok, **kw)
        p = mt.make_plan(d["W"], d["V"], d["chunks"], d["rows_per_block"],
                         d.get("path", REG), d.get("grid", 0), 0,
                         d.get("cluster", 0))
        return mt.mt_plan_check_dtype(0, dtype, cols, p)
    assert chk(16384, cluster=4) == OK          # 4 * 256 * 4 * 4 = 16384
    assert chk(16384, cluster=2) == OOR         # half the row does not fit
    assert chk(16384, cluster=3) == INV
    assert chk(16384, cluster=16) == OK         # 16 CTAs: non-portable size
    assert chk(16384, cluster=32) == INV
    assert chk(16384, cluster=-1) == INV
    assert chk(16384, cluster=4, rows_per_block=2) == INV
    assert chk(4096, cluster=2, W=16, chunks=16, rows_per_block=2) == INV
    assert chk(16384, cluster=4, V=2, chunks=8) == INV   # not 16-byte packs
    assert chk(16384, cluster=4, grid=6) == INV          # not a multiple
    assert chk(16384, cluster=4, grid=8) == OK
    assert chk(16384, "bf16", cluster=4, V=8, chunks=2) == OK
    assert chk(16384, "bf16", cluster=4, V=4, chunks=4) == INV
    assert chk(10 ** 6, cluster=8, chunks=0, path=LOOP) == OK
    s = mt.mt_describe_plan(mt.make_plan(256, 4, 4, 1, cluster=4))
    assert "cluster=4" in s
