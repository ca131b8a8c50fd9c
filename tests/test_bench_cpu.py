"""The benchmark's reference arm (the CPU oracle) and its JSON line, on the
CPU: the keys the line must carry and the arithmetic of its value."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def run_reference(*extra):
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
         "reference", "--steps", "3", "--warmup", "3", *extra],
        cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("extra", [(), ("--op", "cross_entropy", "--dtype",
                                        "bf16", "--rows", "64")])
def test_reference_arm_json_line(extra):
    line = run_reference(*extra)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup",
                "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
                "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    cfg = line["config"]
    assert cfg["rows"] >= cfg["sample_rows_per_step"] >= 1


def test_bench_warmup_must_be_at_least_three():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
         "reference", "--steps", "3", "--warmup", "2"],
        cwd=ROOT, capture_output=True, text=True, timeout=120)
    assert out.returncode != 0


def test_algorithmic_bytes_match_the_documented_formulas():
    from row_reduction_gb300.timing import algorithmic_bytes
    R, C = 1024, 4096
    assert algorithmic_bytes("rmsnorm", R, C) == 33570816
    assert algorithmic_bytes("layernorm", R, C) == 33587200
    assert algorithmic_bytes("residual_layernorm", R, C, h_out=True) == \
        67141632
    assert algorithmic_bytes("residual_rmsnorm", R, C, h_out=True) == \
        67125248
    assert algorithmic_bytes("softmax", R, C) == 33554432
    assert algorithmic_bytes("log_softmax", R, C) == 33554432
    assert algorithmic_bytes("row_sum", R, C) == 16781312
    assert algorithmic_bytes("cross_entropy", R, C, mean=True) == 16785412
    assert algorithmic_bytes("rmsnorm", R, C, dtype="bf16") == \
        4 * R * C + 2 * C


def _line(us=5.9, plan=None):
    import bench
    from row_reduction_gb300.timing import algorithmic_bytes
    b = algorithmic_bytes("rmsnorm", 1024, 4096)
    ach = b / (us * 1e-6) / 1e9
    return {"metric": "m", "value": ach, "unit": "GB/s", "n_gpus": 1,
            "steps": 100, "warmup": 10, "ms_per_step": us / 1e3,
            "us_per_op": us,
            "config": {"op": "rmsnorm", "storage": "f32", "rows": 1024,
                       "cols": 4096,
                       "plan": plan or bench.plan_text("rmsnorm", 1024,
                                                       4096)},
            "roofline": {"achieved": ach, "peak": 6783.1,
                         "frac": ach / 6783.1},
            "rounds": {"us_per_op_median": 5.95, "us_per_op_min": 5.9,
                       "us_per_op_max": 6.0,
                       "samples_us": [5.9, 5.95, 6.0]}}


def test_verify_accepts_a_consistent_line_and_flags_the_rest():
    import bench
    assert bench.verify_line(_line()) == []
    bad = _line()
    bad["value"] *= 1.01
    bad["rounds"]["us_per_op_median"] = 5.0
    problems = bench.verify_line(bad)
    assert any(p.startswith("value") for p in problems)
    assert any(p.startswith("rounds median") for p in problems)
    assert bench.verify_line(_line(plan="path=loop W=1"))[0].startswith(
        "plan")
