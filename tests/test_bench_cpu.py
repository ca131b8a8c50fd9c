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
