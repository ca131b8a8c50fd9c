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


def _figures(us=5.9, plan=None, cpu=True):
    """Raw figures of a run, as run_ours collects them, with long text
    fields so the size cap is tested near its worst case."""
    import bench
    from row_reduction_gb300.timing import algorithmic_bytes
    steps = 20
    f = {"op": "rmsnorm", "dtype": "f32", "rows": 1024, "cols": 4096,
         "steps": steps, "warmup": 5, "world": 1,
         "bytes": algorithmic_bytes("rmsnorm", 1024, 4096),
         "elapsed": us * 1e-6 * steps, "peak": 6783.1,
         "peak_kind": "measured",
         "plan": plan or bench.plan_text("rmsnorm", 1024, 4096),
         "traffic": 32590080, "rounds": [5.91, 5.93, 5.95, 5.97, 6.02],
         "floor": {"copy_us": 5.71, "copy_bytes": 2 * 4 * 1024 * 4096,
                   "empty_us": 1.31, "empty_wave_us": 1.52},
         "e2e_el": 108e-6 * 200, "e2e_steps": 200,
         "h2d": 16777216, "d2h": 16777216, "link_el": 101e-6 * 200,
         "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0,
                    "reasons": ["sw_power_cap"], "samples": 12},
         "pool_sets": 17, "pool_bytes": 17 * 33570816,
         "launches_per_step": 1, "cpu": None}
    if cpu:
        f["cpu"] = {"value": 41.234567, "unit": "GB/s", "cores": 16,
                    "kind": "oracle",
                    "sample": "full 1024x4096 x123 in 5.0 s, 16 row blocks "
                              "on 16 threads",
                    "cpu": "Neoverse-V2 (a long model name, for the size)",
                    "us_per_op": 812.3,
                    "single_thread": {"value": 4.5, "unit": "GB/s"}}
    return f


HEADLINE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup",
                 "ms_per_step", "us_per_op", "higher_is_better", "scaling",
                 "vs_baseline", "dtype", "data", "config", "roofline",
                 "cpu_baseline", "e2e", "gpu_launches", "clocks",
                 "rounds_us", "floor")


def test_headline_fits_the_cap_and_carries_every_key():
    import bench
    line = bench.build_headline(_figures())
    text = bench.headline_json(line)
    assert len(text.encode()) <= bench.HEADLINE_MAX_BYTES
    back = json.loads(text)
    for key in HEADLINE_KEYS:
        assert key in back, key
    assert back["config"]["workload"].startswith("rmsnorm f32 1024x4096")
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in back["roofline"], key
    for key in ("value", "unit", "cores", "kind", "sample", "cpu"):
        assert key in back["cpu_baseline"], key
    for key in ("value", "unit", "h2d_bytes_per_step", "d2h_bytes_per_step",
                "us_per_step", "link_gbs", "frac"):
        assert key in back["e2e"], key
    for key in ("sm_mhz", "sm_max_mhz", "reasons"):
        assert key in back["clocks"], key
    assert back["value"] == pytest.approx(33570816 / 5.9e-6 / 1e9,
                                          rel=1e-5)
    assert back["roofline"]["frac"] == pytest.approx(
        back["roofline"]["achieved"] / 6783.1, rel=1e-5)
    assert back["floor"]["frac_of_copy"] == pytest.approx(5.71 / 5.9,
                                                          rel=1e-3)
    assert back["e2e"]["frac"] == pytest.approx(101 / 108, rel=1e-4)
    assert back["gpu_launches"] == 20


def test_headline_over_the_cap_is_refused():
    import bench
    line = bench.build_headline(_figures())
    line["sweep"] = [{"op": "rmsnorm", "us": 1.0}] * 100
    with pytest.raises(ValueError):
        bench.headline_json(line)


def test_headline_gives_up_optional_fields_before_failing(monkeypatch):
    import bench
    f = _figures(plan="path=staged W=512 V=4 chunks=8 rows_per_block=1 "
                      "threads=512 grid=auto cluster=16 pdl prefetch_next "
                      "whole_tiles")
    f["clocks"]["reasons"] = list(bench.ClockSampler.NAMES)
    line = bench.build_headline(f)
    full = bench.headline_json(line)
    assert json.loads(full) == json.loads(json.dumps(line))
    # A cap between the line with and without the first optional fields:
    # those go, in order, and the rest stays.
    n = len(full.encode())
    monkeypatch.setattr(bench, "HEADLINE_MAX_BYTES", n - 60)
    back = json.loads(bench.headline_json(line))
    assert "cpu" not in back["cpu_baseline"]
    assert "l2" not in back["config"]
    assert "rounds_us" in back and "floor" in back
    # The smallest cap the line can meet: every optional field gone, every
    # key the metric needs kept.
    monkeypatch.setattr(bench, "HEADLINE_MAX_BYTES", 1170)
    back = json.loads(bench.headline_json(line))
    for path in bench.HEADLINE_OPTIONAL:
        node = back
        for key in path[:-1]:
            node = node[key]
        assert path[-1] not in node, path
    for key in ("value", "roofline", "cpu_baseline", "e2e", "clocks",
                "gpu_launches", "config"):
        assert key in back, key
    assert back["roofline"]["traffic"] == f["traffic"]
    assert back["e2e"]["h2d_bytes_per_step"] == f["h2d"]
    assert line["config"]["l2"]            # the caller's line is untouched


def test_headline_is_the_last_stdout_line(capsys):
    import bench
    print('{"op": "rmsnorm", "a sweep row": 1}')
    print("a table row", file=sys.stderr)
    bench.emit_headline(bench.build_headline(_figures(cpu=False)))
    out = capsys.readouterr().out.splitlines()
    last = json.loads(out[-1])
    assert last["metric"] == bench.METRIC and "cpu_baseline" not in last


def test_verify_accepts_a_consistent_line_and_flags_the_rest():
    import bench
    assert bench.verify_line(bench.build_headline(_figures())) == []
    bad = bench.build_headline(_figures())
    bad["value"] *= 1.01
    bad["rounds_us"]["median"] = 9.0
    bad["e2e"]["frac"] *= 1.1
    problems = bench.verify_line(bad)
    assert any(p.startswith("value") for p in problems)
    assert any(p.startswith("rounds_us") for p in problems)
    assert any(p.startswith("e2e.frac") for p in problems)
    assert bench.verify_line(bench.build_headline(
        _figures(plan="path=loop W=1")))[0].startswith("plan")


def test_sweep_covers_every_operator_and_the_loss_only_call():
    import bench
    from row_reduction_gb300 import inputs
    cases = bench.sweep_cases()
    for dt in ("f32", "bf16", "f16"):
        ops = {c[0] for c in cases if c[4] == dt}
        assert ops == set(inputs.ALL_OPS), dt
        assert ("cross_entropy", 1024, 4096, False, dt, False) in cases
