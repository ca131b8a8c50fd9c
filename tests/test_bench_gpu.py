"""GPU checks of the benchmark's own machinery: the measurement aids (the
library's copy and empty kernels) do what their header says, and bench.py's
last stdout line is a complete, self-consistent headline."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import row_reduction_gb300 as mt
from gpu_util import Guarded

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    from row_reduction_gb300 import build
    build.build()


@pytest.mark.parametrize("nbytes", [16, 4096, 16 * 1000 + 16, 33554432])
@pytest.mark.parametrize("threads,unroll,grid,flags", [
    (512, 4, 0, 0), (256, 8, 0, 1), (1024, 2, 0, 0), (32, 1, 1, 1),
    (128, 8, 3, 0), (128, 4, 1024, 1), (64, 2, 5000, 1)])
def test_probe_copy_is_an_exact_copy(nbytes, threads, unroll, grid, flags):
    n = nbytes // 4
    rng = np.random.default_rng(nbytes + threads)
    src_host = rng.integers(-2**31, 2**31 - 1, n, dtype=np.int64).astype(
        np.int32)
    src = Guarded(n, 0, -7, torch.int32, src_host)
    dst = Guarded(n, 0, Guarded.SENTINEL)
    assert src.ptr % 16 == 0 and dst.ptr % 16 == 0
    rc = mt.lib().mt_probe_copy(src.ptr, dst.ptr, nbytes, threads, unroll,
                                grid, flags,
                                torch.cuda.current_stream().cuda_stream)
    assert rc == mt.MT_OK
    torch.cuda.synchronize()
    dst.check()
    got = dst.view.view(torch.int32).cpu().numpy()
    assert np.array_equal(got, src_host)


@pytest.mark.parametrize("nbytes", [16, 16 * 1000 + 16, 33554432])
@pytest.mark.parametrize("threads,unroll,grid,flags", [
    (512, 4, 0, 0), (256, 8, 0, 1), (32, 1, 1, 0), (128, 4, 1024, 1),
    (64, 2, 5000, 1)])
def test_probe_read_writes_each_slices_xor(nbytes, threads, unroll, grid,
                                           flags):
    n = nbytes // 4
    rng = np.random.default_rng(nbytes + threads + 1)
    src_host = rng.integers(0, 2**32, n, dtype=np.uint64).astype(np.uint32)
    src = Guarded(n, 0, -7, torch.int32, src_host.view(np.int32))
    words = 152 * 64
    dst = Guarded(words, 0, -7, torch.int32, np.zeros(words, np.int32))
    rc = mt.lib().mt_probe_read(src.ptr, nbytes, dst.ptr, words, threads,
                                unroll, grid, flags,
                                torch.cuda.current_stream().cuda_stream)
    assert rc == mt.MT_OK
    torch.cuda.synchronize()
    dst.check()
    got = dst.view.cpu().numpy().view(np.uint32)
    # XOR is associative: the CTAs' words together give the whole buffer's
    assert np.bitwise_xor.reduce(got) == np.bitwise_xor.reduce(src_host)
    if grid > 0:
        # CTA b read the 16-byte words [b*per, (b+1)*per); the rest of dst
        # is untouched
        nw = nbytes // 16
        per = -(-nw // grid)
        for b in range(grid):
            lo, hi = b * per * 4, min(nw, (b + 1) * per) * 4
            want = np.bitwise_xor.reduce(src_host[lo:hi]) if lo < hi else 0
            assert got[b] == want, b
        assert not got[grid:].any()


def test_probe_empty_chain_runs():
    s = torch.cuda.current_stream().cuda_stream
    for threads, grid in ((32, 1), (512, 0), (1024, 300)):
        for _ in range(10):
            assert mt.lib().mt_probe_empty(threads, grid, s) == mt.MT_OK
    torch.cuda.synchronize()


def test_bench_headline_is_the_last_line_and_consistent():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "20",
         "--warmup", "5", "--no-sweep", "--cpu-seconds", "1"],
        cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    last = out.stdout.strip().splitlines()[-1]
    import bench
    assert len(last.encode()) <= bench.HEADLINE_MAX_BYTES
    line = json.loads(last)
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup",
                "ms_per_step", "us_per_op", "roofline", "cpu_baseline",
                "e2e", "clocks", "gpu_launches", "rounds_us", "floor"):
        assert key in line, key
    assert line["steps"] == 20 and line["gpu_launches"] == 20
    assert line["value"] > 0 and line["e2e"]["value"] > 0
    assert 0 < line["e2e"]["frac"] <= 1.2
    assert line["floor"]["copy_us"] > 0 and line["floor"]["empty_us"] > 0
    assert line["clocks"]["samples"] >= 1
    assert bench.verify_line(line) == []
