"""The benchmark's replica path on CPU: two gloo ranks, each timing its own
replica, agree on the slowest rank's time, and the whole-job value counts
every rank's bytes.  (Rows are independent, so ranks exchange nothing but
this one timing scalar.)"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        elapsed = [0.25, 0.5][rank]
        m = bench.max_over_ranks(elapsed, "cpu")
        v = bench.job_value(1000, 10, m, world)
        out.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q))
             for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in res:
        assert m == 0.5
        assert v == pytest.approx(2 * 1000 * 10 / 0.5 / 1e9)


def test_reference_arm_other_ranks_exit_without_work():
    import argparse
    import bench
    args = argparse.Namespace(op="rmsnorm", rows=1024, cols=4096, steps=5,
                              warmup=3)
    assert bench.run_reference(args, rank=1, world=2) == 0
