"""The N > 1 path of bench.py is replicas only: each rank runs the whole product,
the step time is the slowest rank's and the job's FLOPs are world x one
replica's. Checked with two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = [3.5, 4.25][rank]                      # the second replica is slower
        worst = bench.reduce_max(ms, dist, "cpu")
        out[rank] = (worst, bench.whole_job_tflops(world, 4.0e12, worst))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_step_and_sum_the_work():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        ps = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in ps:
            p.start()
        for p in ps:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0] == res[1]
    worst, value = res[0]
    assert worst == 4.25
    assert value == pytest.approx(2 * 4.0e12 / 4.25e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(2.0) == 2.0
    assert bench.whole_job_tflops(1, 1e12, 1.0) == pytest.approx(1.0e3)
