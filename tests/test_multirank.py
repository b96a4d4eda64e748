"""The N>1 bench path on CPU: two gloo ranks, the slowest rank's step time and the
whole-job rate (heads are independent, so ranks share no data-path collective)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.max_over_ranks(1.0 + 0.5 * rank)          # rank r took 1 + r/2 ms per step
        rate = bench.whole_job_rate(1000, world, ms)
        q.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_the_whole_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, rate in got:
        assert ms == pytest.approx(1.5)                       # both ranks see the slowest
        assert rate == pytest.approx(2 * 1000 / 1.5e-3)       # all ranks' units over that time


def test_single_process_values_pass_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.25) == 2.25
    assert bench.whole_job_rate(10, 1, 2.0) == pytest.approx(5000.0)
