"""The multi-GPU form of the bench is replicas: every rank runs the same workload
and the job is timed by its slowest rank.  Its host logic (the max over ranks and
the whole-job rates) runs here on two gloo ranks on the CPU."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: decode 10 + r ms, prefill 30 - 5 r ms, step their sum
        dec, pre = 10.0 + rank, 30.0 - 5.0 * rank
        q.put((rank, bench.max_over_ranks([dec, pre, dec + pre], world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # each total is the max over the ranks, and every rank sees the same values
    assert got[0] == got[1] == [11.0, 30.0, 40.0]


def test_job_rates_scale_with_ranks():
    sys.path.insert(0, ROOT)
    import bench
    d1, p1 = bench.job_rates(45.0, 250.0, 1, 1000)
    d2, p2 = bench.job_rates(45.0, 250.0, 2, 1000)
    # 1000 steps of 268,435,456 state bytes in 45 ms; 1000 x 4000 tokens in 250 ms
    assert d1 == pytest.approx(1000 * 268435456 / 0.045 / 1e9)
    assert p1 == pytest.approx(1000 * 4000 / 0.25)
    # replicas: twice the work in the slowest rank's time
    assert d2 == pytest.approx(2 * d1) and p2 == pytest.approx(2 * p1)
    # a slower rank sets the job's time
    d_slow, _ = bench.job_rates(90.0, 250.0, 2, 1000)
    assert d_slow == pytest.approx(d1)
