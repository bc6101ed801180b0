"""bench.py's multi-rank logic on CPU: two gloo ranks (replicas), the job's
step time is the slowest rank's and the throughput counts every rank's
units.  No GPU is involved."""
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


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = [1.5, 4.0][rank]
        ms = bench.max_over_ranks(ms_local, "cpu")
        q.put((rank, ms, bench.whole_job_rate(64, ms, world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_units():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate in got:
        assert ms == 4.0
        assert rate == pytest.approx(2 * 64 / 4.0e-3)


def test_single_process_is_its_own_job():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5, "cpu") == 2.5
    assert bench.whole_job_rate(64, 2.0, 1) == pytest.approx(32000.0)
