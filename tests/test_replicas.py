"""The N > 1 host logic of the bench on CPU: two ranks over gloo, each a replica
that times its own reads; the job's time is the slowest rank's and the job's
units are all ranks' units."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q) -> None:
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [40.0, 55.0][rank]                  # rank 1 is the slow one
        ms = bench.reduce_max(local_ms, world, "cpu")
        q.put((rank, ms, bench.us_per_unit(ms, 1000, world)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_over_all_reads():
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
    for rank, ms, us in got:
        assert ms == 55.0                              # both ranks see the max
        assert us == pytest.approx(1e3 * 55.0 / 2000)  # 2 ranks x 1000 reads


def test_single_rank_is_its_own_time():
    assert bench.reduce_max(12.5, 1) == 12.5
    assert bench.us_per_unit(12.5, 100, 1) == pytest.approx(125.0)
