"""The bench's multi-rank path on CPU: two gloo ranks on 127.0.0.1.

On a GPU node each rank runs an independent replica of the workload (no data-path
collective); the only exchange is the timing, reduced to the slowest rank, and the
reported value counts every rank's tokens over that time.
"""
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
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [10.0, 25.0, 5.0, 7.5][rank]
        bench.barrier(world)
        ms = bench.max_over_ranks(local_ms, world)
        value = bench.job_throughput(64, world, 100, ms)
        q.put((rank, ms, value))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_timing_is_max_over_ranks_and_value_counts_all_ranks(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(world))
    slowest = max([10.0, 25.0, 5.0, 7.5][:world])
    for rank, ms, value in got:
        assert ms == slowest                                   # every rank sees the max
        assert value == pytest.approx(64 * world * 100 / (slowest / 1e3))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    bench.barrier(1)
    assert bench.job_throughput(64, 1, 10, 2.0) == pytest.approx(320000.0)
