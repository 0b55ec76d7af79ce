"""The benchmark's multi-replica aggregation on CPU with gloo, world size 2.

The layer does not exchange data across GPUs (replicas only); what N > 1
needs is the timing protocol: a barrier on both sides of the timed region,
the maximum time over ranks, and whole-job throughput = all ranks' units /
that maximum. These run as two gloo processes on 127.0.0.1.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (world, rank, rank)
        dist.barrier()
        ms = bench.reduce_max(torch, 10.0 + 5.0 * rank, "cpu")  # rank 1 is the slow one
        dist.barrier()
        rate = bench.whole_job_rate(100.0, world, ms * 1e-3)
        q.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_replicas_take_max_time_and_sum_units():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [15.0, 15.0]
    assert all(abs(r[2] - 2 * 100.0 / 0.015) < 1e-6 for r in res)


def test_single_process_is_identity():
    import bench
    assert bench.reduce_max(torch, 3.5, "cpu") == 3.5
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
