"""The multi-rank path of bench.py on CPU: two gloo ranks (world size 2) time different
amounts; the whole-job throughput takes every rank's tokens over the slowest rank's time, and
both ranks agree on it."""
import os

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_here = 100.0 if rank == 0 else 250.0  # rank 1 is the slow replica
        value, ms = bench.replica_throughput(1000, 10, ms_here, True)
        bench.barrier_sync(True)
        q.put((rank, value, ms))
    finally:
        dist.destroy_process_group()


def test_replica_throughput_uses_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for _, value, ms in res:
        assert ms == 250.0
        assert value == pytest.approx(2 * 1000 * 10 / 0.25)


def test_single_process_is_the_identity():
    import bench
    value, ms = bench.replica_throughput(1000, 10, 100.0, False)
    assert (value, ms) == (1000 * 10 / 0.1, 100.0)
