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


def _bias_rank(rank, world, port, q):
    """One replica: route its share of a top-1 batch (oracle gate, FP32 tiny layer), then the
    global bias update through replicas.global_bias_update with the oracle's update rule as
    the update function (on a GPU that function is libmoe's moe_bias_update)."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import numpy as np
        import oracle
        from fp8_gemm_sigmoid_b300 import replicas, synthetic as sy
        cfg = sy.config("tiny_fp32", T=203, top_k=1, seed=11)
        inp = sy.make_inputs(cfg, "cpu", weights=False)
        x, Wg, bias = inp["x"].numpy(), inp["Wg"].numpy(), inp["bias"].numpy()
        a, b = replicas.token_range(cfg["T"], world, rank)
        g = oracle.gate(x[a:b], Wg, bias, cfg["n_group"], cfg["topk_group"], 1, cfg["routed_scaling_factor"])
        counts = torch.from_numpy(oracle.permute(g["topk_idx"], cfg["n_experts"], 0)["counts"].copy())
        b_t = torch.from_numpy(bias.copy())

        def update(c, T_global, cnt, bb):
            bb.copy_(torch.from_numpy(oracle.bias_update(cnt.numpy(), bb.numpy(), T_global, c["top_k"])))

        T_global = replicas.global_bias_update(cfg, counts, b - a, b_t, update)
        q.put((rank, T_global, counts.numpy().tolist(), b_t.numpy().tolist()))
    finally:
        dist.destroy_process_group()


def test_replicas_update_the_bias_from_the_global_histogram():
    import numpy as np
    import oracle
    from fp8_gemm_sigmoid_b300 import synthetic as sy
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 30500 + os.getpid() % 1000
    procs = [ctx.Process(target=_bias_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    # the whole batch routed in one process: its histogram and the oracle's update of it
    cfg = sy.config("tiny_fp32", T=203, top_k=1, seed=11)
    inp = sy.make_inputs(cfg, "cpu", weights=False)
    x, Wg, bias = inp["x"].numpy(), inp["Wg"].numpy(), inp["bias"].numpy()
    g = oracle.gate(x, Wg, bias, cfg["n_group"], cfg["topk_group"], 1, cfg["routed_scaling_factor"])
    counts = oracle.permute(g["topk_idx"], cfg["n_experts"], 0)["counts"]
    want = oracle.bias_update(counts, bias, cfg["T"], 1)
    for _, T_global, c, b in res:
        assert T_global == cfg["T"]
        assert c == counts.tolist()
        assert np.array_equal(np.array(b, np.float32), want)
    # a rank-local update would differ: the split matters
    a, b_ = 0, 102
    g0 = oracle.gate(x[a:b_], Wg, bias, cfg["n_group"], cfg["topk_group"], 1, cfg["routed_scaling_factor"])
    local = oracle.bias_update(oracle.permute(g0["topk_idx"], cfg["n_experts"], 0)["counts"], bias, b_ - a, 1)
    assert not np.array_equal(local, want)


def test_token_range_partitions_the_batch():
    from fp8_gemm_sigmoid_b300 import replicas
    for T in (0, 1, 7, 203, 16384):
        for world in (1, 2, 3, 8):
            spans = [replicas.token_range(T, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(spans[i][1] == spans[i + 1][0] for i in range(world - 1))
            sizes = [e - s for s, e in spans]
            assert max(sizes) - min(sizes) <= 1
