"""The expert-parallel exchange of fp8_gemm_sigmoid_b300.ep on CPU: gloo ranks route their own
tokens, send each row to the rank owning its expert (counts first, then the rows), a stand-in
for the expert FFN multiplies each row by (global expert id + 1), and the reverse exchange
must bring every (token, slot) its own row times its own expert's factor, in the order of the
sender's permutation (DeepSeek-V3 co-design teardown §2.3 dispatch / combine skeleton)."""
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _routing(rank, T, E, K):
    rng = np.random.default_rng(100 + rank)
    p = rng.dirichlet(np.full(E, 0.5))
    return np.stack([rng.choice(E, K, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _rank(rank, world, port, E, K, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from fp8_gemm_sigmoid_b300 import ep
        T = 29 + 17 * rank                       # ranks hold different numbers of tokens
        idx = _routing(rank, T, E, K)
        if rank == 0:
            idx[:, 0] = 0                        # one hot expert on rank 0's side
        feats = (np.arange(T, dtype=np.float32)[:, None] * 10 + rank * 1000
                 + np.arange(4, dtype=np.float32)[None, :])
        perm = oracle.permute(idx, E, 0)         # the sender's permutation (expert-major)
        counts = perm["counts"]
        splits = ep.send_splits(counts, world)
        V = int(counts.sum())
        send = torch.from_numpy(feats[perm["perm_tok"][:V]])
        recv_counts = ep.exchange_counts(torch.from_numpy(counts.copy()), world).numpy()
        rsplits = [int(v) for v in recv_counts.sum(1)]
        recv = ep.exchange_rows(send, splits, rsplits)
        ids = ep.recv_expert_ids(recv_counts)
        epr = ep.experts_per_rank(E, world)
        # the receiving rank regroups by local expert (a one-slot permutation) and back
        lp = oracle.permute(ids[:, None], max(epr, 2), 0)
        grouped = recv.numpy()[lp["perm_tok"]]
        grouped *= (rank * epr + ids[lp["perm_tok"]] + 1).astype(np.float32)[:, None]
        back = ep.exchange_rows(torch.from_numpy(np.ascontiguousarray(grouped[lp["row_of"][:, 0]])), rsplits, splits)
        got = back.numpy()[perm["row_of"]]       # [T, K, 4]
        want = feats[:, None, :] * (idx[:, :, None] + 1).astype(np.float32)
        q.put((rank, bool(np.array_equal(got, want)), int(V), int(sum(rsplits))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world,E,K", [(2, 8, 2), (4, 8, 3), (3, 6, 1)])
def test_ep_exchange_round_trip(world, E, K):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 31500 + (os.getpid() + world * 7) % 1000
    procs = [ctx.Process(target=_rank, args=(r, world, port, E, K, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(world))
    assert all(ok for _, ok, _, _ in res)
    assert sum(v for _, _, v, _ in res) == sum(r for _, _, _, r in res)  # every row sent is received


def test_splits_and_receive_layout():
    from fp8_gemm_sigmoid_b300 import ep
    assert ep.send_splits([3, 0, 2, 5, 1, 1], 3) == [3, 7, 2]
    # source 0 sends 2 rows of local expert 0, source 1 one row of expert 0 and three of expert 1
    assert ep.recv_expert_ids(np.array([[2, 0], [1, 3]])).tolist() == [0, 0, 0, 1, 1, 1]
    with pytest.raises(ValueError):
        ep.experts_per_rank(10, 4)
