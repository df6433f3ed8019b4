"""Expert parallelism across ranks: the exchange logic on two and three CPU ranks
(gloo), with the oracle doing the per-rank device steps. Each rank's result must
equal the single-device oracle forward of its tokens over all experts."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from moe_expert_router_gb300.ep import local_expert_index, plan_splits


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(rank, T, H, I, E, k, skew):
    g = torch.Generator().manual_seed(100)           # weights: the same on every rank
    w1 = (torch.randn((E, 2 * I, H), generator=g) * H ** -0.5).to(torch.bfloat16)
    w2 = (torch.randn((E, H, I), generator=g) * I ** -0.5).to(torch.bfloat16)
    g = torch.Generator().manual_seed(200 + rank)    # tokens and routing: per rank
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    p = torch.arange(1, E + 1, dtype=torch.float64) ** -skew
    if T:
        idx = torch.multinomial(p / p.sum(), T * k, replacement=True, generator=g).to(torch.int32).view(T, k)
    else:
        idx = torch.zeros((0, k), dtype=torch.int32)
    if T > 3:
        idx[1, 0] = -1                                # a dropped slot
    w = torch.rand((T, k), generator=g, dtype=torch.float64)
    return x, idx, w, w1, w2


def _worker(rank, world, port, T_per_rank, E, skew, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import sys
    sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
    import torch.distributed as dist
    from ep_helpers import OracleOps
    from moe_expert_router_gb300.ep import ExpertParallel
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        H, I, k = 32, 16, 3
        T = T_per_rank[rank]
        x, idx, w, w1, w2 = _problem(rank, T, H, I, E, k, skew)
        ep = ExpertParallel(E, ops=OracleOps())
        lo, hi = rank * E // world, (rank + 1) * E // world
        y = ep.forward(x, idx, w, w1[lo:hi].contiguous(), w2[lo:hi].contiguous())
        ref = oracle.expert_forward(x, idx, w, w1, w2)
        assert tuple(y.shape) == (T, H)
        err = float(np.abs(y.numpy() - ref).max()) if T else 0.0
        q.put((rank, err, float(np.abs(ref).max()) if T else 0.0))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((rank, repr(e), None))


@pytest.mark.parametrize("world,T_per_rank,E,skew", [
    (2, [40, 25], 8, 0.0),
    (2, [64, 1], 8, 2.0),            # skewed: one rank receives far more rows
    (3, [30, 0, 17], 6, 1.0),        # a rank with no tokens
])
def test_expert_parallel_matches_single_device(world, T_per_rank, E, skew):
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, T_per_rank, E, skew, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    for rank, err, mx in res:
        assert mx is not None, f"rank {rank}: {err}"
        assert err <= 1e-12 * max(1.0, mx), (rank, err, mx)


def test_plan_splits_and_local_experts():
    counts = np.array([3, 0, 2, 5, 1, 4], np.int32)          # E = 6 over P = 3
    send, per = plan_splits(counts, 3)
    assert send.tolist() == [3, 7, 5]
    assert per.tolist() == [[3, 0], [2, 5], [1, 4]]
    # received from three sources, two local experts
    recv_per = np.array([[1, 2], [0, 0], [3, 1]])
    assert local_expert_index(recv_per).tolist() == [0, 1, 1, 0, 0, 0, 1]
    assert local_expert_index(np.zeros((2, 2), np.int64)).size == 0
