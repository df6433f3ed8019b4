"""Expert parallelism across ranks: the exchange logic (fixed-size blocks, no
host-side split sizes) on two and three CPU ranks (gloo), with the oracle doing
the per-rank device steps. Each rank's result must equal the single-device
oracle forward of its tokens over all experts; with a capacity below T k, the
forward with the slots past a block's capacity dropped."""
import multiprocessing as mp
import os
import socket

import numpy as np
import pytest
import torch

import oracle


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


def _capacity_dropped(idx, E, world, C):
    """The routing with every slot whose routed row lies past its block's capacity
    dropped (-1): the block of rank q holds the routed rows of q's experts from place 0."""
    md = oracle.routing_metadata(idx, E)
    E_loc = E // world
    out = idx.clone().reshape(-1)
    for r, slot in enumerate(md.perm_slot.tolist()):
        e = int(np.searchsorted(md.offsets, r, side="right")) - 1
        q = e // E_loc
        if r - int(md.offsets[q * E_loc]) >= C:
            out[slot] = -1
    return out.view(idx.shape)


def _worker(rank, world, port, T_per_rank, E, skew, q, capacity=None):
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
        ep = ExpertParallel(E, T, H, I, k, ops=OracleOps(), capacity=capacity)
        lo, hi = rank * E // world, (rank + 1) * E // world
        y = ep.forward(x, idx, w, w1[lo:hi].contiguous(), w2[lo:hi].contiguous())
        kept = idx if capacity is None else _capacity_dropped(idx, E, world, ep.C)
        ref = oracle.expert_forward(x, kept, w, w1, w2)
        assert tuple(y.shape) == (T, H)
        err = float(np.abs(y.numpy() - ref).max()) if T else 0.0
        q.put((rank, err, float(np.abs(ref).max()) if T else 0.0))
        dist.destroy_process_group()
    except Exception as e:  # pragma: no cover - reported to the parent
        q.put((rank, repr(e), None))


@pytest.mark.parametrize("world,T_per_rank,E,skew,capacity", [
    (2, [40, 25], 8, 0.0, None),
    (2, [64, 1], 8, 2.0, None),            # skewed: one rank receives far more rows
    (3, [30, 0, 17], 6, 1.0, None),        # a rank with no tokens
    (2, [40, 40], 8, 2.0, 20),             # a capacity below T k: skewed blocks overflow and drop rows
])
def test_expert_parallel_matches_single_device(world, T_per_rank, E, skew, capacity):
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, T_per_rank, E, skew, q, capacity))
             for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in procs]
    for p in procs:
        p.join(timeout=60)
    for rank, err, mx in res:
        assert mx is not None, f"rank {rank}: {err}"
        assert err <= 1e-12 * max(1.0, mx), (rank, err, mx)
