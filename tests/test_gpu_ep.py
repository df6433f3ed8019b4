"""Expert parallelism with the libmoe device steps, on the one GPU a box has: a
single-rank NCCL group (the all-to-alls are identities, the device work is the
real pack / receive metadata / expert path / combine). Multi-rank exchange logic
is covered on CPU ranks in test_ep_gloo.py."""
import socket

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close_y, read_metadata
from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300.workloads import MoEConfig, generate

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def group():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()
    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    yield None
    dist.destroy_process_group()


def test_dispatch_rows_and_combine_rows(group):
    cfg = MoEConfig("case", T=200, H=256, I=128, E=8, k=3)
    inp = generate(cfg, seed=1, device=DEV)
    g = torch.Generator().manual_seed(3)
    idx = torch.randint(0, cfg.E, (cfg.T, cfg.k), generator=g, dtype=torch.int32)
    idx[4, 1] = -1
    w = torch.rand((cfg.T, cfg.k), generator=g)
    idx, w = idx.to(DEV), w.to(DEV)
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    ws = B.new_workspace(shp)
    B.moe_routing_metadata(idx, shp, ws)
    rows = torch.zeros((cfg.R, cfg.H), dtype=torch.bfloat16, device=DEV)
    row_w = torch.zeros((cfg.R,), dtype=torch.float32, device=DEV)
    B.moe_dispatch_rows(inp["x"], shp, rows, ws, topk_w=w, row_weight=row_w)
    md = oracle.routing_metadata(idx.cpu(), cfg.E)
    n = len(md.perm_slot)
    perm = torch.as_tensor(md.perm_slot, dtype=torch.long)
    assert torch.equal(rows[:n].cpu(), inp["x"].cpu()[perm // cfg.k])
    assert torch.equal(row_w[:n].cpu(), w.cpu().reshape(-1)[perm])
    # combine: the sum of each token's rows (here the gathered x rows themselves)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    B.moe_combine_rows(rows, shp, y, ws)
    ref = np.zeros((cfg.T, cfg.H))
    xr = inp["x"].cpu().double().numpy()
    for s_, r in enumerate(md.row_of):
        if r >= 0:
            ref[s_ // cfg.k] += xr[s_ // cfg.k]
    assert_close_y(y, ref, "combine_rows")


@pytest.mark.parametrize("n_ranks,capacity", [(1, None), (4, 90)])
def test_ep_pack_places_rows_by_rank(group, n_ranks, capacity):
    """moe_ep_pack alone, for a P-rank layout on one device: block q holds the routed
    rows of rank q's experts from place 0 (bit-exact x rows and weights), the counts
    of the rows that fit; with a small capacity the overflow flags the error word."""
    cfg = MoEConfig("case", T=120, H=128, I=64, E=8, k=3)
    inp = generate(cfg, seed=6, device=DEV)
    g = torch.Generator().manual_seed(7)
    p = torch.tensor([8.0, 1, 1, 1, 1, 1, 1, 1])          # expert 0 popular: its block overflows
    idx = torch.multinomial(p / p.sum(), cfg.T * cfg.k, replacement=True, generator=g).to(torch.int32)
    idx = idx.view(cfg.T, cfg.k).to(DEV)
    w = torch.rand((cfg.T, cfg.k), generator=g).to(DEV)
    P = n_ranks
    C = capacity or cfg.T * cfg.k
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    ws = B.new_workspace(shp)
    B.moe_routing_metadata(idx, shp, ws)
    send = torch.zeros((P * C, cfg.H), dtype=torch.bfloat16, device=DEV)
    send_w = torch.zeros((P * C,), dtype=torch.float32, device=DEV)
    send_c = torch.zeros((P, cfg.E // P), dtype=torch.int32, device=DEV)
    B.moe_ep_pack(inp["x"], w, shp, P, C, send, send_w, send_c, ws)
    md = oracle.routing_metadata(idx.cpu(), cfg.E)
    E_loc = cfg.E // P
    want_c = np.zeros(cfg.E, np.int64)
    overflow = False
    xs, ws_ = inp["x"].cpu(), w.cpu().reshape(-1)
    for r, slot in enumerate(md.perm_slot.tolist()):
        e = int(np.searchsorted(md.offsets, r, side="right")) - 1
        q = e // E_loc
        pos = r - int(md.offsets[q * E_loc])
        if pos >= C:
            overflow = True
            continue
        want_c[e] += 1
        assert torch.equal(send[q * C + pos].cpu(), xs[slot // cfg.k])
        assert send_w[q * C + pos].item() == ws_[slot].item()
    np.testing.assert_array_equal(send_c.cpu().numpy().reshape(-1), want_c)
    err = B.moe_get_device_error(ws)
    assert bool(err & B.DEVERR_CAPACITY) == overflow
    assert overflow == (capacity is not None)


def test_ep_receive_metadata_matches_routing_metadata(group):
    """The receiver's metadata from the counts alone equals moe_routing_metadata of
    the received rows' local experts (padding slots dropped)."""
    P, C, E_loc = 3, 40, 5
    g = torch.Generator().manual_seed(11)
    recv = torch.zeros((P, E_loc), dtype=torch.int32)
    for p in range(P):
        n = int(torch.randint(0, C + 1, (1,), generator=g))
        cuts = torch.sort(torch.randint(0, n + 1, (E_loc - 1,), generator=g)).values
        recv[p] = torch.diff(torch.cat([torch.tensor([0]), cuts, torch.tensor([n])])).to(torch.int32)
    rshp = B.shape(P * C, 128, 64, E_loc, 1)
    rws = B.new_workspace(rshp)
    B.moe_ep_receive_metadata(recv.to(DEV), P, C, rshp, rws)
    counts, offsets, mt, perm, row_of = read_metadata(rws, rshp)
    idx = torch.full((P * C, 1), -1, dtype=torch.int32)
    for p in range(P):
        experts = np.repeat(np.arange(E_loc, dtype=np.int32), recv[p].numpy())
        idx[p * C:p * C + len(experts), 0] = torch.as_tensor(experts)
    ref = oracle.routing_metadata(idx, E_loc)
    np.testing.assert_array_equal(counts, ref.counts)
    np.testing.assert_array_equal(offsets, ref.offsets)
    np.testing.assert_array_equal(perm, ref.perm_slot)
    np.testing.assert_array_equal(row_of, ref.row_of)
    np.testing.assert_array_equal(mt, np.concatenate([[0], np.cumsum((ref.counts + 255) // 256)]))
    assert B.moe_get_device_error(rws) == 0


def test_expert_parallel_one_rank_equals_single_device_without_host_sync(group):
    from moe_expert_router_gb300.ep import ExpertParallel
    cfg = MoEConfig("case", T=300, H=384, I=256, E=8, k=2)
    inp = generate(cfg, seed=2, device=DEV)
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    ws = B.new_workspace(shp)
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
    B.moe_router(inp["x"], inp["w_r"], shp, B.router_cfg(), idx, w, ws)
    y_direct = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    B.moe_forward(inp["x"], idx, w, inp["w1"], inp["w2"], shp, y_direct, ws)
    ep = ExpertParallel(cfg.E, cfg.T, cfg.H, cfg.I, cfg.k, device=DEV)
    ep.forward(inp["x"], idx, w, inp["w1"], inp["w2"])          # first call: per-device set-up
    torch.cuda.synchronize()
    torch.cuda.set_sync_debug_mode("error")                     # any host sync in a forward raises
    try:
        y_ep = ep.forward(inp["x"], idx, w, inp["w1"], inp["w2"])
    finally:
        torch.cuda.set_sync_debug_mode("default")
    torch.cuda.synchronize()
    assert ep.ops.device_errors() == 0
    ref = oracle.expert_forward(inp["x"].cpu(), idx.cpu(), w.cpu().double(), inp["w1"].cpu(), inp["w2"].cpu())
    assert_close_y(y_ep, ref, "y (expert parallel, one rank)")
    assert_close_y(y_ep, y_direct.float().cpu().double().numpy(), "y (expert parallel vs direct)")
