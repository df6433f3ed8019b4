"""Expert parallelism with the libmoe device steps, on the one GPU a box has: a
single-rank NCCL group (the all-to-alls are identities, the device work is the
real dispatch rows / expert path / combine rows). Multi-rank exchange logic is
covered on CPU ranks in test_ep_gloo.py."""
import socket

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close_y
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


def test_expert_parallel_one_rank_equals_single_device(group):
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
    ep = ExpertParallel(cfg.E, device=DEV)
    y_ep = ep.forward(inp["x"], idx, w, inp["w1"], inp["w2"])
    torch.cuda.synchronize()
    ref = oracle.expert_forward(inp["x"].cpu(), idx.cpu(), w.cpu().double(), inp["w1"].cpu(), inp["w2"].cpu())
    assert_close_y(y_ep, ref, "y (expert parallel, one rank)")
    assert_close_y(y_ep, y_direct.float().cpu().double().numpy(), "y (expert parallel vs direct)")
