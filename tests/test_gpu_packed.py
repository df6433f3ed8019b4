"""Tile-packed forward weights (moe_pack_weights) through the C ABI.

Bars: the packed bytes bit-exact against a re-layout written here with torch
indexing (a pure permutation plus zero padding); the forward with packed
weights bit-identical to the forward with the row-major weights (the same
operand values reach the same MMAs in the same order), and within the parity
bars of the oracle.
"""
import pytest
import torch

import oracle
from gpu_helpers import assert_close_y
from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300.workloads import CONFIGS, MoEConfig, generate

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def _swizzle_rows(tiles):
    """[..., 256, 64] bf16 tile rows -> the 128-byte-swizzled image: 16-byte chunk c of
    row r stored at chunk slot c ^ (r % 8)."""
    *lead, rows, cols = tiles.shape
    chunks = tiles.reshape(*lead, rows, 8, 8)
    r = torch.arange(rows).view(rows, 1)
    slot = torch.arange(8).view(1, 8)
    src = slot ^ (r % 8)                       # the chunk that lands in each slot
    idx = src.view(*([1] * len(lead)), rows, 8, 1).expand(*lead, rows, 8, 8)
    return torch.gather(chunks, -2, idx).reshape(*lead, rows, cols)


def expected_w1p(w1, I, H):
    E = w1.shape[0]
    nt, kbn = -(-I // 128), -(-H // 64)
    out = torch.zeros((E, nt, kbn, 256, 64), dtype=w1.dtype)
    pad = torch.zeros((E, nt * 128, kbn * 64), dtype=w1.dtype)
    for half, lo in ((0, 0), (1, I)):
        pad.zero_()
        pad[:, :I, :H] = w1[:, lo:lo + I, :]
        t = pad.view(E, nt, 128, kbn, 64).permute(0, 1, 3, 2, 4)
        out[:, :, :, 128 * half:128 * half + 128, :] = t
    return _swizzle_rows(out).contiguous().view(torch.uint8).reshape(-1)


def expected_w2p(w2, H, I):
    E = w2.shape[0]
    nt, kbn = -(-H // 256), -(-I // 64)
    pad = torch.zeros((E, nt * 256, kbn * 64), dtype=w2.dtype)
    pad[:, :H, :I] = w2
    t = pad.view(E, nt, 256, kbn, 64).permute(0, 1, 3, 2, 4)
    return _swizzle_rows(t).contiguous().view(torch.uint8).reshape(-1)


CASES = {
    "aligned": MoEConfig("aligned", T=256, H=256, I=256, E=4, k=2),
    "ragged": MoEConfig("ragged", T=300, H=200, I=200, E=6, k=3),        # I, H not tile multiples
    "narrow": MoEConfig("narrow", T=64, H=72, I=40, E=3, k=2),           # one partial tile each way
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_packed_layout_bit_exact(name):
    cfg = CASES[name]
    inp = generate(cfg, seed=3, device=DEV)
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, packed=True)
    w1p, w2p = B.moe_pack_weights(inp["w1"], inp["w2"], shp)
    torch.cuda.synchronize()
    assert torch.equal(w1p.cpu(), expected_w1p(inp["w1"].cpu(), cfg.I, cfg.H))
    assert torch.equal(w2p.cpu(), expected_w2p(inp["w2"].cpu(), cfg.H, cfg.I))


def _forward(cfg, inp, idx, w, w1, w2, packed, staged):
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, packed=packed)
    ws = B.new_workspace(shp, DEV)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    if staged:
        a = torch.empty((cfg.T * cfg.k, cfg.I), dtype=torch.bfloat16, device=DEV)
        B.moe_routing_metadata(idx, shp, ws)
        B.moe_dispatch_gemm1(inp["x"], w1, shp, a, ws)
        B.moe_swiglu_gemm2_combine(a, w, w2, shp, y, ws)
    else:
        B.moe_forward(inp["x"], idx, w, w1, w2, shp, y, ws)
    assert B.moe_get_device_error(ws) == 0
    return y


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("staged", [True, False])
def test_packed_forward_matches_row_major_and_oracle(name, staged):
    cfg = CASES[name]
    inp = generate(cfg, seed=4, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(5)
    idx = torch.stack([torch.randperm(cfg.E, generator=g)[:cfg.k] for _ in range(cfg.T)]).to(torch.int32)
    w = torch.rand((cfg.T, cfg.k), generator=g)
    w = (w / w.sum(1, keepdim=True)).to(DEV)
    idx = idx.to(DEV)
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, packed=True)
    w1p, w2p = B.moe_pack_weights(inp["w1"], inp["w2"], shp)
    y_row = _forward(cfg, inp, idx, w, inp["w1"], inp["w2"], packed=False, staged=staged)
    y_pk = _forward(cfg, inp, idx, w, w1p, w2p, packed=True, staged=staged)
    assert torch.equal(y_row, y_pk)
    y_ref = oracle.expert_forward(inp["x"].cpu(), idx.cpu(), w.cpu().double(), inp["w1"].cpu(), inp["w2"].cpu())
    assert_close_y(y_pk, y_ref, "y (packed weights)")


@pytest.mark.slow
def test_packed_forward_full_size_mid():
    """mid at full size: packed and row-major forwards bit-identical."""
    cfg = CONFIGS["mid"]
    inp = generate(cfg, seed=0, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(6)
    logits = torch.randn((cfg.T, cfg.E), generator=g)
    idx = logits.topk(cfg.k, dim=1).indices.to(torch.int32).to(DEV)
    w = torch.softmax(logits.topk(cfg.k, dim=1).values, dim=1).to(DEV)
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, packed=True)
    w1p, w2p = B.moe_pack_weights(inp["w1"], inp["w2"], shp)
    y_row = _forward(cfg, inp, idx, w, inp["w1"], inp["w2"], packed=False, staged=False)
    y_pk = _forward(cfg, inp, idx, w, w1p, w2p, packed=True, staged=False)
    assert torch.equal(y_row, y_pk)
