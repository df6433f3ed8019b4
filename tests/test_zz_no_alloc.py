"""moe_router_noalloc against moe_router, through the C ABI.

moe_router_noalloc serves callers that may not allocate device memory -- a
plug-in inside a host runtime that owns every byte of device memory and gives
it no workspace. It keeps the router's scratch in a static array inside the
library instead of a caller-supplied workspace. This test checks that it gives
the same routing as the workspace-based entry point on two calls in a row (the
second call must not be disturbed by what the first left in the shared array),
and that it refuses shapes whose scratch does not fit that array. Its split-K
factor can be lower than the workspace router's (the array is smaller), which
changes the fp32 summation order of the logits, so tokens whose top-k choice
is a near-tie (oracle selection gap below 1e-6) are left out of the exact
routing comparison, as in the other router tests.

This file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300.workloads import MoEConfig, generate

pytestmark = pytest.mark.gpu

CASES = [
    MoEConfig("noalloc_softmax", T=4096, H=1024, I=64, E=64, k=6),
    MoEConfig("noalloc_groups", T=2048, H=512, I=64, E=256, k=8, score="sigmoid", scale=2.5,
              n_group=8, topk_group=4, group_topn=2, sel_bias=True),
    # decode-sized: the router's few-token path (logits on the CUDA cores)
    MoEConfig("noalloc_decode", T=64, H=4096, I=64, E=128, k=8, zipf_s=1.2),
]


def _cfg(c):
    return B.router_cfg(c.score, c.normalize, c.scale, c.n_group, c.topk_group, c.group_topn)


def _outputs(c):
    return (torch.empty((c.T, c.k), dtype=torch.int32, device="cuda"),
            torch.empty((c.T, c.k), dtype=torch.float32, device="cuda"),
            torch.zeros((1,), dtype=torch.float32, device="cuda"))


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def test_noalloc_router_matches_workspace_router_twice_in_a_row():
    results = []
    for c in CASES:                                   # two calls in a row, different shapes
        inp = generate(c, seed=21, device="cuda")
        shp = B.shape(c.T, c.H, c.I, c.E, c.k)
        idx_n, w_n, aux_n = _outputs(c)
        B.moe_router_noalloc(inp["x"], inp["w_r"], shp, _cfg(c), idx_n, w_n, aux=aux_n,
                             logit_offset=inp["logit_offset"], sel_bias=inp["sel_bias"])
        ws = B.new_workspace(shp)
        idx_r, w_r, aux_r = _outputs(c)
        B.moe_router(inp["x"], inp["w_r"], shp, _cfg(c), idx_r, w_r, ws, aux=aux_r,
                     logit_offset=inp["logit_offset"], sel_bias=inp["sel_bias"])
        torch.cuda.synchronize()
        results.append((c, idx_n.cpu(), w_n.cpu(), aux_n.cpu(), idx_r.cpu(), w_r.cpu(), aux_r.cpu()))
    for c, idx_n, w_n, aux_n, idx_r, w_r, aux_r in results:
        inp = generate(c, seed=21, device="cuda")
        ref = oracle.router(inp["x"], inp["w_r"], c.k, score=c.score, normalize=c.normalize,
                            scale=c.scale, n_group=c.n_group, topk_group=c.topk_group,
                            group_topn=c.group_topn, logit_offset=inp["logit_offset"],
                            sel_bias=inp["sel_bias"])
        keep = ref.sel_gap >= 1e-6
        if c.n_group > 1:
            keep &= ref.group_gap >= 1e-6
        keep = torch.from_numpy(keep)
        assert torch.equal(idx_n[keep], idx_r[keep]), c.name
        np.testing.assert_allclose(w_n[keep].numpy(), w_r[keep].numpy(), rtol=1e-4, atol=1e-6)
        np.testing.assert_allclose(aux_n.numpy(), aux_r.numpy(), rtol=1e-4)
    # the first case again: the array now holds the second case's scratch
    c = CASES[0]
    inp = generate(c, seed=21, device="cuda")
    shp = B.shape(c.T, c.H, c.I, c.E, c.k)
    idx_n, w_n, aux_n = _outputs(c)
    B.moe_router_noalloc(inp["x"], inp["w_r"], shp, _cfg(c), idx_n, w_n, aux=aux_n)
    torch.cuda.synchronize()
    assert torch.equal(idx_n.cpu(), results[0][1])     # same call, same result
    np.testing.assert_allclose(aux_n.cpu().numpy(), results[0][3].numpy(), rtol=1e-6)
    # no call above ran out of time in a pipeline wait: the static error word is clear
    assert B.moe_router_noalloc_get_error() == 0


def test_noalloc_router_at_the_weight_split_limit():
    """E * H == 2**20 exactly: the bf16 x3 split of w_r fills its region of the array."""
    c = MoEConfig("eh_limit", T=512, H=4096, I=64, E=256, k=8, score="sigmoid", scale=2.5,
                  n_group=8, topk_group=4, group_topn=2, sel_bias=True)
    inp = generate(c, seed=5, device="cuda")
    shp = B.shape(c.T, c.H, c.I, c.E, c.k)
    idx_n, w_n, aux_n = _outputs(c)
    B.moe_router_noalloc(inp["x"], inp["w_r"], shp, _cfg(c), idx_n, w_n, aux=aux_n,
                         sel_bias=inp["sel_bias"])
    ws = B.new_workspace(shp)
    idx_r, w_r, aux_r = _outputs(c)
    B.moe_router(inp["x"], inp["w_r"], shp, _cfg(c), idx_r, w_r, ws, aux=aux_r, sel_bias=inp["sel_bias"])
    torch.cuda.synchronize()
    ref = oracle.router(inp["x"], inp["w_r"], c.k, score=c.score, normalize=c.normalize, scale=c.scale,
                        n_group=c.n_group, topk_group=c.topk_group, group_topn=c.group_topn,
                        sel_bias=inp["sel_bias"])
    keep = torch.from_numpy((ref.sel_gap >= 1e-6) & (ref.group_gap >= 1e-6))
    assert torch.equal(idx_n.cpu()[keep], idx_r.cpu()[keep])
    np.testing.assert_allclose(w_n.cpu()[keep].numpy(), w_r.cpu()[keep].numpy(), rtol=1e-4, atol=1e-6)
    assert B.moe_router_noalloc_get_error() == 0


def test_noalloc_router_rejects_shapes_beyond_its_scratch():
    c = MoEConfig("too_big", T=8193, H=64, I=64, E=128, k=2)      # T * E > 2**20
    shp = B.shape(c.T, c.H, c.I, c.E, c.k)
    x = torch.zeros((c.T, c.H), dtype=torch.bfloat16, device="cuda")
    w_r = torch.zeros((c.E, c.H), dtype=torch.float32, device="cuda")
    idx, w, aux = _outputs(c)
    with pytest.raises(B.MoEError) as e:
        B.moe_router_noalloc(x, w_r, shp, _cfg(c), idx, w, aux=aux)
    assert e.value.status == 2   # MOE_ERR_UNSUPPORTED
    # E * H > 2**20: the bf16 x3 split of w_r would not fit its region
    c = MoEConfig("too_wide", T=64, H=4104, I=64, E=256, k=8)
    shp = B.shape(c.T, c.H, c.I, c.E, c.k)
    x = torch.zeros((c.T, c.H), dtype=torch.bfloat16, device="cuda")
    w_r = torch.zeros((c.E, c.H), dtype=torch.float32, device="cuda")
    idx, w, aux = _outputs(c)
    with pytest.raises(B.MoEError) as e:
        B.moe_router_noalloc(x, w_r, shp, _cfg(c), idx, w, aux=aux)
    assert e.value.status == 2
