"""Seeded shape fuzz of the forward path against the oracle: routing (the router,
group limits, selection bias, both score functions, the few-token router below 257
tokens), the routing metadata and both stages, on randomly drawn small shapes —
K and N tails (H and I any multiple of 8), ragged expert counts, one to eight
experts per token — in bf16, and MXFP8 shapes (H and I multiples of 128); and the
backward (dX, dW1, dW2, the routing-weight and router gradients) on bf16 draws, the
MXFP8 training step on MXFP8 draws, and the router alone on wider draws (E up to
1024, k up to 32, T up to 2048, Zipf logit offsets), with the no-workspace router
bit-identical to it where its static scratch holds the same split-K factor and
within the oracle check's weight bound of it where the factor has to be lower.
Each draw is fixed by its seed. Bars as everywhere: routing sets bit-exact away
from near-ties, y and the gradients within the output bound."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (assert_close_y, check_router_against_oracle, oracle_router, oracle_y_for_tokens,
                         routing_mismatches, run_forward, run_router)
from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300.workloads import MoEConfig

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def draw_cfg(seed: int, mx: bool = False) -> MoEConfig:
    rng = np.random.default_rng(7000 + seed + (500 if mx else 0))
    k = int(rng.integers(1, 9))
    E = int(rng.integers(k, 65))
    if mx:
        H, I = 128 * int(rng.integers(1, 5)), 128 * int(rng.integers(1, 5))
    else:
        H, I = 8 * int(rng.integers(2, 81)), 8 * int(rng.integers(2, 81))
    T = int(rng.integers(1, 701))
    kw = {}
    if rng.random() < 0.5:
        kw.update(score="sigmoid", scale=2.5)
    groups = [g for g in (2, 4, 8) if E % g == 0]
    if groups and rng.random() < 0.5:
        ng = int(rng.choice(groups))
        gs = E // ng
        need = -(-k // gs)                                  # groups needed to hold k experts
        if need <= ng:
            tg = min(ng, need + int(rng.integers(0, 2)))
            kw.update(n_group=ng, topk_group=tg, group_topn=min(gs, int(rng.integers(1, 3))))
    if rng.random() < 0.5:
        kw["sel_bias"] = True
    return MoEConfig(f"fuzz{seed}", T=T, H=H, I=I, E=E, k=k, **kw)


def _routing(cfg, seed):
    from moe_expert_router_gb300.workloads import generate
    inp = generate(cfg, seed=seed, device=DEV)
    idx, w, _, ws = run_router(inp, cfg)
    ref = oracle_router(inp, cfg)
    n, bad, _ = routing_mismatches(idx, ref, cfg)
    assert not bad, f"{cfg}: {len(bad)} of {n} tokens routed differently, e.g. {bad[:5]}"
    return inp, idx, w, ws


@pytest.mark.parametrize("seed", range(48))
def test_fuzz_forward_bf16(seed):
    cfg = draw_cfg(seed)
    inp, idx, w, ws = _routing(cfg, seed)
    y, ws, _ = run_forward(inp, idx, w, cfg, ws=ws, staged=bool(seed % 2))
    assert B.moe_get_device_error(ws) == 0
    y_ref = oracle_y_for_tokens(inp, idx, w, list(range(cfg.T)))
    assert_close_y(y, y_ref, what=f"y ({cfg})")


@pytest.mark.parametrize("seed", range(24))
def test_fuzz_forward_mxfp8(seed):
    from test_gpu_mx import mx_inputs, oracle_weights, run_mx
    cfg = draw_cfg(seed, mx=True)
    inp, idx, w, ws = _routing(cfg, seed)
    inp, idx, w, w1q, w1s, w2q, w2s = mx_inputs(cfg, seed=seed, idx=idx, w=w)
    y, _, _, _, _, err = run_mx(cfg, inp, idx, w, w1q, w1s, w2q, w2s, staged=bool(seed % 2))
    assert err == 0
    xq, xs = oracle.mx_quantize(inp["x"])
    o1q, o1s, o2q, o2s = oracle_weights(inp, cfg)
    y_ref = oracle.expert_forward_mx(xq, xs, idx.cpu(), w.cpu().double(), o1q, o1s, o2q, o2s)
    assert_close_y(y, y_ref, what=f"y MXFP8 ({cfg})")


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_backward_bf16(seed):
    from dataclasses import replace
    from test_gpu_backward import _inputs, check_all, oracle_grads, train_step
    cfg = draw_cfg(100 + seed)
    cfg = replace(cfg, T=min(cfg.T, 400), backward=True)
    inp = _inputs(cfg, seed=seed)
    out = train_step(inp, cfg, staged=bool(seed % 2))
    ref = oracle_grads(inp, cfg, out["idx"], out["w"])
    check_all(out, ref)


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_training_mxfp8(seed):
    from dataclasses import replace
    from test_gpu_mx import check_mx_training
    cfg = draw_cfg(200 + seed, mx=True)
    check_mx_training(replace(cfg, T=min(cfg.T, 400), backward=True), seed=seed)


def draw_router_cfg(seed: int) -> MoEConfig:
    rng = np.random.default_rng(9000 + seed)
    k = int(rng.integers(1, 33))
    E = int(rng.integers(max(k, 2), 1025))
    H = 8 * int(rng.integers(2, 129))
    T = int(rng.integers(1, 2049))
    kw = {}
    if rng.random() < 0.5:
        kw.update(score="sigmoid", scale=2.5)
    groups = [g for g in (2, 4, 8, 16, 32) if E % g == 0]
    if groups and rng.random() < 0.5:
        ng = int(rng.choice(groups))
        gs = E // ng
        need = -(-k // gs)
        if need <= ng:
            tg = min(ng, need + int(rng.integers(0, 2)))
            kw.update(n_group=ng, topk_group=tg, group_topn=min(gs, int(rng.integers(1, 3))))
    if rng.random() < 0.4:
        kw["sel_bias"] = True
    if rng.random() < 0.3:
        kw["zipf_s"] = 1.2
    return MoEConfig(f"router_fuzz{seed}", T=T, H=H, I=8, E=E, k=k, **kw)


@pytest.mark.parametrize("seed", range(32))
def test_fuzz_router(seed):
    from gpu_helpers import router_cfg_of
    from moe_expert_router_gb300.workloads import generate
    cfg = draw_router_cfg(seed)
    inp = generate(cfg, seed=seed, device=DEV)
    idx, w, aux, _ = check_router_against_oracle(inp, cfg, require_order=False)
    if cfg.T * cfg.E <= 1 << 20 and cfg.E * cfg.H <= 1 << 20:
        shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
        idx2 = torch.empty_like(idx)
        w2 = torch.empty_like(w)
        aux2 = torch.zeros_like(aux)
        B.moe_router_noalloc(inp["x"], inp["w_r"], shp, router_cfg_of(cfg), idx2, w2, aux=aux2,
                             logit_offset=inp.get("logit_offset"), sel_bias=inp.get("sel_bias"))
        assert B.moe_router_noalloc_get_error() == 0
        # the aux score is a sum of float atomics, whose order varies from call to call
        torch.testing.assert_close(aux2, aux, rtol=1e-4, atol=0.0)
        if cfg.T * cfg.E * 32 <= 1 << 20:
            # the static scratch holds the partials of any split factor (at most 32):
            # the same split-K as the workspace router, so the same bits
            assert torch.equal(idx2, idx) and torch.equal(w2, w)
        else:
            # a lower split factor sums the fp32 logits in another order: the routing
            # away from near-ties, the weights to the bound of the oracle check
            n, bad, _ = routing_mismatches(idx2, oracle_router(inp, cfg), cfg)
            assert not bad, f"{len(bad)} of {n} tokens routed differently, e.g. {bad[:5]}"
            same = (idx2 == idx).all(1)
            torch.testing.assert_close(w2[same], w[same], rtol=1e-4, atol=1e-6)
