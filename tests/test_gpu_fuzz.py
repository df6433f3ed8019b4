"""Seeded shape fuzz of the forward path against the oracle: routing (the router,
group limits, selection bias, both score functions, the few-token router below 257
tokens), the routing metadata and both stages, on randomly drawn small shapes —
K and N tails (H and I any multiple of 8), ragged expert counts, one to eight
experts per token — in bf16, and MXFP8 shapes (H and I multiples of 128); and the
backward (dX, dW1, dW2, the routing-weight and router gradients) on bf16 draws, and
the MXFP8 training step on MXFP8 draws. Each
draw is fixed by its seed. Bars as everywhere: routing sets bit-exact away from
near-ties, y and the gradients within the output bound."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close_y, oracle_router, oracle_y_for_tokens, routing_mismatches, run_forward, run_router
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
