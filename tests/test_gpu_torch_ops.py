"""The torch.library operators through torch.compile (whole graph, no break) against
the direct ctypes calls: bit-identical routing and y, the aux score to rounding."""
import pytest
import torch

from gpu_helpers import router_cfg_of
from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300 import torch_ops  # noqa: F401  (registers the operators)
from moe_expert_router_gb300.workloads import MoEConfig, generate

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def test_compiled_router_and_forward_equal_the_direct_calls():
    cfg = MoEConfig("case", T=300, H=256, I=384, E=16, k=4, score="sigmoid", scale=2.5, n_group=4, topk_group=2,
                    group_topn=2, sel_bias=True)
    inp = generate(cfg, seed=3, device="cuda")

    def layer(x, w_r, bias, w1, w2):
        idx, w, aux = torch.ops.moe_gb300.router(x, w_r, cfg.k, cfg.score, cfg.normalize, cfg.scale, cfg.n_group,
                                                 cfg.topk_group, cfg.group_topn, bias, None)
        return torch.ops.moe_gb300.forward(x, idx, w, w1, w2), idx, aux

    compiled = torch.compile(layer, fullgraph=True, backend="eager")
    y_c, idx_c, aux_c = compiled(inp["x"], inp["w_r"], inp["sel_bias"], inp["w1"], inp["w2"])

    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    ws = B.new_workspace(shp, "cuda")
    idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device="cuda")
    aux = torch.zeros((1,), dtype=torch.float32, device="cuda")
    B.moe_router(inp["x"], inp["w_r"], shp, router_cfg_of(cfg), idx, w, ws, aux=aux, sel_bias=inp["sel_bias"])
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device="cuda")
    B.moe_forward(inp["x"], idx, w, inp["w1"], inp["w2"], shp, y, ws)
    assert torch.equal(idx_c, idx)
    # the aux score's per-expert sums are accumulated with atomics: equal to rounding
    assert torch.allclose(aux_c, aux, rtol=1e-5, atol=0.0)
    assert torch.equal(y_c, y)


def _layer_grads(fn, inp):
    x = inp["x"].clone().requires_grad_(True)
    w_r = inp["w_r"].clone().requires_grad_(True)
    w1 = inp["w1"].clone().requires_grad_(True)
    w2 = inp["w2"].clone().requires_grad_(True)
    y, idx, w, _ = fn(x, w_r, w1, w2)
    y.backward(inp["dy"])
    return y.detach(), idx, w, x.grad, w_r.grad, w1.grad, w2.grad


def _layer_fn(cfg, inp):
    def fn(x, w_r, w1, w2):
        return torch_ops.moe_layer(x, w_r, w1, w2, cfg.k, cfg.score, cfg.normalize, cfg.scale, cfg.n_group,
                                   cfg.topk_group, cfg.group_topn, inp.get("sel_bias"), inp.get("logit_offset"))
    return fn


@pytest.mark.parametrize("case", ["ragged_sigmoid_groups", "zipf_offsets"])
def test_autograd_layer_equals_the_direct_training_calls(case):
    """moe_layer under autograd: y, the routing and every gradient (x with the router's
    term, w_r, w1, w2) bit-identical to the same training step through the C ABI, which
    the backward tests check against the oracle."""
    from test_gpu_backward import CASES, _inputs, train_step
    cfg = CASES[case]
    inp = _inputs(cfg, seed=5)
    y, idx, w, gx, gwr, g1, g2 = _layer_grads(_layer_fn(cfg, inp), inp)
    out = train_step(inp, cfg, staged=False)
    assert out["err"] == 0
    assert torch.equal(idx, out["idx"]) and torch.equal(w, out["w"]) and torch.equal(y, out["y"])
    assert torch.equal(gx, out["dx"]) and torch.equal(gwr, out["dwr"])
    assert torch.equal(g1, out["dw1"]) and torch.equal(g2, out["dw2"])


def test_compiled_autograd_layer_equals_eager():
    """moe_layer compiled with AOTAutograd (forward and backward graphs traced through the
    operators' shape functions, no graph break): the same y and gradients as eager."""
    from test_gpu_backward import CASES, _inputs
    cfg = CASES["ragged_sigmoid_groups"]
    inp = _inputs(cfg, seed=6)
    fn = _layer_fn(cfg, inp)
    eager = _layer_grads(fn, inp)
    compiled = _layer_grads(torch.compile(fn, fullgraph=True, backend="aot_eager"), inp)
    for a, b in zip(eager, compiled):
        assert torch.equal(a, b)


def test_autograd_mx_layer_equals_the_direct_training_calls():
    """moe_layer(precision="mxfp8") under autograd: y, the routing and every gradient
    bit-identical to the MXFP8 training step through the C ABI (router with logits,
    the MXFP8 forward, bf16 data gradients, MXFP8 weight gradients), whose parts the
    MXFP8 tests check against the oracle; the weight cache quantizes each weight once
    and again after an in-place update."""
    from test_gpu_backward import _inputs
    from moe_expert_router_gb300.mx_cache import MxWeightCache
    cfg = MoEConfig("case", T=300, H=256, I=384, E=16, k=4, score="sigmoid", scale=2.5, n_group=4, topk_group=2,
                    group_topn=2, sel_bias=True, backward=True)
    inp = _inputs(cfg, seed=8)
    cache = MxWeightCache()

    def fn(x, w_r, w1, w2):
        return torch_ops.moe_layer(x, w_r, w1, w2, cfg.k, cfg.score, cfg.normalize, cfg.scale, cfg.n_group,
                                   cfg.topk_group, cfg.group_topn, inp["sel_bias"], None, precision="mxfp8",
                                   weight_cache=cache)

    y, idx, w, gx, gwr, g1, g2 = _layer_grads(fn, inp)
    assert cache.quantizations == 2

    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    R = T * k
    shp = B.shape(T, H, I, E, k, training=True, mxfp8=True)
    ws = B.new_workspace(shp, "cuda")
    rc = router_cfg_of(cfg)
    idx_d = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w_d = torch.empty((T, k), dtype=torch.float32, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    B.moe_router_train(inp["x"], inp["w_r"], shp, rc, idx_d, w_d, logits, ws, sel_bias=inp["sel_bias"])
    w1c = torch.empty(inp["w1"].shape, dtype=torch.uint8, device="cuda")
    w1s = B.mx_scales_empty(inp["w1"].shape, "cuda")
    w2c = torch.empty(inp["w2"].shape, dtype=torch.uint8, device="cuda")
    w2s = B.mx_scales_empty(inp["w2"].shape, "cuda")
    B.moe_mx_quantize(inp["w1"], w1c, w1s)
    B.moe_mx_quantize(inp["w2"], w2c, w2s)
    aq = torch.empty((R, I), dtype=torch.uint8, device="cuda")
    as_ = B.mx_scales_empty((R, I), "cuda")
    h = torch.empty((R, 2 * I), dtype=torch.bfloat16, device="cuda")
    y_d = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    B.moe_routing_metadata(idx_d, shp, ws)
    B.moe_mx_quantize_dispatch(inp["x"], shp, ws)
    B.moe_dispatch_gemm1_mx_train(w1c, w1s, shp, aq, as_, h, ws)
    B.moe_swiglu_gemm2_combine_mx(aq, as_, w_d, w2c, w2s, shp, y_d, ws)
    dtw = torch.empty((T, k), dtype=torch.float32, device="cuda")
    dx = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    dwr = torch.empty((E, H), dtype=torch.float32, device="cuda")
    dw1 = torch.empty_like(inp["w1"])
    dw2 = torch.empty_like(inp["w2"])
    B.moe_backward_stage2_data(inp["dy"], w_d, inp["w2"], h, shp, ws, dtopk_w=dtw)
    B.moe_backward_stage2_weight_mx(inp["dy"], shp, dw2, ws)
    B.moe_router_backward(inp["x"], logits, idx_d, w_d, dtw, shp, rc, dwr, ws)
    B.moe_backward_stage1_data(inp["w1"], shp, dx, ws, w_r=inp["w_r"], topk_idx=idx_d, cfg=rc)
    B.moe_backward_stage1_weight_mx(inp["x"], shp, dw1, ws)
    assert B.moe_get_device_error(ws) == 0
    assert torch.equal(idx, idx_d) and torch.equal(w, w_d) and torch.equal(y, y_d)
    assert torch.equal(gx, dx) and torch.equal(gwr, dwr) and torch.equal(g1, dw1) and torch.equal(g2, dw2)

    # the same parameters again: cache hits; an in-place update of w1 moves its
    # version counter, and the next call quantizes w1 again
    cache2 = MxWeightCache()
    w1p = inp["w1"].clone().requires_grad_(True)
    w2p = inp["w2"].clone().requires_grad_(True)

    def call():
        return torch_ops.moe_layer(inp["x"], inp["w_r"], w1p, w2p, cfg.k, cfg.score, cfg.normalize, cfg.scale,
                                   cfg.n_group, cfg.topk_group, cfg.group_topn, inp["sel_bias"], None,
                                   precision="mxfp8", weight_cache=cache2)[0]

    y1 = call()
    assert cache2.quantizations == 2 and torch.equal(y1, y)
    call()
    assert cache2.quantizations == 2
    with torch.no_grad():
        w1p.mul_(0.5)
    y3 = call()
    assert cache2.quantizations == 3 and not torch.equal(y3, y)
