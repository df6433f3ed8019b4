"""Backward of the expert path and the router (CUDA path through the C ABI)
against the fp64 oracle's backward.

Bars (the same relative-error bounds as the forward outputs): dX, dW1, dW2,
dW_r and the routing-weight gradient within relative Frobenius error 1e-2 and
max abs error 3e-2 * max|ref|. Routing is taken from the GPU router (its
indices are checked against the oracle in the forward tests), so both sides
differentiate the same selection.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close_y, read_metadata, router_cfg_of, tile_sample_tokens
from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300.workloads import CONFIGS, MoEConfig, generate, routing_with_counts

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()   # raises when libmoe.so is missing: there is no fallback


def _cfg(T, H, I, E, k, **kw):
    return MoEConfig("case", T=T, H=H, I=I, E=E, k=k, backward=True, **kw)


def _inputs(cfg, seed=0):
    inp = generate(cfg, seed=seed, device=DEV)
    if inp["dy"] is None:
        g = torch.Generator(device=DEV).manual_seed(seed + 100)
        inp["dy"] = torch.randn((cfg.T, cfg.H), generator=g, device=DEV).to(torch.bfloat16)
    return inp


def train_step(inp, cfg, idx=None, w=None, staged=True, with_router=True):
    """Forward (saving h and the logits) and backward through the C ABI."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    shp = B.shape(T, H, I, E, k, training=True)
    ws = B.new_workspace(shp, DEV)
    rc = router_cfg_of(cfg)
    out = {"ws": ws, "shp": shp}
    logits = None
    if idx is None:
        idx = torch.empty((T, k), dtype=torch.int32, device=DEV)
        w = torch.empty((T, k), dtype=torch.float32, device=DEV)
        logits = torch.empty((T, E), dtype=torch.float32, device=DEV)
        B.moe_router_train(inp["x"], inp["w_r"], shp, rc, idx, w, logits, ws,
                           logit_offset=inp.get("logit_offset"), sel_bias=inp.get("sel_bias"))
    else:
        with_router = False
    a = torch.empty((T * k, I), dtype=torch.bfloat16, device=DEV)
    h = torch.empty((T * k, 2 * I), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    B.moe_routing_metadata(idx, shp, ws)
    B.moe_dispatch_gemm1_train(inp["x"], inp["w1"], shp, a, h, ws)
    B.moe_swiglu_gemm2_combine(a, w, inp["w2"], shp, y, ws)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    dw1 = torch.full((E, 2 * I, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    dw2 = torch.full((E, H, I), float("nan"), dtype=torch.bfloat16, device=DEV)
    dtw = torch.full((T, k), float("nan"), dtype=torch.float32, device=DEV)
    dwr = torch.full((E, H), float("nan"), dtype=torch.float32, device=DEV) if with_router else None
    w_r = inp["w_r"] if with_router else None
    if staged:
        B.moe_backward_stage2_data(inp["dy"], w, inp["w2"], h, shp, ws, dtopk_w=dtw)
        B.moe_backward_stage2_weight(inp["dy"], shp, dw2, ws)
        if with_router:
            B.moe_router_backward(inp["x"], logits, idx, w, dtw, shp, rc, dwr, ws)
        B.moe_backward_stage1_data(inp["w1"], shp, dx, ws, w_r=w_r, topk_idx=idx, cfg=rc)
        B.moe_backward_stage1_weight(inp["x"], shp, dw1, ws)
    else:
        B.moe_backward(inp["x"], idx, w, inp["w1"], inp["w2"], h, inp["dy"], shp, dx, dw1, dw2, ws,
                       w_r=w_r, logits=logits, cfg=rc, dw_r=dwr, dtopk_w=dtw)
    err = B.moe_get_device_error(ws)
    out.update(idx=idx, w=w, logits=logits, a=a, h=h, y=y, dx=dx, dw1=dw1, dw2=dw2, dtw=dtw, dwr=dwr,
               err=err)
    return out


def oracle_grads(inp, cfg, idx, w, with_router=True):
    cpu = {k_: (v.cpu() if isinstance(v, torch.Tensor) else v) for k_, v in inp.items()}
    wd = w.cpu().double()
    b = oracle.expert_backward(cpu["x"], idx.cpu(), wd, cpu["w1"], cpu["w2"], cpu["dy"])
    res = {"dx": b.dx, "dw1": b.dw1, "dw2": b.dw2, "dtw": b.dtopk_w}
    if with_router:
        rb = oracle.router_backward(cpu["x"], cpu["w_r"], idx.cpu(), wd, b.dtopk_w, score=cfg.score,
                                    normalize=cfg.normalize, scale=cfg.scale,
                                    logit_offset=cpu.get("logit_offset"))
        res["dx"] = res["dx"] + rb.dx_add
        res["dwr"] = rb.dw_r
        res["dlogits"] = rb.dlogits
    return res


def check_all(out, ref, with_router=True):
    assert out["err"] == 0, f"device error word {out['err']:#x}"
    assert_close_y(out["dtw"], ref["dtw"], "dtopk_w")
    assert_close_y(out["dw2"], ref["dw2"], "dW2")
    assert_close_y(out["dw1"], ref["dw1"], "dW1")
    assert_close_y(out["dx"], ref["dx"], "dX")
    if with_router:
        assert_close_y(out["dwr"], ref["dwr"], "dW_r")


CASES = {
    "tiny": CONFIGS["tiny"],
    "ragged_sigmoid_groups": _cfg(300, 192, 320, 16, 3, score="sigmoid", scale=2.5, n_group=4,
                                  topk_group=2, sel_bias=True),
    "two_units_per_expert": _cfg(1024, 512, 384, 4, 2),
    "softmax_plain": _cfg(200, 256, 128, 8, 3, normalize=False, scale=1.5),
    "sigmoid_plain": _cfg(200, 256, 128, 8, 3, score="sigmoid", normalize=False, scale=2.0),
    "zipf_offsets": _cfg(512, 256, 192, 32, 4, zipf_s=1.2),
    "h8_i8": _cfg(5, 8, 8, 3, 2),
    # top-1 with normalised weights: every weight is the constant scale, so the
    # router's gradients are exactly zero (the oracle's are)
    "top1_normalized_softmax": _cfg(150, 128, 128, 8, 1),
    "top1_normalized_sigmoid": _cfg(150, 128, 128, 8, 1, score="sigmoid", scale=2.5),
    "one_token": _cfg(1, 64, 64, 4, 2),
    # many experts and a large k: a wide router backward (E = 512), 16 slots per token
    "e512_k16_groups": _cfg(96, 128, 64, 512, 16, score="sigmoid", scale=2.5, n_group=16, topk_group=8,
                            sel_bias=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_backward_matches_oracle(name):
    cfg = CASES[name]
    inp = _inputs(cfg, seed=3)
    out = train_step(inp, cfg)
    ref = oracle_grads(inp, cfg, out["idx"], out["w"])
    check_all(out, ref)


def test_one_shot_equals_staged():
    cfg = CASES["ragged_sigmoid_groups"]
    inp = _inputs(cfg, seed=4)
    a = train_step(inp, cfg, staged=True)
    b = train_step(inp, cfg, staged=False)
    for key in ("dx", "dw1", "dw2", "dtw", "dwr"):
        assert torch.equal(a[key], b[key]), key


def test_saved_h_and_logits():
    cfg = CASES["ragged_sigmoid_groups"]
    inp = _inputs(cfg, seed=5)
    out = train_step(inp, cfg)
    # the stage-1 output a is unchanged by saving h, and h holds W1 x per routed row
    shp_plain = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
    ws = B.new_workspace(shp_plain, DEV)
    a_plain = torch.empty_like(out["a"])
    B.moe_routing_metadata(out["idx"], shp_plain, ws)
    B.moe_dispatch_gemm1(inp["x"], inp["w1"], shp_plain, a_plain, ws)
    R = int(out["idx"].numel())
    assert torch.equal(a_plain[:R], out["a"][:R])
    ref = oracle.routing_metadata(out["idx"].cpu(), cfg.E)
    x = inp["x"].cpu().double()
    h_ref = np.zeros((len(ref.perm_slot), 2 * cfg.I))
    for e in range(cfg.E):
        r0, r1 = int(ref.offsets[e]), int(ref.offsets[e + 1])
        tok = torch.as_tensor(ref.perm_slot[r0:r1] // cfg.k, dtype=torch.long)
        h_ref[r0:r1] = (x[tok] @ inp["w1"][e].cpu().double().T).numpy()
    assert_close_y(out["h"][: len(ref.perm_slot)], h_ref, "h")
    # logits: x W_r^T + offset in fp32
    l_ref = inp["x"].cpu().double() @ inp["w_r"].cpu().double().T
    assert_close_y(out["logits"], l_ref.numpy(), "logits")


def test_empty_experts_and_nan_poison():
    """Experts without rows get exactly zero weight gradients, whatever their weights hold."""
    T, H, I, E, k = 96, 128, 64, 8, 2
    cfg = _cfg(T, H, I, E, k)
    inp = _inputs(cfg, seed=6)
    counts = [40, 0, 60, 50, 0, 42, 0, 0]
    idx, w = routing_with_counts(counts, T, k, seed=2, device=DEV)
    for e, c in enumerate(counts):
        if c == 0:
            inp["w1"][e] = float("nan")
            inp["w2"][e] = float("nan")
    out = train_step(inp, cfg, idx=idx, w=w)
    for e, c in enumerate(counts):
        if c == 0:
            assert not out["dw1"][e].float().abs().max().item()
            assert not out["dw2"][e].float().abs().max().item()
    ref = oracle_grads(inp, cfg, idx, w, with_router=False)
    check_all(out, ref, with_router=False)


def test_dropped_slots_have_zero_weight_gradient():
    T, H, I, E, k = 64, 128, 64, 4, 2
    cfg = _cfg(T, H, I, E, k)
    inp = _inputs(cfg, seed=7)
    idx, w = routing_with_counts([32, 32, 32, 32], T, k, seed=3, device=DEV)
    idx[3, 1] = -1
    idx[10, 0] = E
    out = train_step(inp, cfg, idx=idx, w=w)
    assert out["err"] & B.DEVERR_BAD_EXPERT_INDEX
    out["err"] = 0
    assert out["dtw"][3, 1].item() == 0.0 and out["dtw"][10, 0].item() == 0.0
    ref = oracle_grads(inp, cfg, idx, w, with_router=False)
    check_all(out, ref, with_router=False)


def test_zero_tokens_zero_weight_gradients():
    T, H, I, E, k = 0, 64, 64, 4, 2
    shp = B.shape(T, H, I, E, k, training=True)
    ws = B.new_workspace(shp, DEV)
    dw1 = torch.full((E, 2 * I, H), 1.0, dtype=torch.bfloat16, device=DEV)
    dw2 = torch.full((E, H, I), 1.0, dtype=torch.bfloat16, device=DEV)
    dwr = torch.full((E, H), 1.0, dtype=torch.float32, device=DEV)
    empty = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    B.moe_backward_stage2_data(empty, None, None, None, shp, ws)
    B.moe_backward_stage2_weight(None, shp, dw2, ws)
    B.moe_router_backward(None, None, None, None, None, shp, B.router_cfg(), dwr, ws)
    B.moe_backward_stage1_data(None, shp, None, ws)
    B.moe_backward_stage1_weight(None, shp, dw1, ws)
    torch.cuda.synchronize()
    assert not dw1.float().abs().max().item() and not dw2.float().abs().max().item()
    assert not dwr.abs().max().item()


def weight_grad_experts(counts, n=8):
    """At least n experts (when there are that many) spanning the row-count
    regimes of the weight-gradient GEMMs, whose reduction runs over an expert's
    routed rows: the most and the least loaded expert with rows, and experts
    whose count leaves a last 256-row tile of at most 128 rows, of more than 128
    rows, no partial 64-row k-block, a partial one, and an expert without rows."""
    c = np.asarray(counts)
    live = np.nonzero(c > 0)[0]
    pick = [int(c.argmax()), int(live[np.argmin(c[live])])]
    regimes = [lambda v: 0 < v % 256 <= 128, lambda v: v % 256 > 128, lambda v: v > 0 and v % 64 == 0,
               lambda v: v % 64 != 0, lambda v: v == 0]
    for test in regimes:
        hit = [e for e in range(len(c)) if test(int(c[e])) and e not in pick]
        if hit:
            pick.append(hit[0])
    for e in np.linspace(0, len(c) - 1, num=len(c)).astype(int).tolist():
        if len(pick) >= n:
            break
        if e not in pick:
            pick.append(int(e))
    return pick


@pytest.mark.slow
def test_full_size_train_config_sampled():
    """The training configuration at full size, in the bench's staged launch
    sequence: dX and dtopk_w on the tokens of the first, middle and last rows of
    every 256-row tile of every expert (so every unit of the dA and dX GEMMs is
    reached), dW1 / dW2 of at least eight experts spanning the row-count regimes
    of the weight-gradient GEMMs, dW_r given the GPU's own routing-weight
    gradient."""
    cfg = CONFIGS["train"]
    inp = _inputs(cfg, seed=0)
    out = train_step(inp, cfg)
    assert out["err"] == 0
    idx, w = out["idx"], out["w"]
    T, k, E = cfg.T, cfg.k, cfg.E
    counts, offsets, _, perm, _ = read_metadata(out["ws"], out["shp"])
    toks = tile_sample_tokens(counts, offsets, perm, k, extra=[0, 1, T // 2, T - 1])
    cpu = {k_: (v.cpu() if isinstance(v, torch.Tensor) else v) for k_, v in inp.items()}
    tok_t = torch.as_tensor(toks)
    b = oracle.expert_backward(cpu["x"][tok_t], idx.cpu()[tok_t], w.cpu()[tok_t].double(), cpu["w1"],
                               cpu["w2"], cpu["dy"][tok_t], want_dw=False)
    assert_close_y(out["dtw"].cpu()[tok_t], b.dtopk_w, f"dtopk_w ({len(toks)} tokens)")
    # dX adds the router term, which needs the token's logit gradient: from the oracle's
    # router backward fed with the oracle's own routing-weight gradient of those tokens
    rb = oracle.router_backward(cpu["x"][tok_t], cpu["w_r"], idx.cpu()[tok_t], w.cpu()[tok_t].double(),
                                b.dtopk_w, score=cfg.score, normalize=cfg.normalize, scale=cfg.scale)
    assert_close_y(out["dx"].cpu()[tok_t], b.dx + rb.dx_add, f"dX ({len(toks)} tokens)")
    # weight gradients of experts in every row-count regime
    flat = idx.cpu().reshape(-1).long()
    for e in weight_grad_experts(counts):
        slots = torch.nonzero(flat == e).flatten()
        if len(slots) == 0:
            assert not out["dw1"][e].float().abs().max().item()
            assert not out["dw2"][e].float().abs().max().item()
            continue
        tk = slots // k
        one = torch.zeros((len(tk), 1), dtype=torch.int32)
        be = oracle.expert_backward(cpu["x"][tk], one, w.cpu().reshape(-1)[slots].double().unsqueeze(1),
                                    cpu["w1"][e:e + 1], cpu["w2"][e:e + 1], cpu["dy"][tk])
        assert_close_y(out["dw2"][e], be.dw2[0], f"dW2[{e}] ({len(slots)} rows)")
        assert_close_y(out["dw1"][e], be.dw1[0], f"dW1[{e}] ({len(slots)} rows)")
    # dW_r from the GPU's own routing-weight gradient (the router backward stage alone)
    rfull = oracle.router_backward(cpu["x"], cpu["w_r"], idx.cpu(), w.cpu().double(),
                                   out["dtw"].cpu().double(), score=cfg.score, normalize=cfg.normalize,
                                   scale=cfg.scale)
    assert_close_y(out["dwr"], rfull.dw_r, "dW_r")


def test_training_step_graph_capture_replays():
    """The training step is sync-free too: router, forward and the five backward calls
    captured in one CUDA graph and replayed give the eager results bit for bit (every
    reduction in them has a fixed order)."""
    cfg = _cfg(300, 256, 192, 8, 2)
    inp = _inputs(cfg, seed=5)
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    shp = B.shape(T, H, I, E, k, training=True)
    ws = B.new_workspace(shp, DEV)
    rc = router_cfg_of(cfg)
    o = {
        "idx": torch.empty((T, k), dtype=torch.int32, device=DEV),
        "w": torch.empty((T, k), dtype=torch.float32, device=DEV),
        "logits": torch.empty((T, E), dtype=torch.float32, device=DEV),
        "a": torch.empty((T * k, I), dtype=torch.bfloat16, device=DEV),
        "h": torch.empty((T * k, 2 * I), dtype=torch.bfloat16, device=DEV),
        "y": torch.empty((T, H), dtype=torch.bfloat16, device=DEV),
        "dx": torch.empty((T, H), dtype=torch.bfloat16, device=DEV),
        "dw1": torch.empty((E, 2 * I, H), dtype=torch.bfloat16, device=DEV),
        "dw2": torch.empty((E, H, I), dtype=torch.bfloat16, device=DEV),
        "dtw": torch.empty((T, k), dtype=torch.float32, device=DEV),
        "dwr": torch.empty((E, H), dtype=torch.float32, device=DEV),
    }

    def step():
        B.moe_router_train(inp["x"], inp["w_r"], shp, rc, o["idx"], o["w"], o["logits"], ws)
        B.moe_routing_metadata(o["idx"], shp, ws)
        B.moe_dispatch_gemm1_train(inp["x"], inp["w1"], shp, o["a"], o["h"], ws)
        B.moe_swiglu_gemm2_combine(o["a"], o["w"], inp["w2"], shp, o["y"], ws)
        B.moe_backward_stage2_data(inp["dy"], o["w"], inp["w2"], o["h"], shp, ws, dtopk_w=o["dtw"])
        B.moe_backward_stage2_weight(inp["dy"], shp, o["dw2"], ws)
        B.moe_router_backward(inp["x"], o["logits"], o["idx"], o["w"], o["dtw"], shp, rc, o["dwr"], ws)
        B.moe_backward_stage1_data(inp["w1"], shp, o["dx"], ws, w_r=inp["w_r"], topk_idx=o["idx"], cfg=rc)
        B.moe_backward_stage1_weight(inp["x"], shp, o["dw1"], ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):   # eager run first (per-device set-up happens outside capture)
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = {name: t.clone() for name, t in o.items()}
    for t in o.values():
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    graph.replay()
    torch.cuda.synchronize()
    for name, t in o.items():
        assert torch.equal(t.view(torch.uint8), eager[name].view(torch.uint8)), name
    assert B.moe_get_device_error(ws) == 0
