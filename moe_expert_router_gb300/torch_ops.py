"""PyTorch custom operators over the C ABI, for callers that compile their model.

The guide's op is meant to sit inside a captured, compiled training step (MegaMoE
guide, section "Example 2 — single-node EP8 with full CUDA graph": the expert path
never waits for the host, so it captures cleanly and suits torch.compile). The
ctypes binding is
opaque to torch.compile's tracer; these `torch.library` operators give it a
schema and a shape function (the fake implementation), so a compiled graph
keeps each call as one node instead of breaking around it. Each operator only
allocates its outputs and workspace and calls the library: the arithmetic is
libmoe's, and there is no CPU implementation.

    torch.ops.moe_gb300.router(x, w_r, k, score, normalize, scale, n_group, topk_group,
                               group_topn, sel_bias, logit_offset) -> (topk_idx, topk_w, aux)
    torch.ops.moe_gb300.forward(x, topk_idx, topk_w, w1, w2) -> y
    torch.ops.moe_gb300.forward_mx(x, topk_idx, topk_w, w1_codes, w1_scales, w2_codes,
                                   w2_scales) -> y

Shapes: x bf16 [T, H]; w_r fp32 [E, H]; w1 [E, 2I, H], w2 [E, H, I] (bf16, or
E4M3 codes with k-block-major E8M0 scales from `moe_mx_quantize`); topk_idx int32
[T, k]; topk_w fp32 [T, k]; y bf16 [T, H].

For training, `moe_layer(x, w_r, w1, w2, k, ...)` is the whole layer (router and
expert path, bf16) as one differentiable call: `torch.ops.moe_gb300.layer_train`
runs the router (keeping the fp32 logits), the routing metadata and both stages
(keeping the pre-activation h), and `torch.ops.moe_gb300.layer_backward` runs the
library's backward (dX with the router's term, dW_r, dW1, dW2); `register_autograd`
joins them. Gradients reach the router through y only: topk_idx, topk_w and aux
are returned without a gradient (the library does not differentiate aux).
`moe_layer(..., precision="mxfp8")` runs the expert stages and the weight gradients
in MXFP8 (`layer_train_mx` / `layer_backward_mx`; the data gradients stay bf16, as in
the guide's section "Expert precision") on E4M3 copies of w1 and w2 from an
`MxWeightCache`.
"""
from typing import Optional, Tuple

import torch

from . import binding as B
from .mx_cache import MxWeightCache

_LIB = "moe_gb300"


def _expect(t: torch.Tensor, name: str, dtype: torch.dtype, shape) -> None:
    """The library reads raw pointers: a tensor of another type or size would be
    misread, so each operator checks its arguments here (also in its shape function)."""
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, not {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, not {tuple(t.shape)}")


def _check_router_args(x, w_r, k, sel_bias, logit_offset):
    if x.dim() != 2 or w_r.dim() != 2:
        raise ValueError("x must be [T, H] and w_r [E, H]")
    T, H = x.shape
    E = w_r.shape[0]
    _expect(x, "x", torch.bfloat16, (T, H))
    _expect(w_r, "w_r", torch.float32, (E, H))
    if not 1 <= k <= E:
        raise ValueError(f"k must be in [1, E = {E}], not {k}")
    for name, t in (("sel_bias", sel_bias), ("logit_offset", logit_offset)):
        if t is not None:
            _expect(t, name, torch.float32, (E,))


def _check_expert_weights(x, w1, w2):
    if w1.dim() != 3 or w1.shape[1] % 2:
        raise ValueError("w1 must be [E, 2I, H]")
    E, two_i, H = w1.shape
    if x.shape[1] != H:
        raise ValueError(f"x has {x.shape[1]} columns, w1 {H}")
    _expect(w1, "w1", torch.bfloat16, (E, two_i, H))
    _expect(w2, "w2", torch.bfloat16, (E, H, two_i // 2))


def _check_mx_weights(w1, w2, w1_codes, w1_scales, w2_codes, w2_scales):
    E, two_i, H = w1.shape
    I = two_i // 2
    if H % 128 or I % 128:
        raise ValueError("MXFP8 needs H and I multiples of 128")
    _expect(w1_codes, "w1_codes", torch.uint8, (E, two_i, H))
    _expect(w1_scales, "w1_scales", torch.uint8, (H // 128, E, two_i, 4))
    _expect(w2_codes, "w2_codes", torch.uint8, (E, H, I))
    _expect(w2_scales, "w2_scales", torch.uint8, (I // 128, E, H, 4))


def _check_routing(x, topk_idx, topk_w, E):
    T = x.shape[0]
    if topk_idx.dim() != 2:
        raise ValueError("topk_idx must be [T, k]")
    k = topk_idx.shape[1]
    _expect(topk_idx, "topk_idx", torch.int32, (T, k))
    _expect(topk_w, "topk_w", torch.float32, (T, k))
    if not 1 <= k <= E:
        raise ValueError(f"k must be in [1, E = {E}], not {k}")


def _check_forward_args(x, topk_idx, topk_w, w1, w2):
    if x.dim() != 2:
        raise ValueError("x must be [T, H]")
    _expect(x, "x", torch.bfloat16, tuple(x.shape))
    _check_expert_weights(x, w1, w2)
    _check_routing(x, topk_idx, topk_w, w1.shape[0])


def _check_forward_mx_args(x, topk_idx, topk_w, w1_codes, w1_scales, w2_codes, w2_scales):
    if x.dim() != 2 or w1_codes.dim() != 3:
        raise ValueError("x must be [T, H] and w1_codes [E, 2I, H]")
    _expect(x, "x", torch.bfloat16, tuple(x.shape))
    E, two_i, H = w1_codes.shape
    if x.shape[1] != H or two_i % 2:
        raise ValueError("w1_codes must be [E, 2I, H] with H = x.shape[1]")
    I = two_i // 2
    if H % 128 or I % 128:
        raise ValueError("MXFP8 needs H and I multiples of 128")
    _expect(w1_codes, "w1_codes", torch.uint8, (E, two_i, H))
    _expect(w1_scales, "w1_scales", torch.uint8, (H // 128, E, two_i, 4))
    _expect(w2_codes, "w2_codes", torch.uint8, (E, H, I))
    _expect(w2_scales, "w2_scales", torch.uint8, (I // 128, E, H, 4))
    _check_routing(x, topk_idx, topk_w, E)


@torch.library.custom_op(f"{_LIB}::router", mutates_args=())
def router(x: torch.Tensor, w_r: torch.Tensor, k: int, score: str = "softmax", normalize: bool = True,
           scale: float = 1.0, n_group: int = 1, topk_group: int = 1, group_topn: int = 2,
           sel_bias: Optional[torch.Tensor] = None,
           logit_offset: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    _check_router_args(x, w_r, k, sel_bias, logit_offset)
    T, H = x.shape
    E = w_r.shape[0]
    shp = B.shape(T, H, 8, E, k)                    # I is not used by the router
    ws = B.new_workspace(shp, x.device)
    idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    aux = torch.zeros((1,), dtype=torch.float32, device=x.device)
    B.moe_router(x, w_r, shp, B.router_cfg(score, normalize, scale, n_group, topk_group, group_topn), idx, w, ws,
                 aux=aux, logit_offset=logit_offset, sel_bias=sel_bias)
    return idx, w, aux


@router.register_fake
def _router_fake(x, w_r, k, score="softmax", normalize=True, scale=1.0, n_group=1, topk_group=1, group_topn=2,
                 sel_bias=None, logit_offset=None):
    _check_router_args(x, w_r, k, sel_bias, logit_offset)
    T = x.shape[0]
    return (x.new_empty((T, k), dtype=torch.int32), x.new_empty((T, k), dtype=torch.float32),
            x.new_empty((1,), dtype=torch.float32))


@torch.library.custom_op(f"{_LIB}::forward", mutates_args=())
def forward(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor, w1: torch.Tensor,
            w2: torch.Tensor) -> torch.Tensor:
    _check_forward_args(x, topk_idx, topk_w, w1, w2)
    T, H = x.shape
    E, two_i, _ = w1.shape
    shp = B.shape(T, H, two_i // 2, E, topk_idx.shape[1])
    ws = B.new_workspace(shp, x.device)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    B.moe_forward(x, topk_idx, topk_w, w1, w2, shp, y, ws)
    return y


@forward.register_fake
def _forward_fake(x, topk_idx, topk_w, w1, w2):
    _check_forward_args(x, topk_idx, topk_w, w1, w2)
    return x.new_empty(x.shape, dtype=torch.bfloat16)


@torch.library.custom_op(f"{_LIB}::forward_mx", mutates_args=())
def forward_mx(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor, w1_codes: torch.Tensor,
               w1_scales: torch.Tensor, w2_codes: torch.Tensor, w2_scales: torch.Tensor) -> torch.Tensor:
    _check_forward_mx_args(x, topk_idx, topk_w, w1_codes, w1_scales, w2_codes, w2_scales)
    T, H = x.shape
    E, two_i, _ = w1_codes.shape
    shp = B.shape(T, H, two_i // 2, E, topk_idx.shape[1], mxfp8=True)
    ws = B.new_workspace(shp, x.device)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    B.moe_forward_mx(x, topk_idx, topk_w, w1_codes, w1_scales, w2_codes, w2_scales, shp, y, ws)
    return y


@forward_mx.register_fake
def _forward_mx_fake(x, topk_idx, topk_w, w1_codes, w1_scales, w2_codes, w2_scales):
    _check_forward_mx_args(x, topk_idx, topk_w, w1_codes, w1_scales, w2_codes, w2_scales)
    return x.new_empty(x.shape, dtype=torch.bfloat16)


def _train_workspace(shp, device) -> torch.Tensor:
    # a whole allocation (the caching allocator aligns it to 512 bytes), so the
    # workspace can be an operator output that aliases nothing
    ws = torch.empty(B.moe_workspace_size(shp), dtype=torch.uint8, device=device)
    if ws.data_ptr() % 256:
        raise RuntimeError("libmoe needs a 256-byte aligned workspace")
    B.moe_workspace_init(ws)
    return ws


@torch.library.custom_op(f"{_LIB}::layer_train", mutates_args=())
def layer_train(x: torch.Tensor, w_r: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor, k: int,
                score: str = "softmax", normalize: bool = True, scale: float = 1.0, n_group: int = 1,
                topk_group: int = 1, group_topn: int = 2, sel_bias: Optional[torch.Tensor] = None,
                logit_offset: Optional[torch.Tensor] = None
                ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor,
                           torch.Tensor]:
    """The layer's training forward: (y, topk_idx, topk_w, aux, h, logits, ws); the last
    three are what layer_backward reads."""
    _check_router_args(x, w_r, k, sel_bias, logit_offset)
    _check_expert_weights(x, w1, w2)
    T, H = x.shape
    E, two_i, _ = w1.shape
    I = two_i // 2
    shp = B.shape(T, H, I, E, k, training=True)
    ws = _train_workspace(shp, x.device)
    idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    aux = torch.zeros((1,), dtype=torch.float32, device=x.device)
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    a = torch.empty((T * k, I), dtype=torch.bfloat16, device=x.device)
    h = torch.empty((T * k, 2 * I), dtype=torch.bfloat16, device=x.device)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    cfg = B.router_cfg(score, normalize, scale, n_group, topk_group, group_topn)
    B.moe_router_train(x, w_r, shp, cfg, idx, w, logits, ws, aux=aux, logit_offset=logit_offset,
                       sel_bias=sel_bias)
    B.moe_routing_metadata(idx, shp, ws)
    B.moe_dispatch_gemm1_train(x, w1, shp, a, h, ws)
    B.moe_swiglu_gemm2_combine(a, w, w2, shp, y, ws)
    return y, idx, w, aux, h, logits, ws


@layer_train.register_fake
def _layer_train_fake(x, w_r, w1, w2, k, score="softmax", normalize=True, scale=1.0, n_group=1, topk_group=1,
                      group_topn=2, sel_bias=None, logit_offset=None):
    _check_router_args(x, w_r, k, sel_bias, logit_offset)
    _check_expert_weights(x, w1, w2)
    T, H = x.shape
    E, two_i, _ = w1.shape
    n = B.moe_workspace_size(B.shape(int(T), int(H), int(two_i) // 2, int(E), k, training=True))
    return (x.new_empty((T, H), dtype=torch.bfloat16), x.new_empty((T, k), dtype=torch.int32),
            x.new_empty((T, k), dtype=torch.float32), x.new_empty((1,), dtype=torch.float32),
            x.new_empty((T * k, two_i), dtype=torch.bfloat16), x.new_empty((T, E), dtype=torch.float32),
            x.new_empty((n,), dtype=torch.uint8))


@torch.library.custom_op(f"{_LIB}::layer_backward", mutates_args=("ws",))
def layer_backward(dy: torch.Tensor, x: torch.Tensor, w_r: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor,
                   topk_idx: torch.Tensor, topk_w: torch.Tensor, h: torch.Tensor, logits: torch.Tensor,
                   ws: torch.Tensor, score: str = "softmax", normalize: bool = True, scale: float = 1.0,
                   n_group: int = 1, topk_group: int = 1, group_topn: int = 2
                   ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor]:
    """The layer's backward from dY: (dX, dW_r, dW1, dW2). ws is layer_train's workspace
    (its routing metadata and dispatched rows; the backward also uses it as scratch)."""
    _expect(dy, "dy", torch.bfloat16, tuple(x.shape))
    T, H = x.shape
    E, two_i, _ = w1.shape
    k = topk_idx.shape[1]
    shp = B.shape(T, H, two_i // 2, E, k, training=True)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    dw_r = torch.empty((E, H), dtype=torch.float32, device=x.device)
    dw1 = torch.empty_like(w1)
    dw2 = torch.empty_like(w2)
    dtw = torch.empty((T, k), dtype=torch.float32, device=x.device)   # routing-weight gradient, for dW_r
    cfg = B.router_cfg(score, normalize, scale, n_group, topk_group, group_topn)
    B.moe_backward(x, topk_idx, topk_w, w1, w2, h, dy.contiguous(), shp, dx, dw1, dw2, ws, w_r=w_r,
                   logits=logits, cfg=cfg, dw_r=dw_r, dtopk_w=dtw)
    return dx, dw_r, dw1, dw2


@layer_backward.register_fake
def _layer_backward_fake(dy, x, w_r, w1, w2, topk_idx, topk_w, h, logits, ws, score="softmax", normalize=True,
                         scale=1.0, n_group=1, topk_group=1, group_topn=2):
    return (x.new_empty(x.shape, dtype=torch.bfloat16), w_r.new_empty(w_r.shape, dtype=torch.float32),
            w1.new_empty(w1.shape), w2.new_empty(w2.shape))


def _layer_setup_context(ctx, inputs, output):
    x, w_r, w1, w2, k, score, normalize, scale, n_group, topk_group, group_topn, sel_bias, logit_offset = inputs
    _, idx, w, _, h, logits, ws = output
    ctx.save_for_backward(x, w_r, w1, w2, idx, w, h, logits, ws)
    ctx.cfg = (score, normalize, scale, n_group, topk_group, group_topn)
    ctx.mark_non_differentiable(*output[1:])


def _layer_backward_rule(ctx, dy, *unused):
    x, w_r, w1, w2, idx, w, h, logits, ws = ctx.saved_tensors
    dx, dw_r, dw1, dw2 = layer_backward(dy, x, w_r, w1, w2, idx, w, h, logits, ws, *ctx.cfg)
    return dx, dw_r, dw1, dw2, None, None, None, None, None, None, None, None, None


layer_train.register_autograd(_layer_backward_rule, setup_context=_layer_setup_context)


@torch.library.custom_op(f"{_LIB}::layer_train_mx", mutates_args=())
def layer_train_mx(x: torch.Tensor, w_r: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor, w1_codes: torch.Tensor,
                   w1_scales: torch.Tensor, w2_codes: torch.Tensor, w2_scales: torch.Tensor, k: int,
                   score: str = "softmax", normalize: bool = True, scale: float = 1.0, n_group: int = 1,
                   topk_group: int = 1, group_topn: int = 2, sel_bias: Optional[torch.Tensor] = None,
                   logit_offset: Optional[torch.Tensor] = None
                   ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor,
                              torch.Tensor]:
    """layer_train with the expert stages in MXFP8 (the guide's mxfp8 expert precision):
    the router as in bf16, x quantized by the dispatch, stage 1 on the E4M3 copy of w1
    (keeping h), stage 2 on that of w2. w1 and w2 themselves are only read by the
    backward's data gradients."""
    _check_router_args(x, w_r, k, sel_bias, logit_offset)
    _check_expert_weights(x, w1, w2)
    _check_mx_weights(w1, w2, w1_codes, w1_scales, w2_codes, w2_scales)
    T, H = x.shape
    E, two_i, _ = w1.shape
    I = two_i // 2
    shp = B.shape(T, H, I, E, k, training=True, mxfp8=True)
    ws = _train_workspace(shp, x.device)
    R = T * k
    idx = torch.empty((T, k), dtype=torch.int32, device=x.device)
    w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    aux = torch.zeros((1,), dtype=torch.float32, device=x.device)
    logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    aq = torch.empty((R, I), dtype=torch.uint8, device=x.device)
    as_ = B.mx_scales_empty((R, I), x.device)
    h = torch.empty((R, 2 * I), dtype=torch.bfloat16, device=x.device)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    cfg = B.router_cfg(score, normalize, scale, n_group, topk_group, group_topn)
    B.moe_router_train(x, w_r, shp, cfg, idx, w, logits, ws, aux=aux, logit_offset=logit_offset,
                       sel_bias=sel_bias)
    B.moe_routing_metadata(idx, shp, ws)
    B.moe_mx_quantize_dispatch(x, shp, ws)
    B.moe_dispatch_gemm1_mx_train(w1_codes, w1_scales, shp, aq, as_, h, ws)
    B.moe_swiglu_gemm2_combine_mx(aq, as_, w, w2_codes, w2_scales, shp, y, ws)
    return y, idx, w, aux, h, logits, ws


@layer_train_mx.register_fake
def _layer_train_mx_fake(x, w_r, w1, w2, w1_codes, w1_scales, w2_codes, w2_scales, k, score="softmax",
                         normalize=True, scale=1.0, n_group=1, topk_group=1, group_topn=2, sel_bias=None,
                         logit_offset=None):
    _check_router_args(x, w_r, k, sel_bias, logit_offset)
    _check_expert_weights(x, w1, w2)
    _check_mx_weights(w1, w2, w1_codes, w1_scales, w2_codes, w2_scales)
    T, H = x.shape
    E, two_i, _ = w1.shape
    n = B.moe_workspace_size(B.shape(int(T), int(H), int(two_i) // 2, int(E), k, training=True, mxfp8=True))
    return (x.new_empty((T, H), dtype=torch.bfloat16), x.new_empty((T, k), dtype=torch.int32),
            x.new_empty((T, k), dtype=torch.float32), x.new_empty((1,), dtype=torch.float32),
            x.new_empty((T * k, two_i), dtype=torch.bfloat16), x.new_empty((T, E), dtype=torch.float32),
            x.new_empty((n,), dtype=torch.uint8))


@torch.library.custom_op(f"{_LIB}::layer_backward_mx", mutates_args=("ws",))
def layer_backward_mx(dy: torch.Tensor, x: torch.Tensor, w_r: torch.Tensor, w1: torch.Tensor, w2: torch.Tensor,
                      topk_idx: torch.Tensor, topk_w: torch.Tensor, h: torch.Tensor, logits: torch.Tensor,
                      ws: torch.Tensor, score: str = "softmax", normalize: bool = True, scale: float = 1.0,
                      n_group: int = 1, topk_group: int = 1, group_topn: int = 2
                      ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor, torch.Tensor]:
    """layer_backward of layer_train_mx: the data gradients in bf16 (on w1, w2 and the
    saved h), dW2 and dW1 in MXFP8 (both operands quantized along the routed rows), the
    router's gradients as in bf16. Returns (dX, dW_r, dW1, dW2)."""
    _expect(dy, "dy", torch.bfloat16, tuple(x.shape))
    T, H = x.shape
    E, two_i, _ = w1.shape
    k = topk_idx.shape[1]
    shp = B.shape(T, H, two_i // 2, E, k, training=True, mxfp8=True)
    dy = dy.contiguous()
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    dw_r = torch.empty((E, H), dtype=torch.float32, device=x.device)
    dw1 = torch.empty_like(w1)
    dw2 = torch.empty_like(w2)
    dtw = torch.empty((T, k), dtype=torch.float32, device=x.device)
    cfg = B.router_cfg(score, normalize, scale, n_group, topk_group, group_topn)
    B.moe_backward_stage2_data(dy, topk_w, w2, h, shp, ws, dtopk_w=dtw)
    B.moe_backward_stage2_weight_mx(dy, shp, dw2, ws)
    B.moe_router_backward(x, logits, topk_idx, topk_w, dtw, shp, cfg, dw_r, ws)
    B.moe_backward_stage1_data(w1, shp, dx, ws, w_r=w_r, topk_idx=topk_idx, cfg=cfg)
    B.moe_backward_stage1_weight_mx(x, shp, dw1, ws)
    return dx, dw_r, dw1, dw2


@layer_backward_mx.register_fake
def _layer_backward_mx_fake(dy, x, w_r, w1, w2, topk_idx, topk_w, h, logits, ws, score="softmax",
                            normalize=True, scale=1.0, n_group=1, topk_group=1, group_topn=2):
    return (x.new_empty(x.shape, dtype=torch.bfloat16), w_r.new_empty(w_r.shape, dtype=torch.float32),
            w1.new_empty(w1.shape), w2.new_empty(w2.shape))


def _layer_mx_setup_context(ctx, inputs, output):
    x, w_r, w1, w2 = inputs[:4]
    score, normalize, scale, n_group, topk_group, group_topn = inputs[9:15]
    _, idx, w, _, h, logits, ws = output
    ctx.save_for_backward(x, w_r, w1, w2, idx, w, h, logits, ws)
    ctx.cfg = (score, normalize, scale, n_group, topk_group, group_topn)
    ctx.mark_non_differentiable(*output[1:])


def _layer_mx_backward_rule(ctx, dy, *unused):
    x, w_r, w1, w2, idx, w, h, logits, ws = ctx.saved_tensors
    dx, dw_r, dw1, dw2 = layer_backward_mx(dy, x, w_r, w1, w2, idx, w, h, logits, ws, *ctx.cfg)
    return (dx, dw_r, dw1, dw2) + (None,) * 13


layer_train_mx.register_autograd(_layer_mx_backward_rule, setup_context=_layer_mx_setup_context)

# the E4M3 copies of the expert weights that moe_layer(..., precision="mxfp8") uses when
# no cache is passed; call .invalidate() once per optimizer step
DEFAULT_MX_WEIGHT_CACHE = MxWeightCache()


def moe_layer(x, w_r, w1, w2, k, score="softmax", normalize=True, scale=1.0, n_group=1, topk_group=1,
              group_topn=2, sel_bias=None, logit_offset=None, precision="bf16", weight_cache=None):
    """The MoE layer as one differentiable call: (y, topk_idx, topk_w, aux). x bf16 [T, H],
    w_r fp32 [E, H], w1 bf16 [E, 2I, H], w2 bf16 [E, H, I]; y.backward(dy) fills x.grad
    (with the router's term), w_r.grad, w1.grad and w2.grad through the library.

    precision="mxfp8" runs the expert stages and the weight gradients in MXFP8 (H and I
    multiples of 128): w1 and w2 stay the bf16 parameters, and their E4M3 copies come
    from `weight_cache` (an MxWeightCache; DEFAULT_MX_WEIGHT_CACHE if None), which
    quantizes again when a weight's version counter moves and must be invalidated once
    per optimizer step."""
    if precision == "bf16":
        y, idx, w, aux, _, _, _ = layer_train(x, w_r, w1, w2, k, score, normalize, scale, n_group, topk_group,
                                              group_topn, sel_bias, logit_offset)
    elif precision == "mxfp8":
        cache = DEFAULT_MX_WEIGHT_CACHE if weight_cache is None else weight_cache
        w1c, w1s = cache.get(w1)
        w2c, w2s = cache.get(w2)
        y, idx, w, aux, _, _, _ = layer_train_mx(x, w_r, w1, w2, w1c, w1s, w2c, w2s, k, score, normalize, scale,
                                                 n_group, topk_group, group_topn, sel_bias, logit_offset)
    else:
        raise ValueError(f"precision must be 'bf16' or 'mxfp8', not {precision!r}")
    return y, idx, w, aux
