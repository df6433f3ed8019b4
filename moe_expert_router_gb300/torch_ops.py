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
"""
from typing import Optional, Tuple

import torch

from . import binding as B

_LIB = "moe_gb300"


@torch.library.custom_op(f"{_LIB}::router", mutates_args=())
def router(x: torch.Tensor, w_r: torch.Tensor, k: int, score: str = "softmax", normalize: bool = True,
           scale: float = 1.0, n_group: int = 1, topk_group: int = 1, group_topn: int = 2,
           sel_bias: Optional[torch.Tensor] = None,
           logit_offset: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
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
    T = x.shape[0]
    return (x.new_empty((T, k), dtype=torch.int32), x.new_empty((T, k), dtype=torch.float32),
            x.new_empty((1,), dtype=torch.float32))


@torch.library.custom_op(f"{_LIB}::forward", mutates_args=())
def forward(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor, w1: torch.Tensor,
            w2: torch.Tensor) -> torch.Tensor:
    T, H = x.shape
    E, two_i, _ = w1.shape
    shp = B.shape(T, H, two_i // 2, E, topk_idx.shape[1])
    ws = B.new_workspace(shp, x.device)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    B.moe_forward(x, topk_idx, topk_w, w1, w2, shp, y, ws)
    return y


@forward.register_fake
def _forward_fake(x, topk_idx, topk_w, w1, w2):
    return x.new_empty(x.shape, dtype=torch.bfloat16)


@torch.library.custom_op(f"{_LIB}::forward_mx", mutates_args=())
def forward_mx(x: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor, w1_codes: torch.Tensor,
               w1_scales: torch.Tensor, w2_codes: torch.Tensor, w2_scales: torch.Tensor) -> torch.Tensor:
    T, H = x.shape
    E, two_i, _ = w1_codes.shape
    shp = B.shape(T, H, two_i // 2, E, topk_idx.shape[1], mxfp8=True)
    ws = B.new_workspace(shp, x.device)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=x.device)
    B.moe_forward_mx(x, topk_idx, topk_w, w1_codes, w1_scales, w2_codes, w2_scales, shp, y, ws)
    return y


@forward_mx.register_fake
def _forward_mx_fake(x, topk_idx, topk_w, w1_codes, w1_scales, w2_codes, w2_scales):
    return x.new_empty(x.shape, dtype=torch.bfloat16)
