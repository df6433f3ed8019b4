"""ctypes binding of libmoe.so: the same entry points as include/moe.h.

Argument marshalling only -- every step of the expert path runs in the CUDA
kernels of libmoe. There is no fallback: if the library is missing or cannot be
loaded, every call raises.

Tensors are torch CUDA tensors; the stream defaults to torch's current stream
on the tensors' device.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_CUDA", 4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_DEVICE_FLAGGED"}
DEVERR_BAD_EXPERT_INDEX = 0x1
DEVERR_WAIT_TIMEOUT = 0x2
DEVERR_CAPACITY = 0x4
SCORE_SOFTMAX = 0
SCORE_SIGMOID = 1
SHAPE_TRAINING = 0x1
SHAPE_MXFP8 = 0x2
SHAPE_PACKED_WEIGHTS = 0x4


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("H", ctypes.c_int64), ("I", ctypes.c_int64),
                ("E", ctypes.c_int64), ("k", ctypes.c_int32), ("flags", ctypes.c_int32)]


class RouterCfg(ctypes.Structure):
    _fields_ = [("score_fn", ctypes.c_int32), ("normalize", ctypes.c_int32),
                ("scale", ctypes.c_float), ("n_group", ctypes.c_int32),
                ("topk_group", ctypes.c_int32), ("group_topn", ctypes.c_int32)]


class WsLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("err", "counts", "offsets", "mt_prefix", "perm_slot", "row_of", "meta", "router", "a",
                 "obuf", "combine", "dh", "aw", "dtw_part", "dlogits", "xp", "dyp", "dwr_part", "x_codes", "x_scales", "a_codes", "a_scales",
                 "mx_wgrad", "total")]


# name -> argument types (all return moe_status_t unless listed in _RESTYPES)
_P = ctypes.c_void_p
_SIG = {
    "moe_workspace_size": [ctypes.POINTER(Shape), ctypes.POINTER(ctypes.c_size_t)],
    "moe_workspace_layout": [ctypes.POINTER(Shape), ctypes.POINTER(WsLayout)],
    "moe_workspace_init": [_P, ctypes.c_size_t, _P],
    "moe_router": [_P, _P, _P, _P, ctypes.POINTER(Shape), ctypes.POINTER(RouterCfg), _P, _P, _P,
                   _P, ctypes.c_size_t, _P],
    "moe_router_noalloc": [_P, _P, _P, _P, ctypes.POINTER(Shape), ctypes.POINTER(RouterCfg), _P,
                           _P, _P, _P],
    "moe_router_noalloc_get_error": [ctypes.POINTER(ctypes.c_int32), _P],
    "moe_routing_metadata": [_P, ctypes.POINTER(Shape), _P, ctypes.c_size_t, _P],
    "moe_dispatch_gemm1": [_P, _P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_swiglu_gemm2_combine": [_P, _P, _P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_forward": [_P, _P, _P, _P, _P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_route_logits": [_P, _P, _P, ctypes.POINTER(Shape), ctypes.POINTER(RouterCfg), _P, _P, _P, _P,
                         ctypes.c_size_t, _P],
    "moe_router_train": [_P, _P, _P, _P, ctypes.POINTER(Shape), ctypes.POINTER(RouterCfg), _P, _P,
                         _P, _P, _P, ctypes.c_size_t, _P],
    "moe_dispatch_gemm1_train": [_P, _P, ctypes.POINTER(Shape), _P, _P, _P, ctypes.c_size_t, _P],
    "moe_backward_stage2_data": [_P, _P, _P, _P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_backward_stage2_weight": [_P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_router_backward": [_P, _P, _P, _P, _P, ctypes.POINTER(Shape), ctypes.POINTER(RouterCfg), _P,
                            _P, ctypes.c_size_t, _P],
    "moe_backward_stage1_data": [_P, _P, _P, ctypes.POINTER(RouterCfg), ctypes.POINTER(Shape), _P, _P,
                                 ctypes.c_size_t, _P],
    "moe_backward_stage1_weight": [_P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_backward": [_P, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(Shape),
                     ctypes.POINTER(RouterCfg), _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_mx_quantize": [_P, ctypes.c_int64, ctypes.c_int64, _P, _P, _P],
    "moe_mx_quantize_dispatch": [_P, ctypes.POINTER(Shape), _P, ctypes.c_size_t, _P],
    "moe_dispatch_gemm1_mx": [_P, _P, ctypes.POINTER(Shape), _P, _P, _P, ctypes.c_size_t, _P],
    "moe_dispatch_gemm1_mx_train": [_P, _P, ctypes.POINTER(Shape), _P, _P, _P, _P, ctypes.c_size_t, _P],
    "moe_backward_stage2_weight_mx": [_P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_backward_stage1_weight_mx": [_P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_swiglu_gemm2_combine_mx": [_P, _P, _P, _P, _P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_forward_mx": [_P, _P, _P, _P, _P, _P, _P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_dispatch_rows": [_P, _P, ctypes.POINTER(Shape), _P, _P, _P, ctypes.c_size_t, _P],
    "moe_combine_rows": [_P, ctypes.POINTER(Shape), _P, _P, ctypes.c_size_t, _P],
    "moe_ep_pack": [_P, _P, ctypes.POINTER(Shape), ctypes.c_int32, ctypes.c_int64, _P, _P, _P, _P,
                    ctypes.c_size_t, _P],
    "moe_ep_receive_metadata": [_P, ctypes.c_int32, ctypes.c_int64, ctypes.POINTER(Shape), _P, ctypes.c_size_t,
                                _P],
    "moe_ep_combine": [_P, ctypes.POINTER(Shape), ctypes.c_int32, ctypes.c_int64, _P, _P, ctypes.c_size_t, _P],
    "moe_packed_weights_size": [ctypes.POINTER(Shape), ctypes.POINTER(ctypes.c_size_t),
                                ctypes.POINTER(ctypes.c_size_t)],
    "moe_pack_weights": [_P, _P, ctypes.POINTER(Shape), _P, _P, _P],
    "moe_get_device_error": [_P, ctypes.POINTER(ctypes.c_int32), _P],
    "moe_status_string": [ctypes.c_int],
    "moe_kernel_launch_count": [],
}
_RESTYPES = {"moe_status_string": ctypes.c_char_p, "moe_kernel_launch_count": ctypes.c_uint64}

_lib = None


def load(path: str = LIB_PATH):
    """Load libmoe.so (built by moe_expert_router_gb300.build); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, args in _SIG.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _RESTYPES.get(name, ctypes.c_int)
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoEError(fn, status)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch tensor")
    if not t.is_cuda:
        raise ValueError("libmoe takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream, like):
    if stream is None:
        stream = torch.cuda.current_stream(like.device)
    return ctypes.c_void_p(stream.cuda_stream)


def shape(T, H, I, E, k, training=False, mxfp8=False, packed=False) -> Shape:
    flags = ((SHAPE_TRAINING if training else 0) | (SHAPE_MXFP8 if mxfp8 else 0) |
             (SHAPE_PACKED_WEIGHTS if packed else 0))
    return Shape(int(T), int(H), int(I), int(E), int(k), flags)


def router_cfg(score="softmax", normalize=True, scale=1.0, n_group=1, topk_group=1,
               group_topn=2) -> RouterCfg:
    fn = SCORE_SOFTMAX if score == "softmax" else SCORE_SIGMOID
    return RouterCfg(fn, int(bool(normalize)), float(scale), int(n_group), int(topk_group),
                     int(group_topn))


def moe_workspace_size(shp: Shape) -> int:
    n = ctypes.c_size_t()
    _check("moe_workspace_size", load().moe_workspace_size(ctypes.byref(shp), ctypes.byref(n)))
    return int(n.value)


def moe_workspace_layout(shp: Shape) -> WsLayout:
    L = WsLayout()
    _check("moe_workspace_layout", load().moe_workspace_layout(ctypes.byref(shp), ctypes.byref(L)))
    return L


def moe_workspace_init(ws, stream=None):
    _check("moe_workspace_init",
           load().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream, ws)))


def moe_router(x, w_r, shp, cfg, topk_idx, topk_w, ws, aux=None, logit_offset=None,
               sel_bias=None, stream=None):
    _check("moe_router", load().moe_router(
        _ptr(x), _ptr(w_r), _ptr(logit_offset), _ptr(sel_bias), ctypes.byref(shp),
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(topk_w), _ptr(aux), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream, x)))


def moe_router_noalloc(x, w_r, shp, cfg, topk_idx, topk_w, aux=None, logit_offset=None,
                       sel_bias=None, stream=None):
    """moe_router without a workspace: for callers that may not allocate device
    memory (the scratch lives in a static array inside libmoe; T * E <= 2**20, E * H <= 2**20)."""
    _check("moe_router_noalloc", load().moe_router_noalloc(
        _ptr(x), _ptr(w_r), _ptr(logit_offset), _ptr(sel_bias), ctypes.byref(shp),
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(topk_w), _ptr(aux), _stream(stream, x)))


def moe_router_noalloc_get_error(stream=None) -> int:
    """Wait for the stream, return and clear moe_router_noalloc's error word on
    the current device (0 = none)."""
    import torch
    code = ctypes.c_int32()
    if stream is None:
        stream = torch.cuda.current_stream()
    st = load().moe_router_noalloc_get_error(ctypes.byref(code), ctypes.c_void_p(stream.cuda_stream))
    if st not in (MOE_OK, 5):
        raise MoEError("moe_router_noalloc_get_error", st)
    return int(code.value)


def moe_routing_metadata(topk_idx, shp, ws, stream=None):
    _check("moe_routing_metadata", load().moe_routing_metadata(
        _ptr(topk_idx), ctypes.byref(shp), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream, topk_idx)))


def moe_dispatch_gemm1(x, w1, shp, a, ws, stream=None):
    _check("moe_dispatch_gemm1", load().moe_dispatch_gemm1(
        _ptr(x), _ptr(w1), ctypes.byref(shp), _ptr(a), _ptr(ws), ws.numel() * ws.element_size(),
        _stream(stream, x)))


def moe_swiglu_gemm2_combine(a, topk_w, w2, shp, y, ws, stream=None):
    _check("moe_swiglu_gemm2_combine", load().moe_swiglu_gemm2_combine(
        _ptr(a), _ptr(topk_w), _ptr(w2), ctypes.byref(shp), _ptr(y), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream, a)))


def moe_forward(x, topk_idx, topk_w, w1, w2, shp, y, ws, stream=None):
    _check("moe_forward", load().moe_forward(
        _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(w1), _ptr(w2), ctypes.byref(shp), _ptr(y),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream, x)))


def _cfg_ref(cfg):
    return None if cfg is None else ctypes.byref(cfg)


def _nbytes(ws):
    return ws.numel() * ws.element_size()


def moe_route_logits(logits, shp, cfg, topk_idx, topk_w, ws, aux=None, logit_offset=None,
                     sel_bias=None, stream=None):
    """Routing from given fp32 logits [T, E] (random logits: the `uniform` force-balance mode)."""
    _check("moe_route_logits", load().moe_route_logits(
        _ptr(logits), _ptr(logit_offset), _ptr(sel_bias), ctypes.byref(shp), ctypes.byref(cfg),
        _ptr(topk_idx), _ptr(topk_w), _ptr(aux), _ptr(ws), _nbytes(ws), _stream(stream, logits)))


def moe_router_train(x, w_r, shp, cfg, topk_idx, topk_w, logits, ws, aux=None, logit_offset=None,
                     sel_bias=None, stream=None):
    """moe_router that also writes the fp32 logits [T, E] for moe_router_backward."""
    _check("moe_router_train", load().moe_router_train(
        _ptr(x), _ptr(w_r), _ptr(logit_offset), _ptr(sel_bias), ctypes.byref(shp),
        ctypes.byref(cfg), _ptr(topk_idx), _ptr(topk_w), _ptr(aux), _ptr(logits), _ptr(ws),
        _nbytes(ws), _stream(stream, x)))


def moe_dispatch_gemm1_train(x, w1, shp, a, h, ws, stream=None):
    """moe_dispatch_gemm1 that also stores the pre-activation h [T*k, 2I] (routed order)."""
    _check("moe_dispatch_gemm1_train", load().moe_dispatch_gemm1_train(
        _ptr(x), _ptr(w1), ctypes.byref(shp), _ptr(a), _ptr(h), _ptr(ws), _nbytes(ws),
        _stream(stream, x)))


def moe_backward_stage2_data(dy, topk_w, w2, h, shp, ws, dtopk_w=None, stream=None):
    _check("moe_backward_stage2_data", load().moe_backward_stage2_data(
        _ptr(dy), _ptr(topk_w), _ptr(w2), _ptr(h), ctypes.byref(shp), _ptr(dtopk_w), _ptr(ws),
        _nbytes(ws), _stream(stream, ws)))


def moe_backward_stage2_weight(dy, shp, dw2, ws, stream=None):
    _check("moe_backward_stage2_weight", load().moe_backward_stage2_weight(
        _ptr(dy), ctypes.byref(shp), _ptr(dw2), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_router_backward(x, logits, topk_idx, topk_w, dtopk_w, shp, cfg, dw_r, ws, stream=None):
    _check("moe_router_backward", load().moe_router_backward(
        _ptr(x), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(dtopk_w), ctypes.byref(shp),
        ctypes.byref(cfg), _ptr(dw_r), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_backward_stage1_data(w1, shp, dx, ws, w_r=None, topk_idx=None, cfg=None, stream=None):
    _check("moe_backward_stage1_data", load().moe_backward_stage1_data(
        _ptr(w1), _ptr(w_r), _ptr(topk_idx), _cfg_ref(cfg), ctypes.byref(shp), _ptr(dx), _ptr(ws),
        _nbytes(ws), _stream(stream, ws)))


def moe_backward_stage1_weight(x, shp, dw1, ws, stream=None):
    _check("moe_backward_stage1_weight", load().moe_backward_stage1_weight(
        _ptr(x), ctypes.byref(shp), _ptr(dw1), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_backward(x, topk_idx, topk_w, w1, w2, h, dy, shp, dx, dw1, dw2, ws, w_r=None, logits=None,
                 cfg=None, dw_r=None, dtopk_w=None, stream=None):
    _check("moe_backward", load().moe_backward(
        _ptr(x), _ptr(w_r), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(w1), _ptr(w2), _ptr(h),
        _ptr(dy), ctypes.byref(shp), _cfg_ref(cfg), _ptr(dx), _ptr(dw1), _ptr(dw2), _ptr(dw_r),
        _ptr(dtopk_w), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def mx_scales_empty(shape, device):
    """An uninitialised buffer for the k-block-major E8M0 scales of an MXFP8
    tensor of `shape` (rows = the product of the leading dimensions, cols the
    last, a multiple of 128): uint8 [cols / 128, *shape[:-1], 4] when rows is a
    multiple of 4, else [cols / 128, rows rounded up to 4, 4] -- one 32-bit word
    per row and 128-column block, rows consecutive within a block."""
    shape = tuple(shape)
    rows = 1
    for d in shape[:-1]:
        rows *= d
    lead = shape[:-1] if rows % 4 == 0 else ((rows + 3) // 4 * 4,)
    return torch.empty((shape[-1] // 128,) + lead + (4,), dtype=torch.uint8, device=device)


def moe_mx_quantize(t, codes, scales, stream=None):
    """MXFP8 quantization of a bf16 tensor along its last dimension (a multiple of
    128): codes uint8 of the same shape, scales k-block-major (``mx_scales_empty``)."""
    cols = t.shape[-1]
    rows = t.numel() // cols if cols else 0
    if codes.numel() != t.numel() or scales.numel() * 32 != (rows + 3) // 4 * 4 * cols:
        raise ValueError("codes must match t and scales hold the k-block-major words of rows rounded up to 4")
    _check("moe_mx_quantize", load().moe_mx_quantize(_ptr(t), rows, cols, _ptr(codes), _ptr(scales),
                                                     _stream(stream, t)))


def moe_mx_quantize_dispatch(x, shp, ws, stream=None):
    """The MXFP8 dispatch: x quantized into the workspace in routed-row order."""
    _check("moe_mx_quantize_dispatch", load().moe_mx_quantize_dispatch(
        _ptr(x), ctypes.byref(shp), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_dispatch_gemm1_mx(w1q, w1s, shp, aq, as_, ws, stream=None):
    _check("moe_dispatch_gemm1_mx", load().moe_dispatch_gemm1_mx(
        _ptr(w1q), _ptr(w1s), ctypes.byref(shp), _ptr(aq), _ptr(as_), _ptr(ws), _nbytes(ws),
        _stream(stream, ws)))


def moe_dispatch_gemm1_mx_train(w1q, w1s, shp, aq, as_, h, ws, stream=None):
    _check("moe_dispatch_gemm1_mx_train", load().moe_dispatch_gemm1_mx_train(
        _ptr(w1q), _ptr(w1s), ctypes.byref(shp), _ptr(aq), _ptr(as_), _ptr(h), _ptr(ws), _nbytes(ws),
        _stream(stream, ws)))


def moe_backward_stage2_weight_mx(dy, shp, dw2, ws, stream=None):
    _check("moe_backward_stage2_weight_mx", load().moe_backward_stage2_weight_mx(
        _ptr(dy), ctypes.byref(shp), _ptr(dw2), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_backward_stage1_weight_mx(x, shp, dw1, ws, stream=None):
    _check("moe_backward_stage1_weight_mx", load().moe_backward_stage1_weight_mx(
        _ptr(x), ctypes.byref(shp), _ptr(dw1), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_swiglu_gemm2_combine_mx(aq, as_, topk_w, w2q, w2s, shp, y, ws, stream=None):
    _check("moe_swiglu_gemm2_combine_mx", load().moe_swiglu_gemm2_combine_mx(
        _ptr(aq), _ptr(as_), _ptr(topk_w), _ptr(w2q), _ptr(w2s), ctypes.byref(shp), _ptr(y), _ptr(ws),
        _nbytes(ws), _stream(stream, ws)))


def moe_forward_mx(x, topk_idx, topk_w, w1q, w1s, w2q, w2s, shp, y, ws, stream=None):
    _check("moe_forward_mx", load().moe_forward_mx(
        _ptr(x), _ptr(topk_idx), _ptr(topk_w), _ptr(w1q), _ptr(w1s), _ptr(w2q), _ptr(w2s),
        ctypes.byref(shp), _ptr(y), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_dispatch_rows(x, shp, rows, ws, topk_w=None, row_weight=None, stream=None):
    """rows[r] = x[token of routed row r] (and row_weight[r] = its routing weight): the
    send buffer of an expert-parallel dispatch."""
    _check("moe_dispatch_rows", load().moe_dispatch_rows(
        _ptr(x), _ptr(topk_w), ctypes.byref(shp), _ptr(rows), _ptr(row_weight), _ptr(ws), _nbytes(ws),
        _stream(stream, ws)))


def moe_ep_pack(x, topk_w, shp, n_ranks, capacity, send_rows, send_w, send_counts, ws, stream=None):
    """Expert parallelism, sender: fixed-size send blocks of capacity rows per rank."""
    _check("moe_ep_pack", load().moe_ep_pack(
        _ptr(x), _ptr(topk_w), ctypes.byref(shp), int(n_ranks), int(capacity), _ptr(send_rows), _ptr(send_w),
        _ptr(send_counts), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_ep_receive_metadata(recv_counts, n_ranks, capacity, recv_shp, ws, stream=None):
    """Expert parallelism, receiver: routing metadata of the received blocks from their counts."""
    _check("moe_ep_receive_metadata", load().moe_ep_receive_metadata(
        _ptr(recv_counts), int(n_ranks), int(capacity), ctypes.byref(recv_shp), _ptr(ws), _nbytes(ws),
        _stream(stream, ws)))


def moe_ep_combine(back_rows, shp, n_ranks, capacity, y, ws, stream=None):
    """Expert parallelism, sender: the sum of each token's returned rows."""
    _check("moe_ep_combine", load().moe_ep_combine(
        _ptr(back_rows), ctypes.byref(shp), int(n_ranks), int(capacity), _ptr(y), _ptr(ws), _nbytes(ws),
        _stream(stream, ws)))


def moe_combine_rows(rows, shp, y, ws, stream=None):
    """y[t] = sum of the token's (already weighted) rows, in routed order."""
    _check("moe_combine_rows", load().moe_combine_rows(
        _ptr(rows), ctypes.byref(shp), _ptr(y), _ptr(ws), _nbytes(ws), _stream(stream, ws)))


def moe_get_device_error(ws, stream=None) -> int:
    """Wait for the stream, return and clear the workspace error word (0 = none)."""
    code = ctypes.c_int32()
    st = load().moe_get_device_error(_ptr(ws), ctypes.byref(code), _stream(stream, ws))
    if st not in (MOE_OK, 5):
        raise MoEError("moe_get_device_error", st)
    return int(code.value)


def moe_kernel_launch_count() -> int:
    return int(load().moe_kernel_launch_count())


def moe_packed_weights_size(shp: Shape) -> tuple:
    """Bytes of the tile-packed w1 and w2 for this shape."""
    a, b = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("moe_packed_weights_size", load().moe_packed_weights_size(ctypes.byref(shp), ctypes.byref(a),
                                                                     ctypes.byref(b)))
    return a.value, b.value


def moe_pack_weights(w1, w2, shp: Shape, w1p=None, w2p=None, stream=None):
    """Tile-packed copies of w1 [E, 2I, H] and w2 [E, H, I] (uint8 tensors, allocated when
    not given; either weight may be None to skip it). Pass them to the forward calls with a
    shape made with packed=True."""
    n1, n2 = moe_packed_weights_size(shp)
    like = w1 if w1 is not None else w2
    if w1 is not None and w1p is None:
        w1p = torch.empty(n1, dtype=torch.uint8, device=like.device)
    if w2 is not None and w2p is None:
        w2p = torch.empty(n2, dtype=torch.uint8, device=like.device)
    _check("moe_pack_weights", load().moe_pack_weights(
        _ptr(w1) if w1 is not None else None, _ptr(w2) if w2 is not None else None, ctypes.byref(shp),
        _ptr(w1p) if w1 is not None else None, _ptr(w2p) if w2 is not None else None, _stream(stream, like)))
    return w1p, w2p


def new_workspace(shp: Shape, device=None) -> torch.Tensor:
    """A 256-byte aligned uint8 workspace of the required size, header zeroed."""
    n = moe_workspace_size(shp)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    moe_workspace_init(ws)
    return ws
