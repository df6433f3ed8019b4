"""fp64 CPU oracle of the MegaMoE expert path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the cpu_baseline / reference
legs of ``bench.py`` may import this package. The product library never loads
it. It wraps ``moe_oracle.c`` (plain C, fp64, OpenMP over tokens) through
ctypes; see that file for the definitions and the page sections they follow.

Inputs are torch tensors or numpy arrays. bf16 tensors are passed by their bit
patterns, so the oracle sees their exact values.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_default = None


def compile_source(src: str, out: str) -> str:
    """gcc -O2 -fopenmp: compile one oracle C source into a shared library."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into oracle/liboracle.so unless it is up to date."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def _bind(lib):
    i64, i32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
    vp = ctypes.c_void_p
    lib.oracle_router.argtypes = [i64, i64, i64, i32, vp, vp, vp, vp, i32, i32, f64,
                                  i32, i32, i32, vp, vp, vp, vp, vp, vp]
    lib.oracle_router.restype = ctypes.c_int
    lib.oracle_routing_metadata.argtypes = [i64, i32, i64, vp, vp, vp, vp, vp]
    lib.oracle_routing_metadata.restype = ctypes.c_int64
    lib.oracle_expert_forward.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp, vp, vp,
                                          vp, vp, vp]
    lib.oracle_expert_forward.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_expert_backward.argtypes = [i64, i64, i64, i64, i32, vp, vp, vp, vp, vp, vp,
                                           vp, vp, vp, vp]
    lib.oracle_expert_backward.restype = ctypes.c_int
    lib.oracle_router_backward.argtypes = [i64, i64, i64, i32, vp, vp, vp, i32, i32, f64,
                                           vp, vp, vp, vp, vp, vp]
    lib.oracle_router_backward.restype = ctypes.c_int
    lib.oracle_mx_quantize_bf16.argtypes = [i64, i64, vp, vp, vp]
    lib.oracle_mx_quantize_bf16.restype = ctypes.c_int
    lib.oracle_mx_quantize_f64.argtypes = [i64, i64, vp, vp, vp]
    lib.oracle_mx_quantize_f64.restype = ctypes.c_int
    lib.oracle_expert_forward_mx.argtypes = [i64, i64, i64, i64, i32] + [vp] * 12
    lib.oracle_expert_forward_mx.restype = ctypes.c_int
    lib.oracle_expert_backward_mx.argtypes = [i64, i64, i64, i64, i32] + [vp] * 16
    lib.oracle_expert_backward_mx.restype = ctypes.c_int
    lib.oracle_mx_wgrad.argtypes = [i64, vp, i64, i64, vp, vp, vp]
    lib.oracle_mx_wgrad.restype = ctypes.c_int
    return lib


def _np(a, dtype=None):
    """Host numpy copy of a torch tensor / array; bf16 comes back as uint16 bits."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                a = a.view(torch.int16).numpy().view(np.uint16)
            else:
                a = a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if dtype is not None and a.dtype != dtype:
        a = np.ascontiguousarray(a.astype(dtype))
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class RouterResult:
    topk_idx: np.ndarray    # int32 [T, k], best first
    topk_w: np.ndarray      # float64 [T, k]
    scores: np.ndarray      # float64 [T, E], softmax or sigmoid of the logits
    sel_gap: np.ndarray     # float64 [T], k-th minus (k+1)-th selection score
    group_gap: np.ndarray   # float64 [T], same for groups (+inf without groups)
    aux: float


@dataclass
class Metadata:
    counts: np.ndarray     # int32 [E]
    offsets: np.ndarray    # int32 [E+1]
    perm_slot: np.ndarray  # int32 [offsets[E]]
    row_of: np.ndarray     # int32 [T*k], -1 for dropped slots
    dropped: int


class Oracle:
    """One loaded oracle library (the shipped one, or a test's compiled variant)."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self.lib = _bind(ctypes.CDLL(lib_path))

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def router(self, x, w_r, k, *, score="softmax", normalize=True, scale=1.0, n_group=1,
               topk_group=1, group_topn=2, logit_offset=None, sel_bias=None) -> RouterResult:
        """Scores, (group-limited) top-k, weights and aux for every token of x."""
        xb = _np(x)
        assert xb.dtype == np.uint16, "x must be bf16"
        wr = _np(w_r, np.float32)
        T, H = xb.shape
        E = wr.shape[0]
        off = None if logit_offset is None else _np(logit_offset, np.float32)
        bias = None if sel_bias is None else _np(sel_bias, np.float32)
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float64)
        s = np.empty((T, E), np.float64)
        sg = np.empty((T,), np.float64)
        gg = np.empty((T,), np.float64)
        aux = np.zeros((1,), np.float64)
        rc = self.lib.oracle_router(T, H, E, k, _ptr(xb), _ptr(wr), _ptr(off), _ptr(bias),
                                    0 if score == "softmax" else 1, int(bool(normalize)),
                                    float(scale), int(n_group), int(topk_group), int(group_topn),
                                    _ptr(idx), _ptr(w), _ptr(s), _ptr(sg), _ptr(gg), _ptr(aux))
        if rc != 0:
            raise ValueError("oracle_router rejected its arguments")
        return RouterResult(idx, w, s, sg, gg, float(aux[0]))

    def routing_metadata(self, topk_idx, E) -> Metadata:
        """Per-expert counts, offsets and the stable slot permutation."""
        idx = _np(topk_idx, np.int32)
        T, k = idx.shape
        counts = np.empty((E,), np.int32)
        offsets = np.empty((E + 1,), np.int32)
        perm = np.empty((T * k,), np.int32)
        row_of = np.empty((T * k,), np.int32)
        dropped = self.lib.oracle_routing_metadata(T, k, E, _ptr(idx), _ptr(counts),
                                                   _ptr(offsets), _ptr(perm), _ptr(row_of))
        return Metadata(counts, offsets, perm[: offsets[E]].copy(), row_of, int(dropped))

    def expert_forward(self, x, topk_idx, topk_w, w1, w2, *, want_a=False, want_o=False):
        """y [T, H] float64 (and optionally a / o per slot) for the given routing."""
        xb = _np(x)
        w1b = _np(w1)
        w2b = _np(w2)
        assert xb.dtype == np.uint16 and w1b.dtype == np.uint16 and w2b.dtype == np.uint16
        idx = _np(topk_idx, np.int32)
        w = _np(topk_w, np.float64)
        T, H = xb.shape
        E, twoI, H1 = w1b.shape
        I = twoI // 2
        assert H1 == H and w2b.shape == (E, H, I)
        assert idx.shape == w.shape and idx.shape[0] == T
        k = idx.shape[1]
        y = np.empty((T, H), np.float64)
        a = np.empty((T * k, I), np.float64) if want_a else None
        o = np.empty((T * k, H), np.float64) if want_o else None
        rc = self.lib.oracle_expert_forward(T, H, I, E, k, _ptr(xb), _ptr(idx), _ptr(w),
                                            _ptr(w1b), _ptr(w2b), _ptr(y), _ptr(a), _ptr(o))
        if rc != 0:
            raise ValueError("oracle_expert_forward rejected its arguments")
        if want_a or want_o:
            return y, a, o
        return y

    def expert_backward(self, x, topk_idx, topk_w, w1, w2, dy, *, want_dw=True) -> Backward:
        """dX (expert path), dW1, dW2 and the routing-weight gradient for dY."""
        xb, w1b, w2b, dyb = _np(x), _np(w1), _np(w2), _np(dy)
        assert all(a.dtype == np.uint16 for a in (xb, w1b, w2b, dyb))
        idx = _np(topk_idx, np.int32)
        w = _np(topk_w, np.float64)
        T, H = xb.shape
        E, twoI, _ = w1b.shape
        I = twoI // 2
        k = idx.shape[1]
        dx = np.empty((T, H), np.float64)
        dw1 = np.empty((E, 2 * I, H), np.float64) if want_dw else None
        dw2 = np.empty((E, H, I), np.float64) if want_dw else None
        dtw = np.empty((T, k), np.float64)
        rc = self.lib.oracle_expert_backward(T, H, I, E, k, _ptr(xb), _ptr(idx), _ptr(w), _ptr(w1b),
                                             _ptr(w2b), _ptr(dyb), _ptr(dx), _ptr(dw1), _ptr(dw2),
                                             _ptr(dtw))
        if rc != 0:
            raise ValueError("oracle_expert_backward rejected its arguments")
        return Backward(dx, dw1, dw2, dtw)

    def expert_backward_mx(self, x, xq, xs, topk_idx, topk_w, w1, w1q, w1s, w2, dy, *, want_dw=True,
                           want_slots=False):
        """Backward of the MXFP8 expert precision (see oracle_expert_backward_mx):
        dX (expert path), dW1, dW2 from MXFP8 operands along the routed rows, the
        routing-weight gradient; with want_slots also dH [T*k, 2I] and w a [T*k, I]
        per slot before quantization (as a tuple after the Backward)."""
        xb, w1b, w2b, dyb = _np(x), _np(w1), _np(w2), _np(dy)
        assert all(a.dtype == np.uint16 for a in (xb, w1b, w2b, dyb))
        xqn, xsn = _np(xq, np.uint8), _np(xs, np.uint8)
        w1qn, w1sn = _np(w1q, np.uint8), _np(w1s, np.uint8)
        idx = _np(topk_idx, np.int32)
        w = _np(topk_w, np.float64)
        T, H = xb.shape
        E, twoI, _ = w1b.shape
        I = twoI // 2
        k = idx.shape[1]
        dx = np.empty((T, H), np.float64)
        dw1 = np.empty((E, 2 * I, H), np.float64) if want_dw else None
        dw2 = np.empty((E, H, I), np.float64) if want_dw else None
        dtw = np.empty((T, k), np.float64)
        dh = np.zeros((T * k, 2 * I), np.float64) if want_slots else None
        wa = np.zeros((T * k, I), np.float64) if want_slots else None
        rc = self.lib.oracle_expert_backward_mx(T, H, I, E, k, _ptr(xb), _ptr(xqn), _ptr(xsn), _ptr(idx), _ptr(w),
                                                _ptr(w1b), _ptr(w1qn), _ptr(w1sn), _ptr(w2b), _ptr(dyb), _ptr(dx),
                                                _ptr(dw1), _ptr(dw2), _ptr(dtw), _ptr(dh), _ptr(wa))
        if rc != 0:
            raise ValueError("oracle_expert_backward_mx rejected its arguments")
        if want_slots:
            return Backward(dx, dw1, dw2, dtw), dh, wa
        return Backward(dx, dw1, dw2, dtw)

    def mx_wgrad(self, offsets, a_rows, b_rows):
        """MXFP8 weight gradient of given operands: per expert e (rows offsets[e] ..
        offsets[e+1]-1 of a_rows [R, M] and b_rows [R, N]), Q(A_e)^T Q(B_e) with Q the
        MXFP8 quantization along the rows in blocks of 32 from the expert's first row.
        Returns float64 [E, M, N]. bf16 tensors are taken at their exact values."""
        off = _np(offsets, np.int32)
        A = _np(a_rows)
        B = _np(b_rows)
        A = bf16_bits_to_f64(A) if A.dtype == np.uint16 else np.ascontiguousarray(A, np.float64)
        B = bf16_bits_to_f64(B) if B.dtype == np.uint16 else np.ascontiguousarray(B, np.float64)
        E = len(off) - 1
        M, N = A.shape[1], B.shape[1]
        dw = np.empty((E, M, N), np.float64)
        rc = self.lib.oracle_mx_wgrad(E, _ptr(off), M, N, _ptr(A), _ptr(B), _ptr(dw))
        if rc != 0:
            raise ValueError("oracle_mx_wgrad rejected its arguments")
        return dw

    def mx_quantize(self, a):
        """MXFP8 quantization along the last dimension: (codes uint8, scales uint8 [.., cols/32]).

        `a` is bf16 (tensor) or float64 (array / tensor); any leading shape."""
        arr = _np(a)
        shape = arr.shape
        cols = shape[-1]
        rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
        codes = np.empty(shape, np.uint8)
        scales = np.empty(shape[:-1] + (cols // 32,), np.uint8)
        if arr.dtype == np.uint16:
            rc = self.lib.oracle_mx_quantize_bf16(rows, cols, _ptr(arr), _ptr(codes), _ptr(scales))
        else:
            arr = np.ascontiguousarray(arr, np.float64)
            rc = self.lib.oracle_mx_quantize_f64(rows, cols, _ptr(arr), _ptr(codes), _ptr(scales))
        if rc != 0:
            raise ValueError("oracle_mx_quantize rejected its arguments")
        return codes, scales

    def expert_forward_mx(self, xq, xs, topk_idx, topk_w, w1q, w1s, w2q, w2s, *, want_a=False):
        """y [T, H] float64 of the MXFP8 expert path (optionally a before quantization and
        its codes and scales per slot)."""
        xq, xs = _np(xq, np.uint8), _np(xs, np.uint8)
        w1q, w1s = _np(w1q, np.uint8), _np(w1s, np.uint8)
        w2q, w2s = _np(w2q, np.uint8), _np(w2s, np.uint8)
        idx = _np(topk_idx, np.int32)
        w = _np(topk_w, np.float64)
        T, H = xq.shape
        E, twoI, _ = w1q.shape
        I = twoI // 2
        k = idx.shape[1]
        y = np.empty((T, H), np.float64)
        a = np.empty((T * k, I), np.float64) if want_a else None
        ac = np.empty((T * k, I), np.uint8) if want_a else None
        asc = np.empty((T * k, I // 32), np.uint8) if want_a else None
        rc = self.lib.oracle_expert_forward_mx(T, H, I, E, k, _ptr(xq), _ptr(xs), _ptr(idx), _ptr(w),
                                               _ptr(w1q), _ptr(w1s), _ptr(w2q), _ptr(w2s), _ptr(y),
                                               _ptr(a), _ptr(ac), _ptr(asc))
        if rc != 0:
            raise ValueError("oracle_expert_forward_mx rejected its arguments")
        return (y, a, ac, asc) if want_a else y

    def router_backward(self, x, w_r, topk_idx, topk_w, dtopk_w, *, score="softmax",
                        normalize=True, scale=1.0, logit_offset=None) -> RouterBackward:
        """Logit gradient from the routing-weight gradient, and its dX / dW_r."""
        xb = _np(x)
        wr = _np(w_r, np.float32)
        idx = _np(topk_idx, np.int32)
        w = _np(topk_w, np.float64)
        dw = _np(dtopk_w, np.float64)
        off = None if logit_offset is None else _np(logit_offset, np.float32)
        T, H = xb.shape
        E = wr.shape[0]
        k = idx.shape[1]
        dl = np.empty((T, E), np.float64)
        dxa = np.zeros((T, H), np.float64)
        dwr = np.empty((E, H), np.float64)
        rc = self.lib.oracle_router_backward(T, H, E, k, _ptr(xb), _ptr(wr), _ptr(off),
                                             0 if score == "softmax" else 1, int(bool(normalize)),
                                             float(scale), _ptr(idx), _ptr(w), _ptr(dw), _ptr(dl),
                                             _ptr(dxa), _ptr(dwr))
        if rc != 0:
            raise ValueError("oracle_router_backward rejected its arguments")
        return RouterBackward(dl, dxa, dwr)


@dataclass
class Backward:
    dx: np.ndarray          # float64 [T, H]  (expert path only, router part not added)
    dw1: np.ndarray         # float64 [E, 2I, H] or None
    dw2: np.ndarray         # float64 [E, H, I] or None
    dtopk_w: np.ndarray     # float64 [T, k]


@dataclass
class RouterBackward:
    dlogits: np.ndarray     # float64 [T, E]
    dx_add: np.ndarray      # float64 [T, H] router contribution to dX
    dw_r: np.ndarray        # float64 [E, H]


def default() -> Oracle:
    """The oracle built from moe_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def router(*args, **kwargs) -> RouterResult:
    return default().router(*args, **kwargs)


def routing_metadata(*args, **kwargs) -> Metadata:
    return default().routing_metadata(*args, **kwargs)


def expert_forward(*args, **kwargs):
    return default().expert_forward(*args, **kwargs)


def num_threads() -> int:
    return default().num_threads()


def expert_backward(*args, **kwargs) -> Backward:
    return default().expert_backward(*args, **kwargs)


def router_backward(*args, **kwargs) -> RouterBackward:
    return default().router_backward(*args, **kwargs)


def mx_quantize(*args, **kwargs):
    return default().mx_quantize(*args, **kwargs)


def expert_backward_mx(*args, **kwargs):
    return default().expert_backward_mx(*args, **kwargs)


def mx_wgrad(*args, **kwargs):
    return default().mx_wgrad(*args, **kwargs)


def bf16_bits_to_f64(bits):
    """Exact values of bf16 bit patterns (uint16) as float64."""
    b = np.ascontiguousarray(bits, np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def expert_forward_mx(*args, **kwargs):
    return default().expert_forward_mx(*args, **kwargs)


def e4m3_values():
    """float64 [256]: the value of every E4M3 code (NaN for 0x7F and 0xFF), from the
    format's definition (sign, 4 exponent bits with bias 7, 3 mantissa bits)."""
    v = np.empty(256, np.float64)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            v[c] = np.nan
            continue
        mag = m / 8.0 * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        v[c] = -mag if s else mag           # code 0x80 is -0.0
    return v


def mx_dequantize(codes, scales):
    """Values of an MXFP8 matrix: code value times its block's 2^(scale - 127)."""
    codes = np.asarray(codes)
    scales = np.asarray(scales)
    vals = e4m3_values()[codes]
    blk = np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=-1)
    return vals * blk
