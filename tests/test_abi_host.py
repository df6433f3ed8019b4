"""The C-ABI library on a host without a GPU: it builds, loads, exports every
symbol include/moe.h declares, and its host-only entry points behave.

No compute entry point is called here with valid arguments (that needs a GPU);
argument errors are returned before any CUDA call, so they are checked.
"""
import ctypes
import os
import re

import pytest

from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300 import build as moe_build
from moe_expert_router_gb300.workloads import CONFIGS

HEADER = os.path.join(moe_build.ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    moe_build.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(moe_[a-z_0-9]+)\s*\(", text,
                                 flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("moe_router", "moe_routing_metadata", "moe_dispatch_gemm1",
                 "moe_swiglu_gemm2_combine", "moe_forward", "moe_workspace_size",
                 "moe_get_device_error"):
        assert want in names, names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), f"libmoe.so does not export {name}"
    assert set(names) == set(B._SIG), "binding and header disagree"


def test_library_does_not_link_the_oracle():
    data = open(moe_build.LIB_PATH, "rb").read()
    assert b"oracle_" not in data and b"liboracle" not in data


def test_workspace_size_and_layout(lib):
    for cfg in CONFIGS.values():
        shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
        n = B.moe_workspace_size(shp)
        L = B.moe_workspace_layout(shp)
        R = cfg.T * cfg.k
        assert L.total == n
        offs = [L.counts, L.offsets, L.mt_prefix, L.perm_slot, L.row_of, L.meta, L.router, L.a, L.obuf]
        assert all(o % 256 == 0 for o in offs) and offs == sorted(offs) and L.err == 0
        assert L.offsets - L.counts >= 4 * cfg.E
        assert L.row_of - L.perm_slot >= 4 * R
        assert L.a - L.router >= 4 * cfg.T * cfg.E + 8 * cfg.E
        assert L.obuf - L.a >= 2 * R * cfg.I
        assert n - L.obuf >= 2 * R * cfg.H


@pytest.mark.parametrize("bad,status", [
    ((4, 60, 64, 4, 2), 2),      # H % 8
    ((4, 64, 36, 4, 2), 2),      # I % 8
    ((4, 64, 64, 4, 5), 2),      # k > E
    ((4, 64, 64, 2048, 2), 2),   # E > 1024
    ((4, 64, 64, 64, 33), 2),    # k > 32
    ((-1, 64, 64, 4, 2), 1),     # negative T
    ((4, 0, 64, 4, 2), 1),       # H = 0
])
def test_shape_validation(lib, bad, status):
    n = ctypes.c_size_t()
    shp = B.shape(*bad)
    assert lib.moe_workspace_size(ctypes.byref(shp), ctypes.byref(n)) == status


def test_null_arguments_rejected_before_any_device_call(lib):
    shp = B.shape(16, 64, 64, 4, 2)
    cfg = B.router_cfg()
    assert lib.moe_router(None, None, None, None, ctypes.byref(shp), ctypes.byref(cfg), None, None,
                          None, None, 0, None) == 1
    assert lib.moe_forward(None, None, None, None, None, ctypes.byref(shp), None, None, 0, None) == 1
    assert lib.moe_routing_metadata(None, ctypes.byref(shp), None, 0, None) == 1
    assert lib.moe_dispatch_gemm1(None, None, ctypes.byref(shp), None, None, 0, None) == 1
    assert lib.moe_swiglu_gemm2_combine(None, None, None, ctypes.byref(shp), None, None, 0,
                                        None) == 1
    assert lib.moe_get_device_error(None, None, None) == 1
    assert lib.moe_route_logits(None, None, None, ctypes.byref(shp), ctypes.byref(cfg), None, None, None,
                                None, 0, None) == 1
    assert lib.moe_dispatch_rows(None, None, ctypes.byref(shp), None, None, None, 0, None) == 1
    assert lib.moe_combine_rows(None, ctypes.byref(shp), None, None, 0, None) == 1
    # misaligned workspace and a too-small workspace (host checks, no device touched)
    x = ctypes.c_void_p(1 << 20)
    assert lib.moe_routing_metadata(x, ctypes.byref(shp), ctypes.c_void_p((1 << 20) + 16), 1 << 30,
                                    None) == 1
    assert lib.moe_routing_metadata(x, ctypes.byref(shp), ctypes.c_void_p(1 << 20), 256, None) == 4


def test_router_config_validation(lib):
    shp = B.shape(16, 64, 64, 64, 8)
    p = ctypes.c_void_p(1 << 20)
    for cfg, want in [(B.router_cfg(n_group=7, topk_group=2), 1),     # E % n_group
                      (B.router_cfg(n_group=8, topk_group=9), 1),     # topk_group > n_group
                      (B.router_cfg(n_group=16, topk_group=1), 1),    # 1 group of 4 experts < k = 8
                      (B.router_cfg(n_group=64, topk_group=4), 2),    # n_group > 32
                      (B.RouterCfg(7, 1, 1.0, 1, 1, 2), 1)]:          # bad score function
        st = lib.moe_router(p, p, None, None, ctypes.byref(shp), ctypes.byref(cfg), p, p, None, p,
                            1 << 40, None)
        assert st == want, (cfg.n_group, cfg.topk_group, st)


def test_status_strings_and_counter(lib):
    for s in range(6):
        assert B.load().moe_status_string(s)
    assert B.moe_kernel_launch_count() >= 0


def test_training_workspace_layout(lib):
    for cfg in CONFIGS.values():
        R = cfg.T * cfg.k
        base = B.moe_workspace_layout(B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
        assert base.dh == base.aw == base.dtw_part == base.dlogits == base.xp == base.dyp == base.dwr_part == base.total
        L = B.moe_workspace_layout(B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, training=True))
        offs = [L.obuf, L.dh, L.aw, L.dtw_part, L.dlogits, L.xp, L.dyp, L.dwr_part, L.total]
        assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
        assert L.obuf == base.obuf                      # the forward regions do not move
        assert L.aw - L.dh >= 2 * R * 2 * cfg.I
        assert L.dtw_part - L.aw >= 2 * R * cfg.I
        assert L.dlogits - L.dtw_part >= 4 * R * ((cfg.I + 255) // 256)
        assert L.xp - L.dlogits >= 4 * cfg.T * cfg.E
        assert L.dyp - L.xp >= 2 * R * cfg.H
        assert L.dwr_part - L.dyp >= 2 * R * cfg.H
        assert L.total - L.dwr_part >= 4 * 8 * cfg.E * cfg.H


def test_training_calls_need_a_training_workspace(lib):
    p = ctypes.c_void_p(1 << 20)
    cfg = B.router_cfg()
    plain = B.shape(16, 64, 64, 4, 2)
    train = B.shape(16, 64, 64, 4, 2, training=True)
    big = 1 << 40
    # a forward-only shape: rejected on the host before any device call
    assert lib.moe_dispatch_gemm1_train(p, p, ctypes.byref(plain), p, p, p, big, None) == 1
    assert lib.moe_backward_stage2_data(p, p, p, p, ctypes.byref(plain), p, p, big, None) == 1
    assert lib.moe_backward_stage2_weight(p, ctypes.byref(plain), p, p, big, None) == 1
    assert lib.moe_router_backward(p, p, p, p, p, ctypes.byref(plain), ctypes.byref(cfg), p, p, big,
                                   None) == 1
    assert lib.moe_backward_stage1_data(p, None, None, None, ctypes.byref(plain), p, p, big, None) == 1
    assert lib.moe_backward_stage1_weight(p, ctypes.byref(plain), p, p, big, None) == 1
    # missing outputs / inputs
    assert lib.moe_router_train(p, p, None, None, ctypes.byref(train), ctypes.byref(cfg), p, p, None,
                                None, p, big, None) == 1
    assert lib.moe_dispatch_gemm1_train(p, p, ctypes.byref(train), p, None, p, big, None) == 1
    assert lib.moe_backward_stage2_data(p, p, p, None, ctypes.byref(train), None, p, big, None) == 1
    assert lib.moe_backward_stage2_weight(p, ctypes.byref(train), None, p, big, None) == 1
    assert lib.moe_backward_stage1_data(p, p, None, ctypes.byref(cfg), ctypes.byref(train), p, p, big,
                                        None) == 1     # w_r without topk_idx
    assert lib.moe_backward(p, p, None, p, p, p, p, p, p, ctypes.byref(train), ctypes.byref(cfg), p, p, p,
                            p, p, p, big, None) == 1   # w_r without logits
    # unknown shape flags
    bad = B.Shape(16, 64, 64, 4, 2, 8)
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == 1


def test_mxfp8_layout_and_argument_checks(lib):
    for cfg in CONFIGS.values():
        if cfg.H % 128 or cfg.I % 128:
            continue
        R = cfg.T * cfg.k
        base = B.moe_workspace_layout(B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k))
        assert base.x_codes == base.a_scales == base.total
        L = B.moe_workspace_layout(B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, mxfp8=True))
        offs = [L.dlogits, L.x_codes, L.x_scales, L.a_codes, L.a_scales, L.total]
        assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
        assert L.x_scales - L.x_codes >= R * cfg.H
        assert L.a_codes - L.x_scales >= R * cfg.H // 32
        assert L.a_scales - L.a_codes >= R * cfg.I
        assert L.total - L.a_scales >= R * cfg.I // 32
    p = ctypes.c_void_p(1 << 20)
    big = 1 << 40
    shp = B.shape(16, 256, 256, 4, 2, mxfp8=True)
    odd = B.shape(16, 192, 256, 4, 2, mxfp8=True)           # H % 128 != 0
    assert lib.moe_mx_quantize(p, 4, 48, p, p, None) == 1     # cols % 128
    assert lib.moe_mx_quantize(p, 4, 64, p, p, None) == 1
    assert lib.moe_mx_quantize(None, 4, 128, p, p, None) == 1
    assert lib.moe_dispatch_gemm1_mx(p, p, ctypes.byref(odd), p, p, p, big, None) == 2
    assert lib.moe_dispatch_gemm1_mx(p, p, ctypes.byref(shp), p, None, p, big, None) == 1
    assert lib.moe_mx_quantize_dispatch(p, ctypes.byref(odd), p, big, None) == 2
    assert lib.moe_mx_quantize_dispatch(None, ctypes.byref(shp), p, big, None) == 1
    assert lib.moe_swiglu_gemm2_combine_mx(p, p, p, p, p, ctypes.byref(odd), p, p, big, None) == 2
    plain = B.shape(16, 256, 256, 4, 2)
    assert lib.moe_forward_mx(p, p, p, p, p, p, p, ctypes.byref(plain), p, p, big, None) == 1


def test_packed_weight_sizes_and_flag_checks(lib):
    for cfg in CONFIGS.values():
        n1, n2 = B.moe_packed_weights_size(B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, packed=True))
        assert n1 == 32768 * cfg.E * -(-cfg.I // 128) * -(-cfg.H // 64)
        assert n2 == 32768 * cfg.E * -(-cfg.H // 256) * -(-cfg.I // 64)
        assert n1 >= 2 * cfg.E * 2 * cfg.I * cfg.H and n2 >= 2 * cfg.E * cfg.H * cfg.I
    size = ctypes.c_size_t(0)
    for bad in (B.shape(16, 64, 64, 4, 2, training=True, packed=True),
                B.shape(16, 128, 128, 4, 2, mxfp8=True, packed=True)):
        assert lib.moe_workspace_size(ctypes.byref(bad), ctypes.byref(size)) == 2
    shp = B.shape(16, 64, 64, 4, 2, packed=True)
    p = ctypes.c_void_p(1 << 20)
    # source and destination must come in pairs (checked before any device call)
    assert lib.moe_pack_weights(p, None, ctypes.byref(shp), None, None, None) == 1
    assert lib.moe_pack_weights(None, p, ctypes.byref(shp), None, None, None) == 1
    misaligned = ctypes.c_void_p((1 << 20) + 8)
    assert lib.moe_pack_weights(p, None, ctypes.byref(shp), misaligned, None, None) == 1


def test_mx_scale_layout_helpers():
    """The k-block-major scale buffers (rows rounded up to 4) and the test-side
    re-layout to the oracle's row-major scales, on host tensors (no device call)."""
    import numpy as np
    import torch
    from gpu_helpers import kmajor_scales_to_rows
    assert tuple(B.mx_scales_empty((5, 3, 256), "cpu").shape) == (2, 16, 4)   # 15 rows -> 16
    assert tuple(B.mx_scales_empty((2, 8, 384), "cpu").shape) == (3, 2, 8, 4)
    # byte j of word [kb][r] is the scale of columns 128 kb + 32 j .. of row r
    rows, cols = 6, 512
    rs = np.arange(rows * cols // 32, dtype=np.uint8).reshape(rows, cols // 32)
    km = np.zeros((cols // 128, 8, 4), np.uint8)
    for r in range(rows):
        for c in range(cols // 32):
            km[c // 4, r, c % 4] = rs[r, c]
    np.testing.assert_array_equal(kmajor_scales_to_rows(km, rows=rows), rs)
    # a scale buffer of the wrong size is refused before any library call
    t = torch.zeros((6, 512), dtype=torch.bfloat16)
    codes = torch.empty((6, 512), dtype=torch.uint8)
    with pytest.raises(ValueError):
        B.moe_mx_quantize(t, codes, torch.empty((6 * 16,), dtype=torch.uint8))
