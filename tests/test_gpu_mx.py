"""MXFP8 expert precision (CUDA path through the C ABI) against the fp64 oracle.

Bars: the quantizer's E4M3 codes and E8M0 scales bit-exact (integer output of
exact inputs); the expert path's y within relative Frobenius error 1e-2 and max
abs error 3e-2 * max|y_ref| of the oracle's MXFP8 forward fed the same codes.
The SwiGLU output a is quantized from fp32 on the GPU and from fp64 in the
oracle, so a few of its codes may sit one step apart at rounding boundaries;
those are counted and bounded, not required equal.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import MAX_ABS_FRAC, assert_close_y, kmajor_scales_to_rows, read_metadata, tile_sample_tokens
from moe_expert_router_gb300 import binding as B
from moe_expert_router_gb300.workloads import CONFIGS, MoEConfig, generate, routing_with_counts

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.load()


def gpu_quantize(t):
    """codes [..., cols] and k-block-major scales [cols / 128, ..., 4] of t."""
    codes = torch.empty(t.shape, dtype=torch.uint8, device=DEV)
    scales = B.mx_scales_empty(t.shape, DEV)
    B.moe_mx_quantize(t, codes, scales)
    return codes, scales


@pytest.mark.parametrize("kind", ["normal", "wide_range", "zeros_and_tiny", "saturating"])
def test_quantizer_bit_exact(kind):
    g = torch.Generator(device="cpu").manual_seed(hash(kind) % 1000)
    x = torch.randn((97, 512), generator=g, dtype=torch.float32)
    if kind == "wide_range":
        x = x * torch.exp2(torch.randint(-40, 40, (97, 16), generator=g).float()).repeat_interleave(32, 1)
    elif kind == "zeros_and_tiny":
        x[::3] = 0.0
        x[1::3] *= 2.0 ** -128                        # bf16 subnormal range
        x[5, 64:96] = 0.0
    elif kind == "saturating":
        x *= 100.0
        x[:, ::32] = 1.9 * 2.0 ** 8                   # block maxima with mantissa 1.9: scaled to 486 -> 448
    xb = x.to(torch.bfloat16)
    codes, scales = gpu_quantize(xb.to(DEV))
    rc, rs = oracle.mx_quantize(xb)
    np.testing.assert_array_equal(kmajor_scales_to_rows(scales.cpu().numpy(), rows=xb.shape[0]), rs)
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)


def _cfg(T, H, I, E, k, **kw):
    return MoEConfig("case", T=T, H=H, I=I, E=E, k=k, **kw)


def mx_inputs(cfg, seed=0, idx=None, w=None):
    inp = generate(cfg, seed=seed, device=DEV)
    if idx is None:
        shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)
        ws = B.new_workspace(shp, DEV)
        idx = torch.empty((cfg.T, cfg.k), dtype=torch.int32, device=DEV)
        w = torch.empty((cfg.T, cfg.k), dtype=torch.float32, device=DEV)
        B.moe_router(inp["x"], inp["w_r"], shp, B.router_cfg(cfg.score, cfg.normalize, cfg.scale, cfg.n_group,
                                                             cfg.topk_group, cfg.group_topn),
                     idx, w, ws, logit_offset=inp["logit_offset"], sel_bias=inp["sel_bias"])
    E, I, H = cfg.E, cfg.I, cfg.H
    w1q, w1s = gpu_quantize(inp["w1"].view(E * 2 * I, H))
    w2q, w2s = gpu_quantize(inp["w2"].view(E * H, I))
    # scales k-block-major: [H / 128, E, 2I, 4] and [I / 128, E, H, 4]
    return (inp, idx, w, w1q.view(E, 2 * I, H), w1s.view(H // 128, E, 2 * I, 4), w2q.view(E, H, I),
            w2s.view(I // 128, E, H, 4))


def oracle_weights(inp, cfg, experts=None):
    """The oracle's own MXFP8 quantization of w1 and w2 (of `experts` only when
    given), from the bf16 weights: the codes and scales the oracle's forward is fed."""
    w1, w2 = inp["w1"], inp["w2"]
    if experts is not None:
        sel = torch.as_tensor(experts, dtype=torch.long).to(w1.device)
        w1, w2 = w1[sel], w2[sel]
    w1q, w1s = oracle.mx_quantize(w1.cpu())
    w2q, w2s = oracle.mx_quantize(w2.cpu())
    return w1q, w1s, w2q, w2s


def run_mx(cfg, inp, idx, w, w1q, w1s, w2q, w2s, staged):
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, mxfp8=True)
    ws = B.new_workspace(shp, DEV)
    y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=DEV)
    R = cfg.T * cfg.k
    aq = torch.empty((R, cfg.I), dtype=torch.uint8, device=DEV)
    as_ = B.mx_scales_empty((R, cfg.I), DEV)
    if staged:
        B.moe_routing_metadata(idx, shp, ws)
        B.moe_mx_quantize_dispatch(inp["x"], shp, ws)
        B.moe_dispatch_gemm1_mx(w1q, w1s, shp, aq, as_, ws)
        B.moe_swiglu_gemm2_combine_mx(aq, as_, w, w2q, w2s, shp, y, ws)
    else:
        B.moe_forward_mx(inp["x"], idx, w, w1q, w1s, w2q, w2s, shp, y, ws)
        L = B.moe_workspace_layout(shp)
        aq = ws[L.a_codes:L.a_codes + R * cfg.I].view(R, cfg.I)
        R4 = (R + 3) // 4 * 4
        as_ = ws[L.a_scales:L.a_scales + R4 * cfg.I // 32].view(cfg.I // 128, R4, 4)
    err = B.moe_get_device_error(ws)
    return y, aq, as_, ws, shp, err


CASES = {
    "small": _cfg(256, 256, 256, 8, 2),
    "ragged": _cfg(300, 384, 384, 6, 3),
    "tile_tails": _cfg(200, 512, 512, 4, 2),          # I / 96 and H / 224 leave partial tiles
    "sigmoid_groups": _cfg(128, 256, 640, 16, 4, score="sigmoid", scale=2.5, n_group=4, topk_group=2,
                           sel_bias=True),
    "one_token": _cfg(1, 128, 128, 4, 2),
    # T k = 999: the scale arrays' rows are padded to 1000 (k-block-major words)
    "odd_rows": _cfg(333, 384, 256, 5, 3),
    # the largest E and k: 2048 slots over 1024 experts, most of them empty or one-row
    "e1024_k32": _cfg(64, 128, 128, 1024, 32),
}


def test_quantizing_dispatch_is_the_quantizer_in_routed_order():
    cfg = CASES["ragged"]
    inp, idx, w, *_ = mx_inputs(cfg, seed=6)
    shp = B.shape(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k, mxfp8=True)
    ws = B.new_workspace(shp, DEV)
    B.moe_routing_metadata(idx, shp, ws)
    B.moe_mx_quantize_dispatch(inp["x"], shp, ws)
    L = B.moe_workspace_layout(shp)
    R = cfg.T * cfg.k
    codes = ws[L.x_codes:L.x_codes + R * cfg.H].view(R, cfg.H).cpu().numpy()
    R4 = (R + 3) // 4 * 4
    scales = kmajor_scales_to_rows(ws[L.x_scales:L.x_scales + R4 * cfg.H // 32].view(cfg.H // 128, R4, 4).cpu().numpy(),
                                   rows=R)
    _, _, _, perm, _ = read_metadata(ws, shp)
    rc, rs = oracle.mx_quantize(inp["x"])
    tok = perm // cfg.k
    np.testing.assert_array_equal(codes[: len(perm)], rc[tok])
    np.testing.assert_array_equal(scales[: len(perm)], rs[tok])


@pytest.mark.parametrize("T,H,E,k,drop", [
    (70, 1152, 8, 3, True),     # a full and a partial 1024-column chunk per token; 207 routed rows
    (50, 4224, 6, 2, False),    # 33 k-blocks: the scale transpose takes two column tiles
    (1, 128, 4, 4, True),       # one token, one k-block, a dropped slot
])
def test_quantizing_dispatch_ragged_and_dropped(T, H, E, k, drop):
    """The token-major dispatch at the edges of its tiling: codes and scale words of the
    routed rows [0, routed) are the oracle's quantization of each row's token, and
    the rows past the routed count (those of dropped slots) are left untouched."""
    g = torch.Generator().manual_seed(T + H)
    x = (torch.randn(T, H, generator=g) * 3.0).to(torch.bfloat16)
    idx = torch.stack([torch.randperm(E, generator=g)[:k] for _ in range(T)]).to(torch.int32)
    if drop:
        idx[0, k - 1] = -1
        idx[T // 2, 0] = E
    shp = B.shape(T, H, 128, E, k, mxfp8=True)
    ws = B.new_workspace(shp, DEV)
    L = B.moe_workspace_layout(shp)
    R = T * k
    R4 = (R + 3) // 4 * 4
    ws[L.x_codes:L.x_codes + R * H] = 0xAB
    ws[L.x_scales:L.x_scales + R4 * H // 32] = 0xCD
    B.moe_routing_metadata(idx.to(DEV), shp, ws)
    B.moe_mx_quantize_dispatch(x.to(DEV), shp, ws)
    torch.cuda.synchronize()
    err = B.moe_get_device_error(ws)
    assert bool(err & B.DEVERR_BAD_EXPERT_INDEX) == drop
    codes = ws[L.x_codes:L.x_codes + R * H].view(R, H).cpu().numpy()
    raw = ws[L.x_scales:L.x_scales + R4 * H // 32].view(H // 128, R4, 4).cpu().numpy()
    scales = kmajor_scales_to_rows(raw, rows=R)
    _, _, _, perm, _ = read_metadata(ws, shp)
    n = len(perm)
    assert n == R - (2 if drop else 0)
    rc, rs = oracle.mx_quantize(x)
    tok = perm // k
    np.testing.assert_array_equal(codes[:n], rc[tok])
    np.testing.assert_array_equal(scales[:n], rs[tok])
    assert (codes[n:] == 0xAB).all()
    assert (raw[:, n:R4, :] == 0xCD).all()


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("staged", [True, False])
def test_mx_forward_matches_oracle(name, staged):
    cfg = CASES[name]
    inp, idx, w, w1q, w1s, w2q, w2s = mx_inputs(cfg, seed=2)
    y, aq, as_, ws, shp, err = run_mx(cfg, inp, idx, w, w1q, w1s, w2q, w2s, staged)
    assert err == 0, f"device error word {err:#x}"
    xq, xs = oracle.mx_quantize(inp["x"])
    o1q, o1s, o2q, o2s = oracle_weights(inp, cfg)
    # the weight quantization the GPU path was given is the oracle's, bit for bit
    for gq, oq in ((w1q, o1q), (w2q, o2q)):
        np.testing.assert_array_equal(gq.cpu().numpy(), oq)
    for gs, os_ in ((w1s, o1s), (w2s, o2s)):
        np.testing.assert_array_equal(kmajor_scales_to_rows(gs.cpu().numpy()), os_)
    y_ref, _, ac_ref, as_ref = oracle.expert_forward_mx(xq, xs, idx.cpu(), w.cpu().double(), o1q, o1s, o2q, o2s,
                                                        want_a=True)
    assert_close_y(y, y_ref, "y (MXFP8)")
    # a: codes in routed order on the GPU, in slot order in the oracle
    _, _, _, perm, _ = read_metadata(ws, shp)
    g_codes = aq.cpu().numpy()[: len(perm)]
    r_codes = ac_ref[perm]
    g_sc = kmajor_scales_to_rows(as_.cpu().numpy(), rows=cfg.T * cfg.k)[: len(perm)]
    r_sc = as_ref[perm]
    assert (g_sc != r_sc).mean() <= 0.01, "block scales of a differ too often"
    same = np.repeat(g_sc == r_sc, 32, axis=1)
    vals = oracle.e4m3_values()
    step = np.repeat(np.ldexp(1.0, r_sc.astype(np.int64) - 127 - 9), 32, axis=1)   # one subnormal step
    g_val = vals[g_codes] * step * 512
    r_val = vals[r_codes] * step * 512
    differ = same & (g_codes != r_codes)
    assert differ.mean() <= 0.01, f"{differ.mean():.3%} of a's codes differ"
    # where the block scales agree, a differing code is the neighbouring E4M3 value
    # (a value at a rounding boundary, computed in fp32 here and in fp64 there)
    assert np.all(np.abs(g_val - r_val)[differ] <= np.maximum(0.13 * np.abs(r_val), step)[differ])


def test_mx_unused_experts_with_nan_codes_are_never_read():
    T, H, I, E, k = 96, 256, 256, 8, 2
    cfg = _cfg(T, H, I, E, k)
    counts = [40, 0, 60, 50, 0, 42, 0, 0]
    idx, w = routing_with_counts(counts, T, k, seed=4, device=DEV)
    inp, idx, w, w1q, w1s, w2q, w2s = mx_inputs(cfg, seed=3, idx=idx, w=w)
    y0, *_ = run_mx(cfg, inp, idx, w, w1q, w1s, w2q, w2s, staged=True)
    for e, c in enumerate(counts):
        if c == 0:
            w1q[e] = 0x7F      # E4M3 NaN
            w2q[e] = 0x7F
            w1s[:, e] = 0xFF   # E8M0 NaN (scales are [K / 128, E, rows, 4])
            w2s[:, e] = 0xFF
    y1, *_rest, err = run_mx(cfg, inp, idx, w, w1q, w1s, w2q, w2s, staged=True)
    assert err == 0
    assert torch.isfinite(y1.float()).all()
    assert torch.equal(y0, y1)


def test_mx_bf16_agreement_is_within_quantization_error():
    """Sanity of the precision itself: MXFP8 y stays within a few percent of the bf16 path."""
    cfg = CASES["ragged"]
    inp, idx, w, w1q, w1s, w2q, w2s = mx_inputs(cfg, seed=5)
    y_mx, *_ = run_mx(cfg, inp, idx, w, w1q, w1s, w2q, w2s, staged=True)
    y_bf = oracle.expert_forward(inp["x"].cpu(), idx.cpu(), w.cpu().double(), inp["w1"].cpu(), inp["w2"].cpu())
    rel = np.linalg.norm(y_mx.float().cpu().double().numpy() - y_bf) / np.linalg.norm(y_bf)
    assert 1e-3 < rel < 0.08, rel


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mid", "large_group"])
def test_mx_full_size_sampled(name):
    """A full-size configuration in MXFP8 (one-shot call): y on the tokens of the
    first, middle and last rows of every 256-row tile of every expert (so every
    unit of both MXFP8 GEMMs is reached), plus the first, middle and last
    tokens, against the oracle's MXFP8 forward on its own quantization of x and
    of the weights."""
    cfg = CONFIGS[name]
    inp, idx, w, w1q, w1s, w2q, w2s = mx_inputs(cfg, seed=0)
    y, aq, as_, ws, shp, err = run_mx(cfg, inp, idx, w, w1q, w1s, w2q, w2s, staged=False)
    assert err == 0
    counts, offsets, _, perm, _ = read_metadata(ws, shp)
    toks = torch.as_tensor(tile_sample_tokens(counts, offsets, perm, cfg.k, extra=[0, 1, cfg.T // 2, cfg.T - 1]))
    xq, xs = oracle.mx_quantize(inp["x"][toks.to(DEV)])
    idx_s = idx.cpu()[toks].long()
    used = torch.unique(idx_s)
    remap = torch.full((cfg.E,), -1, dtype=torch.long)
    remap[used] = torch.arange(used.numel())
    o1q, o1s, o2q, o2s = oracle_weights(inp, cfg, experts=used)
    y_ref = oracle.expert_forward_mx(xq, xs, remap[idx_s].to(torch.int32), w.cpu()[toks].double(),
                                     o1q, o1s, o2q, o2s)
    assert_close_y(y.cpu()[toks], y_ref, f"y (MXFP8, {len(toks)} tokens)")


# ------------------------------------------------------------------ MXFP8 training step

def mx_train_step(cfg, inp, idx, w, w1q, w1s, w2q, w2s):
    """The MXFP8 training step through the C ABI: MXFP8 forward saving h, the
    bf16 data-gradient backward on it, MXFP8 weight gradients."""
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.k
    shp = B.shape(T, H, I, E, k, training=True, mxfp8=True)
    ws = B.new_workspace(shp, DEV)
    R = T * k
    aq = torch.empty((R, I), dtype=torch.uint8, device=DEV)
    as_ = B.mx_scales_empty((R, I), DEV)
    h = torch.empty((R, 2 * I), dtype=torch.bfloat16, device=DEV)
    y = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    dw1 = torch.full((E, 2 * I, H), float("nan"), dtype=torch.bfloat16, device=DEV)
    dw2 = torch.full((E, H, I), float("nan"), dtype=torch.bfloat16, device=DEV)
    dtw = torch.full((T, k), float("nan"), dtype=torch.float32, device=DEV)
    B.moe_routing_metadata(idx, shp, ws)
    B.moe_mx_quantize_dispatch(inp["x"], shp, ws)
    B.moe_dispatch_gemm1_mx_train(w1q, w1s, shp, aq, as_, h, ws)
    B.moe_swiglu_gemm2_combine_mx(aq, as_, w, w2q, w2s, shp, y, ws)
    B.moe_backward_stage2_data(inp["dy"], w, inp["w2"], h, shp, ws, dtopk_w=dtw)
    B.moe_backward_stage2_weight_mx(inp["dy"], shp, dw2, ws)
    B.moe_backward_stage1_data(inp["w1"], shp, dx, ws)
    B.moe_backward_stage1_weight_mx(inp["x"], shp, dw1, ws)
    err = B.moe_get_device_error(ws)
    return {"y": y, "h": h, "dx": dx, "dw1": dw1, "dw2": dw2, "dtw": dtw, "err": err, "ws": ws, "shp": shp}


def _with_dy(inp, cfg, seed):
    g = torch.Generator(device=DEV).manual_seed(seed + 100)
    inp["dy"] = torch.randn((cfg.T, cfg.H), generator=g, device=DEV).to(torch.bfloat16)
    return inp


TRAIN_CASES = {
    # about 64 rows per expert: one partial k-block of 128 rows, partial 32-row blocks
    "small": (_cfg(256, 256, 256, 8, 2), None),
    # counts around the 32-row block and 128-row k-block edges, an expert without rows;
    # I = 384 leaves a partial 224-column n-tile of dW2 and 2I = 768 three m-tiles of dW1
    "ragged": (_cfg(320, 256, 384, 8, 2), [0, 1, 33, 128, 129, 300, 5, 44]),
    # 256 rows per expert: two full k-blocks
    "two_kblocks": (_cfg(512, 512, 256, 4, 2), None),
    # 256 experts with about two rows each: 256 padded k-blocks, mostly zero rows
    "many_experts": (_cfg(64, 128, 128, 256, 8), None),
}


# The MXFP8 weight gradients quantize dH and w a, which the GPU keeps in bf16
# while the oracle carries them in fp64. A perturbation delta (relative) of a
# value moves its E4M3 code by one step Delta (2^-4 .. 2^-3 relative) with
# probability about delta / Delta, so the quantized operand differs from the
# oracle's by a relative RMS of about sqrt(delta * Delta); with delta of a bf16
# rounding and the SiLU's approximation (a few 2^-10) that is 1-2 %, which no
# summation averages away. Hence two checks: the weight-gradient kernels against
# the oracle's MXFP8 weight gradient of the GPU's own bf16 operands (the same
# codes on both sides: only the fp32 accumulation and the bf16 output differ),
# and the whole chain against the oracle with the bound MX_WGRAD_REL_FRO.
MX_WGRAD_REL_FRO = 3e-2
MX_WGRAD_MAX_ABS_FRAC = 1e-1
# one bf16 rounding of the output (RMS ~2^-9 / sqrt(3) relative) plus fp32 sums
WGRAD_KERNEL_REL_FRO = 5e-3


def _assert_close_bound(g, r, rel_bound, abs_frac, what):
    g = g.detach().float().cpu().double().numpy() if isinstance(g, torch.Tensor) else np.asarray(g, np.float64)
    r = np.asarray(r, np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    rel = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300)
    assert rel <= rel_bound, f"{what}: relative Frobenius error {rel:.3e} > {rel_bound}"
    assert np.abs(g - r).max() <= abs_frac * np.abs(r).max(), f"{what}: max abs error"
    return rel


def check_wgrad_operands(ws, shp, cfg, idx, inp):
    """The transposed MXFP8 operands the weight gradients read, bit-exact against the
    oracle's quantizer: dY^T and x^T over every expert's rows (the oracle's routing
    metadata), quantized along the rows in 32-row blocks from the expert's first row,
    each expert's segment padded with zero rows to whole 128-row k-blocks. Workspace
    layout (white box): after the padded offsets, codes of dY^T [H, ld], (w a)^T,
    dH^T and x^T [H, ld], then their scales as k-block-major words [ld / 128][C]."""
    H, I, E, k = cfg.H, cfg.I, cfg.E, cfg.k
    md = oracle.routing_metadata(idx.cpu(), E)
    L = B.moe_workspace_layout(shp)
    ld = (cfg.T * k + 128 * E + 127) // 128 * 128
    align = lambda v: (v + 255) // 256 * 256
    codes0 = L.mx_wgrad + align(4 * (E + 1))
    scales0 = codes0 + align((2 * H + 3 * I) * ld)
    operands = {"dY": (0, inp["dy"]), "x": (H + 3 * I, inp["x"])}
    for name, (row_off, src) in operands.items():
        codes = ws[codes0 + row_off * ld:codes0 + (row_off + H) * ld].view(H, ld).cpu().numpy()
        words = ws[scales0 + row_off * (ld // 32):scales0 + (row_off + H) * (ld // 32)].view(ld // 128, H, 4)
        words = words.cpu().numpy()
        kp = 0
        for e in range(E):
            cnt = int(md.counts[e])
            seg = (cnt + 127) // 128 * 128
            if seg == 0:
                continue
            tok = torch.as_tensor(md.perm_slot[md.offsets[e]:md.offsets[e + 1]] // k, dtype=torch.long)
            m = torch.zeros((seg, H), dtype=torch.bfloat16)
            m[:cnt] = src.cpu()[tok]
            rc, rs = oracle.mx_quantize(m.t().contiguous())
            np.testing.assert_array_equal(codes[:, kp:kp + seg], rc, err_msg=f"{name}^T codes, expert {e}")
            blocks = range(kp // 32, (kp + seg) // 32)
            got = np.stack([words[b // 4, :, b % 4] for b in blocks], axis=1)
            np.testing.assert_array_equal(got, rs, err_msg=f"{name}^T scales, expert {e}")
            kp += seg


@pytest.mark.parametrize("name", sorted(TRAIN_CASES))
def test_mx_training_step_matches_oracle(name):
    cfg, counts = TRAIN_CASES[name]
    idx = w = None
    if counts is not None:
        idx, w = routing_with_counts(counts, cfg.T, cfg.k, seed=9, device=DEV)
    check_mx_training(cfg, idx, w, seed=4)


def check_mx_training(cfg, idx=None, w=None, seed=4):
    """The MXFP8 training step against the oracle: the forward, the bf16 data
    gradients and the operands they leave, the weight-gradient kernels on the
    GPU's own operands, and the whole chain."""
    inp, idx, w, w1q, w1s, w2q, w2s = mx_inputs(cfg, seed=seed, idx=idx, w=w)
    inp = _with_dy(inp, cfg, seed)
    out = mx_train_step(cfg, inp, idx, w, w1q, w1s, w2q, w2s)
    assert out["err"] == 0, f"device error word {out['err']:#x}"
    xq, xs = oracle.mx_quantize(inp["x"])
    o1q, o1s, o2q, o2s = oracle_weights(inp, cfg)
    y_ref = oracle.expert_forward_mx(xq, xs, idx.cpu(), w.cpu().double(), o1q, o1s, o2q, o2s)
    assert_close_y(out["y"], y_ref, "y (MXFP8 training forward)")
    b, dh_ref, wa_ref = oracle.expert_backward_mx(inp["x"], xq, xs, idx.cpu(), w.cpu().double(), inp["w1"], o1q,
                                                  o1s, inp["w2"], inp["dy"], want_slots=True)
    # the data-gradient path (bf16): its outputs and the operands it leaves for the weight gradients
    assert_close_y(out["dtw"], b.dtopk_w, "dtopk_w")
    assert_close_y(out["dx"], b.dx, "dX")
    ws, shp = out["ws"], out["shp"]
    _, offsets, _, perm, _ = read_metadata(ws, shp)
    L = B.moe_workspace_layout(shp)
    R, n = cfg.T * cfg.k, len(perm)
    dh = ws[L.dh:L.dh + 2 * R * 2 * cfg.I].view(torch.bfloat16).view(R, 2 * cfg.I)[:n]
    aw = ws[L.aw:L.aw + 2 * R * cfg.I].view(torch.bfloat16).view(R, cfg.I)[:n]
    dyp = ws[L.dyp:L.dyp + 2 * R * cfg.H].view(torch.bfloat16).view(R, cfg.H)[:n]
    assert_close_y(dh, dh_ref[perm], "dH (routed order)")
    assert_close_y(aw, wa_ref[perm], "w a (routed order)")
    tok = torch.as_tensor(perm // cfg.k, dtype=torch.long)
    assert torch.equal(dyp.cpu(), inp["dy"].cpu()[tok])
    check_wgrad_operands(ws, shp, cfg, idx, inp)
    # the MXFP8 weight-gradient kernels on the GPU's own operands
    dw2_k = oracle.mx_wgrad(offsets, dyp, aw)
    dw1_k = oracle.mx_wgrad(offsets, dh, inp["x"].cpu()[tok])
    _assert_close_bound(out["dw2"], dw2_k, WGRAD_KERNEL_REL_FRO, MAX_ABS_FRAC, "dW2 kernel (own operands)")
    _assert_close_bound(out["dw1"], dw1_k, WGRAD_KERNEL_REL_FRO, MAX_ABS_FRAC, "dW1 kernel (own operands)")
    # the whole chain against the oracle
    _assert_close_bound(out["dw2"], b.dw2, MX_WGRAD_REL_FRO, MX_WGRAD_MAX_ABS_FRAC, "dW2 (MXFP8)")
    _assert_close_bound(out["dw1"], b.dw1, MX_WGRAD_REL_FRO, MX_WGRAD_MAX_ABS_FRAC, "dW1 (MXFP8)")
    flat = idx.cpu().reshape(-1)
    for e in range(cfg.E):
        if int((flat == e).sum()) == 0:
            assert not out["dw1"][e].float().abs().max().item()
            assert not out["dw2"][e].float().abs().max().item()


def test_mx_training_weight_gradients_differ_from_bf16_by_quantization_only():
    """Sanity of the precision: the MXFP8 weight gradients stay within a few percent
    of the bf16 backward's and are not identical to them."""
    cfg, _ = TRAIN_CASES["small"]
    inp, idx, w, w1q, w1s, w2q, w2s = mx_inputs(cfg, seed=8)
    inp = _with_dy(inp, cfg, 8)
    out = mx_train_step(cfg, inp, idx, w, w1q, w1s, w2q, w2s)
    b = oracle.expert_backward(inp["x"], idx.cpu(), w.cpu().double(), inp["w1"], inp["w2"], inp["dy"])
    for name, ref in (("dw1", b.dw1), ("dw2", b.dw2)):
        g = out[name].float().cpu().double().numpy()
        rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        assert 1e-3 < rel < 0.1, (name, rel)
