// moe_abi.cu -- the extern "C" entry points declared in include/moe.h:
// argument validation, workspace carving, TMA descriptor encoding and the
// kernel launches of each stage. No allocation, no host synchronisation
// (except moe_get_device_error), no CPU fallback.
#include <atomic>
#include <mutex>

#include "internal.cuh"

namespace moe {

namespace {

std::atomic<uint64_t> g_launches{0};

constexpr int kMaxDevices = 64;
struct DeviceState {
    bool ready = false;
    moe_status_t status = MOE_OK;
    int num_sms = 0;
};
std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Per-device set-up: check for an sm_103 GPU, cache the SM count, raise the
// dynamic shared memory limits. A device is marked ready only once this
// succeeded (an unsupported architecture is remembered); a failed CUDA call is
// retried by the next entry point, and only the error it raised is cleared.
moe_status_t device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            d.status = MOE_ERR_UNSUPPORTED;
        } else if (setup_metadata_kernels() != cudaSuccess || setup_gemm_kernels() != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        } else {
            d.num_sms = sms;
            d.status = MOE_OK;
        }
        d.ready = true;
    }
    *out = &d;
    return d.status;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_shape(const moe_shape_t *s) {
    if (s == nullptr) return MOE_ERR_INVALID_ARG;
    if (s->T < 0 || s->H <= 0 || s->I <= 0 || s->E <= 0 || s->k <= 0 ||
        (s->flags & ~(MOE_SHAPE_TRAINING | MOE_SHAPE_MXFP8 | MOE_SHAPE_PACKED_WEIGHTS)) != 0)
        return MOE_ERR_INVALID_ARG;
    if ((s->flags & MOE_SHAPE_PACKED_WEIGHTS) && (s->flags & (MOE_SHAPE_TRAINING | MOE_SHAPE_MXFP8)))
        return MOE_ERR_UNSUPPORTED;
    if (s->k > 32 || s->k > s->E || s->E > 1024) return MOE_ERR_UNSUPPORTED;
    if (s->H % 8 != 0 || s->I % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->T * s->k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (s->E * 2 * s->I >= (int64_t(1) << 31) || s->E * s->H >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (s->H >= (int64_t(1) << 31) || s->I >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// Columns of the MXFP8 weight-gradient operands: every expert's rows padded to
// whole 128-row k-blocks, at most T*k + 128 E in all (a multiple of 128).
size_t mx_wgrad_ld(const moe_shape_t &s) {
    return (static_cast<size_t>(s.T) * s.k + 128 * static_cast<size_t>(s.E) + 127) / 128 * 128;
}

moe_ws_layout_t make_layout(const moe_shape_t &s) {
    const size_t T = s.T, H = s.H, I = s.I, E = s.E, R = s.T * s.k;
    moe_ws_layout_t L;
    size_t off = kWsHeaderBytes;
    L.err = 0;
    L.counts = off;    off = align256(off + 4 * E);
    L.offsets = off;   off = align256(off + 4 * (E + 1));
    L.mt_prefix = off; off = align256(off + 4 * (E + 1));
    L.perm_slot = off; off = align256(off + 4 * R);
    L.row_of = off;    off = align256(off + 4 * R);
    L.meta = off;      off = align256(off + 4 * E * ((R + kMetaChunk - 1) / kMetaChunk));
    L.router = off;    off = align256(off + router_scratch_bytes(T, H, E, router_splits(T, H, E)));
    L.a = off;         off = align256(off + 2 * R * I);
    L.obuf = off;      off = align256(off + 2 * R * H);
    L.combine = off;   off = align256(off + 4 * T * ((H + kBN - 1) / kBN));
    if (s.flags & MOE_SHAPE_TRAINING) {
        L.dh = off;       off = align256(off + 2 * R * 2 * I);
        L.aw = off;       off = align256(off + 2 * R * I);
        L.dtw_part = off; off = align256(off + 4 * R * ((I + kBN - 1) / kBN));
        L.dlogits = off;  off = align256(off + 4 * T * E);
        L.xp = off;       off = align256(off + 2 * R * H);
        L.dyp = off;      off = align256(off + 2 * R * H);
        L.dwr_part = off; off = align256(off + 4 * static_cast<size_t>(kDwrSegments) * E * H);
    } else {
        L.dh = L.aw = L.dtw_part = L.dlogits = L.xp = L.dyp = L.dwr_part = off;
    }
    if (s.flags & MOE_SHAPE_MXFP8) {
        L.x_codes = off;  off = align256(off + R * H);
        // scales: k-block-major words over the routed rows rounded up to 4
        L.x_scales = off; off = align256(off + mx_rows(R) * (H / 32));
        L.a_codes = off;  off = align256(off + R * I);
        L.a_scales = off; off = align256(off + mx_rows(R) * (I / 32));
    } else {
        L.x_codes = L.x_scales = L.a_codes = L.a_scales = off;
    }
    if ((s.flags & MOE_SHAPE_MXFP8) && (s.flags & MOE_SHAPE_TRAINING)) {
        // the weight gradients' operands quantized along the routed rows, transposed:
        // dY, w a, dH and x, each [columns, mx_wgrad_ld(s)] codes + [columns, ld / 32] scales
        const size_t ld = mx_wgrad_ld(s);
        L.mx_wgrad = off;
        off = align256(off + 4 * (E + 1));
        off = align256(off + (2 * H + 3 * I) * ld);
        off = align256(off + (2 * H + 3 * I) * (ld / 32));
    } else {
        L.mx_wgrad = off;
    }
    L.total = off;
    return L;
}

// MXFP8 weight-gradient operands (training + MXFP8 workspaces): the padded row
// offsets, then codes and scales of dY^T [H, ld], (w a)^T [I, ld], dH^T [2I, ld]
// and x^T [H, ld], ld = mx_wgrad_ld.
struct MxWgradWs {
    int32_t *kpad;
    uint8_t *dy_c, *aw_c, *dh_c, *x_c;
    uint8_t *dy_s, *aw_s, *dh_s, *x_s;
    int64_t ld;
};

MxWgradWs carve_mx_wgrad(void *ws, const moe_shape_t &s) {
    const moe_ws_layout_t L = make_layout(s);
    const size_t H = s.H, I = s.I, E = s.E;
    MxWgradWs m;
    m.ld = static_cast<int64_t>(mx_wgrad_ld(s));
    uint8_t *b = static_cast<uint8_t *>(ws) + L.mx_wgrad;
    m.kpad = reinterpret_cast<int32_t *>(b);
    uint8_t *c = b + align256(4 * (E + 1));
    m.dy_c = c;
    m.aw_c = m.dy_c + H * m.ld;
    m.dh_c = m.aw_c + I * m.ld;
    m.x_c = m.dh_c + 2 * I * m.ld;
    uint8_t *sc = c + align256((2 * H + 3 * I) * m.ld);
    const size_t lds = m.ld / 32;
    m.dy_s = sc;
    m.aw_s = m.dy_s + H * lds;
    m.dh_s = m.aw_s + I * lds;
    m.x_s = m.dh_s + 2 * I * lds;
    return m;
}

// Workspace header words (see internal.cuh for bytes 0-32).
constexpr size_t kHdrSchedDA = 40, kHdrSchedDX = 48, kHdrSchedDW2 = 56, kHdrSchedDW1 = 64;
constexpr size_t kHdrSchedDW2Mx = 72, kHdrSchedDW1Mx = 80;

struct Ws {
    int32_t *err, *ticket, *counts, *offsets, *mt_prefix, *perm_slot, *row_of, *sched1, *sched2;
    int32_t *meta, *meta_ticket;
    int32_t *sched_da, *sched_dx, *sched_dw2, *sched_dw1;
    RouterScratch router;
    __nv_bfloat16 *a, *obuf;
    int32_t *combine;           // stage 2's fused-combine counters [T, ceil(H / 256)]
    __nv_bfloat16 *dh, *aw;     // training only
    float *dtw_part, *dlogits;  // training only
    __nv_bfloat16 *xp, *dyp;    // training only: x and dY rows in routed order
    float *dwr_part;            // training only: partial sums of dW_r
    uint8_t *x_codes, *x_scales, *a_codes, *a_scales;   // MXFP8 only
    bool training, mxfp8;
};

Ws carve(void *ws, const moe_shape_t &s) {
    const moe_ws_layout_t L = make_layout(s);
    uint8_t *b = static_cast<uint8_t *>(ws);
    Ws w;
    w.err = reinterpret_cast<int32_t *>(b + L.err);
    w.ticket = reinterpret_cast<int32_t *>(b + 4);
    w.counts = reinterpret_cast<int32_t *>(b + L.counts);
    w.offsets = reinterpret_cast<int32_t *>(b + L.offsets);
    w.mt_prefix = reinterpret_cast<int32_t *>(b + L.mt_prefix);
    w.perm_slot = reinterpret_cast<int32_t *>(b + L.perm_slot);
    w.row_of = reinterpret_cast<int32_t *>(b + L.row_of);
    w.meta = reinterpret_cast<int32_t *>(b + L.meta);
    w.meta_ticket = reinterpret_cast<int32_t *>(b + 32);
    w.sched1 = reinterpret_cast<int32_t *>(b + 8);
    w.sched2 = reinterpret_cast<int32_t *>(b + 16);
    w.sched_da = reinterpret_cast<int32_t *>(b + kHdrSchedDA);
    w.sched_dx = reinterpret_cast<int32_t *>(b + kHdrSchedDX);
    w.sched_dw2 = reinterpret_cast<int32_t *>(b + kHdrSchedDW2);
    w.sched_dw1 = reinterpret_cast<int32_t *>(b + kHdrSchedDW1);
    w.router = carve_router_scratch(b + L.router, s.T, s.H, s.E, router_splits(s.T, s.H, s.E),
                                    w.ticket, reinterpret_cast<int32_t *>(b + 24));
    w.a = reinterpret_cast<__nv_bfloat16 *>(b + L.a);
    w.obuf = reinterpret_cast<__nv_bfloat16 *>(b + L.obuf);
    w.combine = reinterpret_cast<int32_t *>(b + L.combine);
    w.training = (s.flags & MOE_SHAPE_TRAINING) != 0;
    w.dh = reinterpret_cast<__nv_bfloat16 *>(b + L.dh);
    w.aw = reinterpret_cast<__nv_bfloat16 *>(b + L.aw);
    w.dtw_part = reinterpret_cast<float *>(b + L.dtw_part);
    w.dlogits = reinterpret_cast<float *>(b + L.dlogits);
    w.xp = reinterpret_cast<__nv_bfloat16 *>(b + L.xp);
    w.dyp = reinterpret_cast<__nv_bfloat16 *>(b + L.dyp);
    w.dwr_part = reinterpret_cast<float *>(b + L.dwr_part);
    w.mxfp8 = (s.flags & MOE_SHAPE_MXFP8) != 0;
    w.x_codes = b + L.x_codes;
    w.x_scales = b + L.x_scales;
    w.a_codes = b + L.a_codes;
    w.a_scales = b + L.a_scales;
    return w;
}

moe_status_t check_ws(const moe_shape_t &s, const void *ws, size_t ws_bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < make_layout(s).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// A GemmLaunch with the metadata pointers of the workspace filled in.
GemmLaunch base_launch(const moe_shape_t &s, const Ws &w, const DeviceState &d) {
    GemmLaunch p{};
    p.counts = w.counts;
    p.offsets = w.offsets;
    p.mt_prefix = w.mt_prefix;
    p.perm_slot = w.perm_slot;
    p.err = w.err;
    p.E = static_cast<int>(s.E);
    p.k = s.k;
    p.R = static_cast<int>(s.T * s.k);
    p.T = static_cast<int>(s.T);
    p.num_sms = d.num_sms;
    return p;
}

// Stage 1: the dispatch (x rows copied into routed order), then tensor maps +
// launch (metadata must already be in ws). The dispatched rows go to obuf, idle
// until stage 2 writes its rows there, or with h (training) to xp, which the
// backward reads again. With h, the pre-activation is stored too (a, h gate and
// h up in 32 x 32 boxes).
moe_status_t run_gemm1(const moe_shape_t &s, const void *x, const void *w1, void *a, void *h, const Ws &w,
                       const DeviceState &d, cudaStream_t st) {
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    __nv_bfloat16 *xp = h ? w.xp : w.obuf;
    CUtensorMap tm_x, tm_w1, tm_out, tm_hg, tm_hu;
    const uint32_t box = h ? 32 : 64;
    if (!encode_bf16_2d(&tm_x, xp, s.H, R, kBK, 128) ||
        !encode_bf16_2d(&tm_w1, w1, s.H, static_cast<uint64_t>(s.E) * 2 * s.I, kBK, 128) ||
        !encode_bf16_2d(&tm_out, a, s.I, R, box, 32))
        return MOE_ERR_CUDA;
    if (launch_dispatch_rows(static_cast<const __nv_bfloat16 *>(x), w.row_of, s.T, s.k, s.H, xp, nullptr, nullptr,
                             st) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (h && (!encode_bf16_2d_strided(&tm_hg, h, s.I, R, 2 * s.I, 32, 32) ||
              !encode_bf16_2d_strided(&tm_hu, static_cast<__nv_bfloat16 *>(h) + s.I, s.I, R, 2 * s.I, 32, 32)))
        return MOE_ERR_CUDA;
    GemmLaunch p = base_launch(s, w, d);
    p.tm_a = &tm_x;
    p.tm_b = &tm_w1;
    if (s.flags & MOE_SHAPE_PACKED_WEIGHTS) {   // w1 is the packed tile array
        p.bpack = static_cast<const uint8_t *>(w1);
        p.tm_b = &tm_x;
    }
    p.tm_out = &tm_out;
    p.tm_out2 = h ? &tm_hg : nullptr;
    p.tm_out3 = h ? &tm_hu : nullptr;
    p.sched = w.sched1;
    p.out = static_cast<__nv_bfloat16 *>(a);
    p.out2 = static_cast<__nv_bfloat16 *>(h);
    p.out3 = h ? static_cast<__nv_bfloat16 *>(h) + s.I : nullptr;
    p.K = static_cast<int>(s.H);
    p.n_out = static_cast<int>(s.I);
    p.n_tile = kBN / 2;
    p.b_rows = static_cast<int>(2 * s.I);
    p.half = static_cast<int>(s.I);
    p.out_ld = static_cast<int>(2 * s.I);
    p.save_h = h != nullptr;
    return cuda_status(launch_gemm1_swiglu(p, st));
}

// Where stage 2 sums each token's k rows. Fused into its epilogue (counters set
// by the routing metadata) the sum costs no launch and no second pass, but each
// epilogue warp then waits for its stores to land and reads the completed
// tokens' rows back before it can take the next accumulator: the more rows a
// unit holds, the longer that delays the MMAs. Measured fused against the
// combine kernel: mid (384 rows per expert) stage 2 + combine 0.149 -> 0.192 ms,
// large_group (256) 1.859 -> 1.933 ms, its 32-expert slice slower as well, while
// zipf_decode (4 rows per expert) gains, 0.184 -> 0.167 ms. Fused while the
// experts average at most kFusedCombineMaxRowsPerExpert routed rows.
constexpr int64_t kFusedCombineMaxRowsPerExpert = 64;
bool fused_combine(const moe_shape_t &s) { return s.T * s.k <= kFusedCombineMaxRowsPerExpert * s.E; }

// Stage 2: GEMM2 with the weighted scatter, then the k-way combine (fused into
// the GEMM's epilogue for few routed rows, else the combine kernel).
moe_status_t run_gemm2(const moe_shape_t &s, const void *a, const float *topk_w, const void *w2,
                       void *y, const Ws &w, const DeviceState &d, cudaStream_t st) {
    CUtensorMap tm_a, tm_w2, tm_out;
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    if (!encode_bf16_2d(&tm_a, a, s.I, R, kBK, 128)) return MOE_ERR_CUDA;
    if (!encode_bf16_2d(&tm_w2, w2, s.I, static_cast<uint64_t>(s.E) * s.H, kBK, 256))
        return MOE_ERR_CUDA;
    if (!encode_bf16_2d(&tm_out, w.obuf, s.H, R, 64, 32)) return MOE_ERR_CUDA;
    GemmLaunch p = base_launch(s, w, d);
    p.tm_a = &tm_a;
    p.tm_b = &tm_w2;
    if (s.flags & MOE_SHAPE_PACKED_WEIGHTS) {   // w2 is the packed tile array
        p.bpack = static_cast<const uint8_t *>(w2);
        p.tm_b = &tm_a;
    }
    p.tm_out = &tm_out;
    p.sched = w.sched2;
    p.topk_w = topk_w;
    p.out = w.obuf;
    const bool fused = fused_combine(s);
    if (fused) {
        p.row_of = w.row_of;
        p.y = static_cast<__nv_bfloat16 *>(y);
        p.ccnt = w.combine;
    }
    p.K = static_cast<int>(s.I);
    p.n_out = static_cast<int>(s.H);
    p.n_tile = kBN;
    p.b_rows = static_cast<int>(s.H);
    moe_status_t r = cuda_status(launch_gemm2_scatter(p, st));
    if (r != MOE_OK || fused) return r;
    CombineLaunch c;
    c.obuf = w.obuf;
    c.row_of = w.row_of;
    c.y = static_cast<__nv_bfloat16 *>(y);
    c.T = static_cast<int>(s.T);
    c.H = static_cast<int>(s.H);
    c.k = s.k;
    return cuda_status(launch_combine(c, st));
}

// Stage 1 in MXFP8: the dispatched E4M3 x rows (routed order, in ws) and E4M3
// w1 through TMA, scales into tensor memory per stage; the epilogue quantizes a
// per 32 columns.
moe_status_t run_gemm1_mx(const moe_shape_t &s, const void *w1q, const void *w1s, void *aq, void *as, void *h,
                          const Ws &w, const DeviceState &d, cudaStream_t st) {
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    CUtensorMap tm_x, tm_w1, tm_xs, tm_w1s;
    if (!encode_u8_2d(&tm_x, w.x_codes, s.H, R, 128, 128) ||
        !encode_u8_2d(&tm_w1, w1q, s.H, static_cast<uint64_t>(s.E) * 2 * s.I, 128, 96) ||
        !encode_sf_words(&tm_xs, w.x_scales, mx_rows(R), s.H / 128, kSfBoxRowsA) ||
        !encode_sf_words(&tm_w1s, w1s, static_cast<uint64_t>(s.E) * 2 * s.I, s.H / 128, 96))
        return MOE_ERR_CUDA;
    GemmLaunch p = base_launch(s, w, d);
    p.tm_a = &tm_x;
    p.tm_b = &tm_w1;
    p.tm_out = &tm_w1;
    p.tm_sfa = &tm_xs;
    p.tm_sfb = &tm_w1s;
    p.sf_rows = static_cast<int64_t>(mx_rows(R));         // the scale rows of x and a
    p.sched = w.sched1;
    p.out = static_cast<__nv_bfloat16 *>(aq);             // E4M3 codes [R, I]
    p.out_sf = static_cast<uint8_t *>(as);
    p.out2 = static_cast<__nv_bfloat16 *>(h);             // training: h gate / up halves [R, 2I]
    p.out3 = h ? static_cast<__nv_bfloat16 *>(h) + s.I : nullptr;
    p.out_ld = static_cast<int>(2 * s.I);
    p.K = static_cast<int>(s.H);
    p.n_out = static_cast<int>(s.I);
    p.n_tile = 96;
    p.b_rows = static_cast<int>(2 * s.I);
    p.half = static_cast<int>(s.I);
    return cuda_status(launch_gemm1_mx(p, st));
}

// The MXFP8 dispatch: x quantized straight into routed order (needs the metadata;
// obuf, idle until stage 2, holds the row-major scales in between).
moe_status_t run_mx_dispatch(const moe_shape_t &s, const void *x, const Ws &w, cudaStream_t st) {
    return cuda_status(launch_mx_quantize_dispatch(static_cast<const __nv_bfloat16 *>(x), w.row_of, w.offsets + s.E,
                                                   s.k, s.T, s.H, w.x_codes, w.x_scales,
                                                   reinterpret_cast<uint8_t *>(w.obuf), st));
}

// Stage 2 in MXFP8: E4M3 a and w2 through TMA, weighted rows into obuf, then the k-way combine.
moe_status_t run_gemm2_mx(const moe_shape_t &s, const void *aq, const void *as, const float *topk_w,
                          const void *w2q, const void *w2s, void *y, const Ws &w, const DeviceState &d,
                          cudaStream_t st) {
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    CUtensorMap tm_a, tm_w2, tm_out, tm_as, tm_w2s;
    if (!encode_u8_2d(&tm_a, aq, s.I, R, 128, 128) ||
        !encode_u8_2d(&tm_w2, w2q, s.I, static_cast<uint64_t>(s.E) * s.H, 128, 224) ||
        !encode_bf16_2d(&tm_out, w.obuf, s.H, R, 32, 32) ||
        !encode_sf_words(&tm_as, as, mx_rows(R), s.I / 128, kSfBoxRowsA) ||
        !encode_sf_words(&tm_w2s, w2s, static_cast<uint64_t>(s.E) * s.H, s.I / 128, 224))
        return MOE_ERR_CUDA;
    GemmLaunch p = base_launch(s, w, d);
    p.tm_a = &tm_a;
    p.tm_b = &tm_w2;
    p.tm_out = &tm_out;
    p.tm_sfa = &tm_as;
    p.tm_sfb = &tm_w2s;
    p.sched = w.sched2;
    p.topk_w = topk_w;
    p.out = w.obuf;
    p.K = static_cast<int>(s.I);
    p.n_out = static_cast<int>(s.H);
    p.n_tile = 224;
    p.b_rows = static_cast<int>(s.H);
    moe_status_t r = cuda_status(launch_gemm2_mx(p, st));
    if (r != MOE_OK) return r;
    CombineLaunch c;
    c.obuf = w.obuf;
    c.row_of = w.row_of;
    c.y = static_cast<__nv_bfloat16 *>(y);
    c.T = static_cast<int>(s.T);
    c.H = static_cast<int>(s.H);
    c.k = s.k;
    return cuda_status(launch_combine(c, st));
}

// Stage 2 backward, data: dY's rows dispatched into routed order (dyp, read
// again by the weight part), rows of dropped slots zeroed, dA GEMM with the
// SwiGLU backward epilogue, then the routing-weight gradient.
moe_status_t run_bwd_stage2_data(const moe_shape_t &s, const void *dy, const float *topk_w, const void *w2,
                                 const void *h, float *dtopk_w, const Ws &w, const DeviceState &d,
                                 cudaStream_t st) {
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    CUtensorMap tm_dy, tm_w2, tm_dg, tm_du, tm_aw;
    // w2 [E, H, I] read MN-major: K = H rows of expert e, N = I
    if (!encode_bf16_2d(&tm_dy, w.dyp, s.H, R, kBK, 128) ||
        !encode_bf16_3d(&tm_w2, w2, s.I, s.H, s.E, 64, kBK) ||
        !encode_bf16_2d_strided(&tm_dg, w.dh, s.I, R, 2 * s.I, 32, 32) ||
        !encode_bf16_2d_strided(&tm_du, w.dh + s.I, s.I, R, 2 * s.I, 32, 32) ||
        !encode_bf16_2d(&tm_aw, w.aw, s.I, R, 32, 32))
        return MOE_ERR_CUDA;
    moe_status_t r = cuda_status(launch_dispatch_rows(static_cast<const __nv_bfloat16 *>(dy), w.row_of, s.T, s.k,
                                                      s.H, w.dyp, nullptr, nullptr, st));
    if (r != MOE_OK) return r;
    r = cuda_status(launch_zero_tail_rows(w.dh, w.aw, w.offsets + s.E, static_cast<int>(R), static_cast<int>(s.I),
                                          st));
    if (r != MOE_OK) return r;
    GemmLaunch p = base_launch(s, w, d);
    p.tm_a = &tm_dy;
    p.tm_b = &tm_w2;
    p.tm_out = &tm_dg;
    p.tm_out2 = &tm_du;
    p.tm_out3 = &tm_aw;
    p.h = static_cast<const __nv_bfloat16 *>(h);
    p.sched = w.sched_da;
    p.topk_w = topk_w;
    p.out = w.dh;
    p.out2 = w.dh + s.I;
    p.out3 = w.aw;
    p.dtw_part = w.dtw_part;
    p.K = static_cast<int>(s.H);
    p.n_out = static_cast<int>(s.I);
    p.n_tile = kBN;
    p.half = static_cast<int>(s.I);
    p.out_ld = static_cast<int>(2 * s.I);
    if ((r = cuda_status(launch_bwd_da(p, st))) != MOE_OK) return r;
    if (dtopk_w == nullptr) return MOE_OK;
    DtwReduceLaunch q;
    q.dtw_part = w.dtw_part;
    q.n_part = static_cast<int>((s.I + kBN - 1) / kBN);
    q.R = static_cast<int>(R);
    q.T = static_cast<int>(s.T);
    q.k = s.k;
    q.row_of = w.row_of;
    q.dtopk_w = dtopk_w;
    return cuda_status(launch_dtw_reduce(q, st));
}

// Stage 2 backward, weights: dW2[e] (M = H rows, N = I, K = e's rows): A = the
// dY rows dispatched by the data part, B = w a rows, both MN-major through TMA.
moe_status_t run_bwd_stage2_weight(const moe_shape_t &s, void *dw2, const Ws &w, const DeviceState &d,
                                   cudaStream_t st) {
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    CUtensorMap tm_dy_mn, tm_aw_mn, tm_dw2;
    if (!encode_bf16_2d(&tm_dy_mn, w.dyp, s.H, R, 64, kBK) ||
        !encode_bf16_2d(&tm_aw_mn, w.aw, s.I, R, 64, kBK) ||
        !encode_bf16_3d(&tm_dw2, dw2, s.I, s.H, s.E, 32, 32))
        return MOE_ERR_CUDA;
    GemmLaunch q = base_launch(s, w, d);
    q.tm_a = &tm_dy_mn;
    q.tm_b = &tm_aw_mn;
    q.tm_out = &tm_dw2;
    q.sched = w.sched_dw2;
    q.n_out = static_cast<int>(s.I);
    q.n_tile = kBN;
    q.m_total = static_cast<int>(s.H);
    return cuda_status(launch_bwd_dw2(q, st));
}

// Router backward: logit gradient into the workspace, then dW_r.
moe_status_t run_router_bwd(const moe_shape_t &s, const void *x, const float *logits, const int32_t *topk_idx,
                            const float *topk_w, const float *dtopk_w, const moe_router_cfg_t &cfg, float *dw_r,
                            const Ws &w, cudaStream_t st) {
    RouterBwdLaunch p;
    p.logits = logits;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.dtopk_w = dtopk_w;
    p.T = static_cast<int>(s.T);
    p.H = static_cast<int>(s.H);
    p.E = static_cast<int>(s.E);
    p.k = s.k;
    p.score_fn = cfg.score_fn;
    p.normalize = cfg.normalize;
    p.scale = cfg.scale;
    p.dl = w.dlogits;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.offsets = w.offsets;
    p.counts = w.counts;
    p.perm_slot = w.perm_slot;
    p.dw_r = dw_r;
    p.dwr_part = w.dwr_part;
    moe_status_t r = cuda_status(launch_router_dlogits(p, st));
    if (r != MOE_OK) return r;
    return cuda_status(launch_router_dwr(p, st));
}

// Stage 1 backward, data: dX rows GEMM, then the per-token sum (+ router term).
moe_status_t run_bwd_stage1_data(const moe_shape_t &s, const void *w1, const float *w_r, const int32_t *topk_idx,
                                 int dense_router, void *dx, const Ws &w, const DeviceState &d, cudaStream_t st) {
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    CUtensorMap tm_dh, tm_w1, tm_xr;
    // w1 [E, 2I, H] read MN-major: K = 2I rows of expert e, N = H
    if (!encode_bf16_2d(&tm_dh, w.dh, 2 * s.I, R, kBK, 128) ||
        !encode_bf16_3d(&tm_w1, w1, s.H, 2 * s.I, s.E, 64, kBK) ||
        !encode_bf16_2d(&tm_xr, w.obuf, s.H, R, 64, 32))
        return MOE_ERR_CUDA;
    GemmLaunch p = base_launch(s, w, d);
    p.tm_a = &tm_dh;
    p.tm_b = &tm_w1;
    p.tm_out = &tm_xr;
    p.sched = w.sched_dx;
    p.out = w.obuf;
    p.K = static_cast<int>(2 * s.I);
    p.n_out = static_cast<int>(s.H);
    p.n_tile = kBN;
    moe_status_t r = cuda_status(launch_bwd_dx(p, st));
    if (r != MOE_OK) return r;
    CombineBwdLaunch c;
    c.xbuf = w.obuf;
    c.row_of = w.row_of;
    c.topk_idx = topk_idx;
    c.dl = w_r ? w.dlogits : nullptr;
    c.w_r = w_r;
    c.dense = dense_router;
    c.dx = static_cast<__nv_bfloat16 *>(dx);
    c.T = static_cast<int>(s.T);
    c.H = static_cast<int>(s.H);
    c.E = static_cast<int>(s.E);
    c.k = s.k;
    return cuda_status(launch_combine_bwd(c, st));
}

// Stage 1 backward, weights: dW1[e] (M = 2I rows, N = H, K = e's rows): A = dH
// rows, B = the x rows dispatched by the training forward (xp), both MN-major
// through TMA.
moe_status_t run_bwd_stage1_weight(const moe_shape_t &s, void *dw1, const Ws &w, const DeviceState &d,
                                   cudaStream_t st) {
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    CUtensorMap tm_dh_mn, tm_x_mn, tm_dw1;
    if (!encode_bf16_2d(&tm_dh_mn, w.dh, 2 * s.I, R, 64, kBK) ||
        !encode_bf16_2d(&tm_x_mn, w.xp, s.H, R, 64, kBK) ||
        !encode_bf16_3d(&tm_dw1, dw1, s.H, 2 * s.I, s.E, 32, 32))
        return MOE_ERR_CUDA;
    GemmLaunch q = base_launch(s, w, d);
    q.tm_a = &tm_dh_mn;
    q.tm_b = &tm_x_mn;
    q.tm_out = &tm_dw1;
    q.sched = w.sched_dw1;
    q.n_out = static_cast<int>(s.H);
    q.n_tile = kBN;
    q.m_total = static_cast<int>(2 * s.I);
    return cuda_status(launch_bwd_dw1(q, st));
}

// An MXFP8 weight gradient: dW[e] = Q(A_e)^T Q(B_e) over expert e's routed rows,
// from the transposed, row-quantized operands (M = a_cols rows, N = b_cols).
moe_status_t run_wgrad_mx(const moe_shape_t &s, const MxWgradWs &m, const uint8_t *a_c, const uint8_t *a_s,
                          int64_t a_cols, const uint8_t *b_c, const uint8_t *b_s, int64_t b_cols, void *dw,
                          int32_t *sched, const Ws &w, const DeviceState &d, cudaStream_t st) {
    CUtensorMap tm_a, tm_b, tm_dw, tm_as, tm_bs;
    if (!encode_u8_2d(&tm_a, a_c, m.ld, a_cols, 128, 128) || !encode_u8_2d(&tm_b, b_c, m.ld, b_cols, 128, 224) ||
        !encode_bf16_3d(&tm_dw, dw, b_cols, a_cols, s.E, 32, 32) ||
        !encode_sf_words(&tm_as, a_s, a_cols, m.ld / 128, kSfBoxRowsA) ||
        !encode_sf_words(&tm_bs, b_s, b_cols, m.ld / 128, 224))
        return MOE_ERR_CUDA;
    GemmLaunch q = base_launch(s, w, d);
    q.tm_a = &tm_a;
    q.tm_b = &tm_b;
    q.tm_out = &tm_dw;
    q.kpad = m.kpad;
    q.tm_sfa = &tm_as;
    q.tm_sfb = &tm_bs;
    q.sched = sched;
    q.K = static_cast<int>(m.ld);     // scale bytes per operand row: K / 32
    q.n_out = static_cast<int>(b_cols);
    q.n_tile = 224;
    q.m_total = static_cast<int>(a_cols);
    q.b_rows = 0;                     // the B operand's rows are shared by every expert
    return cuda_status(launch_wgrad_mx(q, st));
}

// Stage 2 backward, weights, MXFP8: dW2[e] = Q(dY)^T Q(w a) over e's rows (the
// dY rows and w a left in the workspace by the stage-2 data part).
moe_status_t run_bwd_stage2_weight_mx(const moe_shape_t &s, void *dw2, const Ws &w, const DeviceState &d,
                                      cudaStream_t st, void *ws) {
    const MxWgradWs m = carve_mx_wgrad(ws, s);
    const int E = static_cast<int>(s.E);
    moe_status_t r = cuda_status(launch_mx_wgrad_offsets(w.counts, E, m.kpad, st));
    if (r != MOE_OK) return r;
    if ((r = cuda_status(launch_mx_quantize_rows_t(w.dyp, s.H, nullptr, s.k, w.counts, w.offsets, m.kpad, E,
                                                   static_cast<int>(s.H), m.ld, m.dy_c, m.dy_s, st))) != MOE_OK ||
        (r = cuda_status(launch_mx_quantize_rows_t(w.aw, s.I, nullptr, s.k, w.counts, w.offsets, m.kpad, E,
                                                   static_cast<int>(s.I), m.ld, m.aw_c, m.aw_s, st))) != MOE_OK)
        return r;
    int32_t *sched = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(ws) + kHdrSchedDW2Mx);
    return run_wgrad_mx(s, m, m.dy_c, m.dy_s, s.H, m.aw_c, m.aw_s, s.I, dw2, sched, w, d, st);
}

// Stage 1 backward, weights, MXFP8: dW1[e] = Q(dH)^T Q(x) over e's rows (dH from
// the stage-2 data part; x's rows gathered by token).
moe_status_t run_bwd_stage1_weight_mx(const moe_shape_t &s, const void *x, void *dw1, const Ws &w,
                                      const DeviceState &d, cudaStream_t st, void *ws) {
    const MxWgradWs m = carve_mx_wgrad(ws, s);
    const int E = static_cast<int>(s.E);
    moe_status_t r = cuda_status(launch_mx_wgrad_offsets(w.counts, E, m.kpad, st));
    if (r != MOE_OK) return r;
    if ((r = cuda_status(launch_mx_quantize_rows_t(w.dh, 2 * s.I, nullptr, s.k, w.counts, w.offsets, m.kpad, E,
                                                   static_cast<int>(2 * s.I), m.ld, m.dh_c, m.dh_s, st))) != MOE_OK ||
        (r = cuda_status(launch_mx_quantize_rows_t(static_cast<const __nv_bfloat16 *>(x), s.H, w.perm_slot, s.k,
                                                   w.counts, w.offsets, m.kpad, E, static_cast<int>(s.H), m.ld,
                                                   m.x_c, m.x_s, st))) != MOE_OK)
        return r;
    int32_t *sched = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(ws) + kHdrSchedDW1Mx);
    return run_wgrad_mx(s, m, m.dh_c, m.dh_s, 2 * s.I, m.x_c, m.x_s, s.H, dw1, sched, w, d, st);
}

moe_status_t run_metadata(const moe_shape_t &s, const int32_t *topk_idx, const Ws &w, cudaStream_t st) {
    MetadataLaunch m;
    m.topk_idx = topk_idx;
    m.R = static_cast<int>(s.T * s.k);
    m.E = static_cast<int>(s.E);
    m.counts = w.counts;
    m.offsets = w.offsets;
    m.mt_prefix = w.mt_prefix;
    m.perm_slot = w.perm_slot;
    m.row_of = w.row_of;
    m.err = w.err;
    m.block_hist = w.meta;
    m.ticket = w.meta_ticket;
    m.combine.cnt = fused_combine(s) ? w.combine : nullptr;
    m.combine.T = static_cast<int>(s.T);
    m.combine.k = s.k;
    m.combine.n_tiles = static_cast<int>((s.H + kBN - 1) / kBN);
    return cuda_status(launch_routing_metadata(m, st));
}

}  // namespace

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;
}  // namespace

namespace {

// bf16 tensor of rank 2 or 3 (dims[0] contiguous, byte strides for the others)
// with a box_inner x box_rows (x 1) box, zero fill out of bounds, and the
// swizzle span equal to the box row (64 or 128 bytes).
// Looks up cuTensorMapEncodeTiled once; false when the driver lacks it.
bool encode_ready() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        else
            cudaGetLastError();   // clear only the error the failed lookup raised
    });
    return g_encode != nullptr;
}

bool encode_bf16(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
                 const cuuint64_t *byte_strides, uint32_t box_inner, uint32_t box_rows) {
    if (!encode_ready()) return false;
    if (box_inner * 2 != 128 && box_inner * 2 != 64) return false;
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, byte_strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    box_inner * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool encode_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows) {
    return encode_bf16_2d_strided(map, base, inner, rows, inner, box_inner, box_rows);
}

bool encode_u8_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                  uint32_t box_rows) {
    if (!encode_ready() || box_inner != 128) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_sf_words(CUtensorMap *map, const void *base, uint64_t rows, uint64_t k_blocks, uint32_t box_rows) {
    if (!encode_ready() || rows % 4 != 0) return false;
    cuuint64_t dims[2] = {rows, k_blocks};
    cuuint64_t strides[1] = {rows * 4};
    cuuint32_t box[2] = {box_rows, 1};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_bf16_2d_strided(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                            uint64_t row_stride, uint32_t box_inner, uint32_t box_rows) {
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride * 2};
    return encode_bf16(map, base, 2, dims, strides, box_inner, box_rows);
}

bool encode_bf16_3d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint64_t depth,
                    uint32_t box_inner, uint32_t box_rows) {
    cuuint64_t dims[3] = {inner, rows, depth};
    cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
    return encode_bf16(map, base, 3, dims, strides, box_inner, box_rows);
}

void note_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_workspace_size(const moe_shape_t *shape, size_t *bytes) {
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    const moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    *bytes = make_layout(*shape).total;
    return MOE_OK;
}

moe_status_t moe_workspace_layout(const moe_shape_t *shape, moe_ws_layout_t *layout) {
    if (layout == nullptr) return MOE_ERR_INVALID_ARG;
    const moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    *layout = make_layout(*shape);
    return MOE_OK;
}

moe_status_t moe_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    if (ws == nullptr || ws_bytes < kWsHeaderBytes || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(ws, 0, kWsHeaderBytes, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {

moe_status_t check_router_cfg(const moe_shape_t *shape, const moe_router_cfg_t *cfg) {
    if (cfg->score_fn != MOE_SCORE_SOFTMAX && cfg->score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (cfg->n_group < 1 || cfg->n_group > 32) return MOE_ERR_UNSUPPORTED;
    if (cfg->n_group > 1) {
        if (shape->E % cfg->n_group != 0 || cfg->topk_group < 1 || cfg->topk_group > cfg->n_group ||
            cfg->group_topn < 1 || cfg->group_topn > shape->E / cfg->n_group)
            return MOE_ERR_INVALID_ARG;
        if (static_cast<int64_t>(cfg->topk_group) * (shape->E / cfg->n_group) < shape->k)
            return MOE_ERR_INVALID_ARG;
    }
    return MOE_OK;
}

moe_status_t router_impl(const void *x, const float *w_r, const float *logit_offset, const float *sel_bias,
                         const moe_shape_t *shape, const moe_router_cfg_t *cfg, int32_t *topk_idx,
                         float *topk_w, float *aux, float *logits, void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;  // nothing to route or compute
    if (cfg == nullptr || x == nullptr || w_r == nullptr || topk_idx == nullptr || topk_w == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_r) || !aligned16(topk_idx) || !aligned16(topk_w))
        return MOE_ERR_INVALID_ARG;
    if ((logit_offset && (reinterpret_cast<uintptr_t>(logit_offset) & 3u)) ||
        (sel_bias && (reinterpret_cast<uintptr_t>(sel_bias) & 3u)) ||
        (aux && (reinterpret_cast<uintptr_t>(aux) & 3u)))
        return MOE_ERR_INVALID_ARG;
    if (logits != nullptr && !aligned16(logits)) return MOE_ERR_INVALID_ARG;
    if ((r = check_router_cfg(shape, cfg)) != MOE_OK) return r;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *shape);
    RouterLaunch p;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.w_r = w_r;
    p.logit_offset = logit_offset;
    p.sel_bias = sel_bias;
    p.T = static_cast<int>(shape->T);
    p.H = static_cast<int>(shape->H);
    p.E = static_cast<int>(shape->E);
    p.k = shape->k;
    p.score_fn = cfg->score_fn;
    p.normalize = cfg->normalize;
    p.scale = cfg->scale;
    p.n_group = cfg->n_group;
    p.topk_group = cfg->topk_group;
    p.group_topn = cfg->group_topn;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.aux = aux;
    p.logits = logits;
    p.err = w.err;
    p.num_sms = d->num_sms;
    p.scratch = w.router;
    return cuda_status(launch_router(p, static_cast<cudaStream_t>(stream)));
}

// Common checks of the training entry points: a training workspace.
moe_status_t check_training(const moe_shape_t *shape, const void *ws, size_t ws_bytes) {
    moe_status_t r = check_ws(*shape, ws, ws_bytes);
    if (r != MOE_OK) return r;
    return (shape->flags & MOE_SHAPE_TRAINING) ? MOE_OK : MOE_ERR_INVALID_ARG;
}

bool dense_router_grad(const moe_router_cfg_t &cfg) {
    return cfg.score_fn == MOE_SCORE_SOFTMAX && !cfg.normalize;
}

}  // namespace

extern "C" {

moe_status_t moe_router(const void *x, const float *w_r, const float *logit_offset,
                        const float *sel_bias, const moe_shape_t *shape,
                        const moe_router_cfg_t *cfg, int32_t *topk_idx, float *topk_w, float *aux,
                        void *ws, size_t ws_bytes, void *stream) {
    return router_impl(x, w_r, logit_offset, sel_bias, shape, cfg, topk_idx, topk_w, aux, nullptr, ws,
                       ws_bytes, stream);
}

moe_status_t moe_route_logits(const float *logits, const float *logit_offset, const float *sel_bias,
                              const moe_shape_t *shape, const moe_router_cfg_t *cfg, int32_t *topk_idx,
                              float *topk_w, float *aux, void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;
    if (cfg == nullptr || logits == nullptr || topk_idx == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(logits) || !aligned16(topk_idx) || !aligned16(topk_w)) return MOE_ERR_INVALID_ARG;
    if ((logit_offset && (reinterpret_cast<uintptr_t>(logit_offset) & 3u)) ||
        (sel_bias && (reinterpret_cast<uintptr_t>(sel_bias) & 3u)) ||
        (aux && (reinterpret_cast<uintptr_t>(aux) & 3u)))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_router_cfg(shape, cfg)) != MOE_OK) return r;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *shape);
    RouterLaunch p{};
    p.logit_offset = logit_offset;
    p.sel_bias = sel_bias;
    p.T = static_cast<int>(shape->T);
    p.H = static_cast<int>(shape->H);
    p.E = static_cast<int>(shape->E);
    p.k = shape->k;
    p.score_fn = cfg->score_fn;
    p.normalize = cfg->normalize;
    p.scale = cfg->scale;
    p.n_group = cfg->n_group;
    p.topk_group = cfg->topk_group;
    p.group_topn = cfg->group_topn;
    p.topk_idx = topk_idx;
    p.topk_w = topk_w;
    p.aux = aux;
    p.logits = nullptr;
    p.err = w.err;
    p.num_sms = d->num_sms;
    p.scratch = w.router;
    return cuda_status(launch_route_logits(p, logits, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_router_train(const void *x, const float *w_r, const float *logit_offset,
                              const float *sel_bias, const moe_shape_t *shape,
                              const moe_router_cfg_t *cfg, int32_t *topk_idx, float *topk_w,
                              float *aux, float *logits, void *ws, size_t ws_bytes, void *stream) {
    if (shape != nullptr && shape->T > 0 && logits == nullptr) return MOE_ERR_INVALID_ARG;
    return router_impl(x, w_r, logit_offset, sel_bias, shape, cfg, topk_idx, topk_w, aux, logits, ws,
                       ws_bytes, stream);
}

moe_status_t moe_routing_metadata(const int32_t *topk_idx, const moe_shape_t *shape, void *ws,
                                  size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;  // nothing to route or compute
    if (topk_idx == nullptr || !aligned16(topk_idx)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_metadata(*shape, topk_idx, carve(ws, *shape), static_cast<cudaStream_t>(stream));
}

moe_status_t moe_dispatch_gemm1(const void *x, const void *w1, const moe_shape_t *shape, void *a,
                                void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;  // nothing to route or compute
    if (x == nullptr || w1 == nullptr || a == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w1) || !aligned16(a)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_gemm1(*shape, x, w1, a, nullptr, carve(ws, *shape), *d, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_swiglu_gemm2_combine(const void *a, const float *topk_w, const void *w2,
                                      const moe_shape_t *shape, void *y, void *ws,
                                      size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;  // nothing to route or compute
    if (a == nullptr || topk_w == nullptr || w2 == nullptr || y == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(topk_w) || !aligned16(w2) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_gemm2(*shape, a, topk_w, w2, y, carve(ws, *shape), *d, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_packed_weights_size(const moe_shape_t *shape, size_t *w1p_bytes, size_t *w2p_bytes) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    constexpr size_t kTile = 32768;
    if (w1p_bytes) *w1p_bytes = kTile * static_cast<size_t>(packed_w1_tiles(shape->E, shape->H, shape->I));
    if (w2p_bytes) *w2p_bytes = kTile * static_cast<size_t>(packed_w2_tiles(shape->E, shape->H, shape->I));
    return MOE_OK;
}

moe_status_t moe_pack_weights(const void *w1, const void *w2, const moe_shape_t *shape, void *w1p, void *w2p,
                              void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if ((w1 == nullptr) != (w1p == nullptr) || (w2 == nullptr) != (w2p == nullptr)) return MOE_ERR_INVALID_ARG;
    if ((w1 && (!aligned16(w1) || !aligned16(w1p))) || (w2 && (!aligned16(w2) || !aligned16(w2p))))
        return MOE_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (w1 && (r = cuda_status(launch_pack_w1(static_cast<const __nv_bfloat16 *>(w1), shape->E, shape->H, shape->I,
                                              w1p, st))) != MOE_OK)
        return r;
    if (w2)
        r = cuda_status(launch_pack_w2(static_cast<const __nv_bfloat16 *>(w2), shape->E, shape->H, shape->I, w2p, st));
    return r;
}

moe_status_t moe_forward(const void *x, const int32_t *topk_idx, const float *topk_w, const void *w1,
                         const void *w2, const moe_shape_t *shape, void *y, void *ws,
                         size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;  // nothing to route or compute
    if (x == nullptr || topk_idx == nullptr || topk_w == nullptr || w1 == nullptr || w2 == nullptr ||
        y == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(w1) ||
        !aligned16(w2) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *shape);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((r = run_metadata(*shape, topk_idx, w, st)) != MOE_OK) return r;
    if ((r = run_gemm1(*shape, x, w1, w.a, nullptr, w, *d, st)) != MOE_OK) return r;
    return run_gemm2(*shape, w.a, topk_w, w2, y, w, *d, st);
}

moe_status_t moe_dispatch_gemm1_train(const void *x, const void *w1, const moe_shape_t *shape,
                                      void *a, void *h, void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;
    if (x == nullptr || w1 == nullptr || a == nullptr || h == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w1) || !aligned16(a) || !aligned16(h)) return MOE_ERR_INVALID_ARG;
    if ((r = check_training(shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_gemm1(*shape, x, w1, a, h, carve(ws, *shape), *d, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_backward_stage2_data(const void *dy, const float *topk_w, const void *w2, const void *h,
                                      const moe_shape_t *shape, float *dtopk_w, void *ws, size_t ws_bytes,
                                      void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;
    if (dy == nullptr || topk_w == nullptr || w2 == nullptr || h == nullptr) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned16(topk_w) || !aligned16(w2) || !aligned16(h) ||
        (dtopk_w && !aligned16(dtopk_w)))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_training(shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_bwd_stage2_data(*shape, dy, topk_w, w2, h, dtopk_w, carve(ws, *shape), *d,
                               static_cast<cudaStream_t>(stream));
}

moe_status_t moe_backward_stage2_weight(const void *dy, const moe_shape_t *shape, void *dw2, void *ws,
                                        size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (dw2 == nullptr || !aligned16(dw2)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (shape->T == 0)  // no rows: every expert's weight gradient is zero
        return cuda_status(cudaMemsetAsync(dw2, 0, 2 * static_cast<size_t>(shape->E) * shape->H * shape->I, st));
    if (dy == nullptr || !aligned16(dy)) return MOE_ERR_INVALID_ARG;
    if ((r = check_training(shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_bwd_stage2_weight(*shape, dw2, carve(ws, *shape), *d, st);
}

moe_status_t moe_router_backward(const void *x, const float *logits, const int32_t *topk_idx,
                                 const float *topk_w, const float *dtopk_w, const moe_shape_t *shape,
                                 const moe_router_cfg_t *cfg, float *dw_r, void *ws, size_t ws_bytes,
                                 void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (cfg == nullptr || dw_r == nullptr || !aligned16(dw_r)) return MOE_ERR_INVALID_ARG;
    if ((r = check_router_cfg(shape, cfg)) != MOE_OK) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (shape->T == 0)
        return cuda_status(cudaMemsetAsync(dw_r, 0, 4 * static_cast<size_t>(shape->E) * shape->H, st));
    if (x == nullptr || logits == nullptr || topk_idx == nullptr || topk_w == nullptr || dtopk_w == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(logits) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(dtopk_w))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_training(shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_router_bwd(*shape, x, logits, topk_idx, topk_w, dtopk_w, *cfg, dw_r, carve(ws, *shape), st);
}

moe_status_t moe_backward_stage1_data(const void *w1, const float *w_r, const int32_t *topk_idx,
                                      const moe_router_cfg_t *cfg, const moe_shape_t *shape, void *dx,
                                      void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (w_r != nullptr && cfg == nullptr) return MOE_ERR_INVALID_ARG;
    if (shape->T == 0) return MOE_OK;
    if (w1 == nullptr || dx == nullptr || (w_r != nullptr && topk_idx == nullptr)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w1) || !aligned16(dx) || (w_r && !aligned16(w_r)) || (topk_idx && !aligned16(topk_idx)))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_training(shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_bwd_stage1_data(*shape, w1, w_r, topk_idx, w_r ? dense_router_grad(*cfg) : 0, dx,
                               carve(ws, *shape), *d, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_backward_stage1_weight(const void *x, const moe_shape_t *shape, void *dw1, void *ws,
                                        size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (dw1 == nullptr || !aligned16(dw1)) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (shape->T == 0)
        return cuda_status(cudaMemsetAsync(dw1, 0, 4 * static_cast<size_t>(shape->E) * shape->I * shape->H, st));
    if (x == nullptr || !aligned16(x)) return MOE_ERR_INVALID_ARG;
    if ((r = check_training(shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_bwd_stage1_weight(*shape, dw1, carve(ws, *shape), *d, st);
}

moe_status_t moe_backward(const void *x, const float *w_r, const float *logits, const int32_t *topk_idx,
                          const float *topk_w, const void *w1, const void *w2, const void *h, const void *dy,
                          const moe_shape_t *shape, const moe_router_cfg_t *cfg, void *dx, void *dw1,
                          void *dw2, float *dw_r, float *dtopk_w, void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (w_r != nullptr && (logits == nullptr || cfg == nullptr || dw_r == nullptr || dtopk_w == nullptr ||
                           topk_idx == nullptr))
        return MOE_ERR_INVALID_ARG;
    if ((r = moe_backward_stage2_data(dy, topk_w, w2, h, shape, dtopk_w, ws, ws_bytes, stream)) != MOE_OK ||
        (r = moe_backward_stage2_weight(dy, shape, dw2, ws, ws_bytes, stream)) != MOE_OK)
        return r;
    if (w_r != nullptr &&
        (r = moe_router_backward(x, logits, topk_idx, topk_w, dtopk_w, shape, cfg, dw_r, ws, ws_bytes, stream)) !=
            MOE_OK)
        return r;
    if ((r = moe_backward_stage1_data(w1, w_r, topk_idx, cfg, shape, dx, ws, ws_bytes, stream)) != MOE_OK)
        return r;
    return moe_backward_stage1_weight(x, shape, dw1, ws, ws_bytes, stream);
}

moe_status_t moe_mx_quantize(const void *in, int64_t rows, int64_t cols, void *codes, void *scales,
                             void *stream) {
    if (rows < 0 || cols <= 0 || cols % 128 != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (in == nullptr || codes == nullptr || scales == nullptr || !aligned16(in) || !aligned16(codes) ||
        !aligned16(scales))
        return MOE_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    moe_status_t r = device_state(&d);
    if (r != MOE_OK) return r;
    return cuda_status(launch_mx_quantize(static_cast<const __nv_bfloat16 *>(in), rows, cols,
                                          static_cast<uint8_t *>(codes), static_cast<uint8_t *>(scales),
                                          static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_mx_quantize_dispatch(const void *x, const moe_shape_t *shape, void *ws, size_t ws_bytes,
                                      void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->H % 128 || shape->I % 128) return MOE_ERR_UNSUPPORTED;
    if (shape->T == 0) return MOE_OK;
    if (x == nullptr || !aligned16(x)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    if (!(shape->flags & MOE_SHAPE_MXFP8)) return MOE_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_mx_dispatch(*shape, x, carve(ws, *shape), static_cast<cudaStream_t>(stream));
}

moe_status_t moe_dispatch_gemm1_mx(const void *w1_codes, const void *w1_scales, const moe_shape_t *shape,
                                   void *a_codes, void *a_scales, void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->H % 128 || shape->I % 128) return MOE_ERR_UNSUPPORTED;
    if (shape->T == 0) return MOE_OK;
    if (!w1_codes || !w1_scales || !a_codes || !a_scales) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w1_codes) || !aligned16(w1_scales) || !aligned16(a_codes) || !aligned16(a_scales))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    if (!(shape->flags & MOE_SHAPE_MXFP8)) return MOE_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_gemm1_mx(*shape, w1_codes, w1_scales, a_codes, a_scales, nullptr, carve(ws, *shape), *d,
                        static_cast<cudaStream_t>(stream));
}

moe_status_t moe_swiglu_gemm2_combine_mx(const void *a_codes, const void *a_scales, const float *topk_w,
                                         const void *w2_codes, const void *w2_scales,
                                         const moe_shape_t *shape, void *y, void *ws, size_t ws_bytes,
                                         void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->H % 128 || shape->I % 128) return MOE_ERR_UNSUPPORTED;
    if (shape->T == 0) return MOE_OK;
    if (!a_codes || !a_scales || !topk_w || !w2_codes || !w2_scales || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(a_codes) || !aligned16(a_scales) || !aligned16(topk_w) || !aligned16(w2_codes) ||
        !aligned16(w2_scales) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_gemm2_mx(*shape, a_codes, a_scales, topk_w, w2_codes, w2_scales, y, carve(ws, *shape), *d,
                        static_cast<cudaStream_t>(stream));
}

moe_status_t moe_forward_mx(const void *x, const int32_t *topk_idx, const float *topk_w,
                            const void *w1_codes, const void *w1_scales, const void *w2_codes,
                            const void *w2_scales, const moe_shape_t *shape, void *y, void *ws,
                            size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->H % 128 || shape->I % 128) return MOE_ERR_UNSUPPORTED;
    if (shape->T == 0) return MOE_OK;
    if (!x || !topk_idx || !topk_w || !w1_codes || !w1_scales || !w2_codes || !w2_scales || !y)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(topk_idx) || !aligned16(topk_w) || !aligned16(w1_codes) ||
        !aligned16(w1_scales) || !aligned16(w2_codes) || !aligned16(w2_scales) || !aligned16(y))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    if (!(shape->flags & MOE_SHAPE_MXFP8)) return MOE_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *shape);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((r = run_metadata(*shape, topk_idx, w, st)) != MOE_OK) return r;
    if ((r = run_mx_dispatch(*shape, x, w, st)) != MOE_OK) return r;
    if ((r = run_gemm1_mx(*shape, w1_codes, w1_scales, w.a_codes, w.a_scales, nullptr, w, *d, st)) != MOE_OK)
        return r;
    return run_gemm2_mx(*shape, w.a_codes, w.a_scales, topk_w, w2_codes, w2_scales, y, w, *d, st);
}

moe_status_t moe_dispatch_gemm1_mx_train(const void *w1_codes, const void *w1_scales, const moe_shape_t *shape,
                                         void *a_codes, void *a_scales, void *h, void *ws, size_t ws_bytes,
                                         void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->H % 128 || shape->I % 128) return MOE_ERR_UNSUPPORTED;
    if (shape->T == 0) return MOE_OK;
    if (!w1_codes || !w1_scales || !a_codes || !a_scales || !h) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w1_codes) || !aligned16(w1_scales) || !aligned16(a_codes) || !aligned16(a_scales) ||
        !aligned16(h))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_training(shape, ws, ws_bytes)) != MOE_OK) return r;
    if (!(shape->flags & MOE_SHAPE_MXFP8)) return MOE_ERR_INVALID_ARG;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_gemm1_mx(*shape, w1_codes, w1_scales, a_codes, a_scales, h, carve(ws, *shape), *d,
                        static_cast<cudaStream_t>(stream));
}

// Common checks of the MXFP8 weight-gradient entry points.
static moe_status_t check_wgrad_mx(const moe_shape_t *shape, const void *in, void *dw, void *ws,
                                   size_t ws_bytes) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->H % 128 || shape->I % 128) return MOE_ERR_UNSUPPORTED;
    if (dw == nullptr || !aligned16(dw)) return MOE_ERR_INVALID_ARG;
    if (shape->T == 0) return MOE_OK;
    if (in == nullptr || !aligned16(in)) return MOE_ERR_INVALID_ARG;
    if ((r = check_training(shape, ws, ws_bytes)) != MOE_OK) return r;
    return (shape->flags & MOE_SHAPE_MXFP8) ? MOE_OK : MOE_ERR_INVALID_ARG;
}

moe_status_t moe_backward_stage2_weight_mx(const void *dy, const moe_shape_t *shape, void *dw2, void *ws,
                                           size_t ws_bytes, void *stream) {
    moe_status_t r = check_wgrad_mx(shape, dy, dw2, ws, ws_bytes);
    if (r != MOE_OK) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (shape->T == 0)
        return cuda_status(cudaMemsetAsync(dw2, 0, 2 * static_cast<size_t>(shape->E) * shape->H * shape->I, st));
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_bwd_stage2_weight_mx(*shape, dw2, carve(ws, *shape), *d, st, ws);
}

moe_status_t moe_backward_stage1_weight_mx(const void *x, const moe_shape_t *shape, void *dw1, void *ws,
                                           size_t ws_bytes, void *stream) {
    moe_status_t r = check_wgrad_mx(shape, x, dw1, ws, ws_bytes);
    if (r != MOE_OK) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (shape->T == 0)
        return cuda_status(cudaMemsetAsync(dw1, 0, 4 * static_cast<size_t>(shape->E) * shape->I * shape->H, st));
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    return run_bwd_stage1_weight_mx(*shape, x, dw1, carve(ws, *shape), *d, st, ws);
}

moe_status_t moe_dispatch_rows(const void *x, const float *topk_w, const moe_shape_t *shape, void *rows,
                               float *row_weight, void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;
    if (x == nullptr || rows == nullptr || !aligned16(x) || !aligned16(rows)) return MOE_ERR_INVALID_ARG;
    if (row_weight != nullptr && (topk_w == nullptr || (reinterpret_cast<uintptr_t>(row_weight) & 3u) ||
                                  (reinterpret_cast<uintptr_t>(topk_w) & 3u)))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *shape);
    return cuda_status(launch_dispatch_rows(static_cast<const __nv_bfloat16 *>(x), w.row_of, shape->T, shape->k,
                                            shape->H, static_cast<__nv_bfloat16 *>(rows), topk_w, row_weight,
                                            static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_combine_rows(const void *rows, const moe_shape_t *shape, void *y, void *ws, size_t ws_bytes,
                              void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (shape->T == 0) return MOE_OK;
    if (rows == nullptr || y == nullptr || !aligned16(rows) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *shape);
    CombineLaunch c;
    c.obuf = static_cast<const __nv_bfloat16 *>(rows);
    c.row_of = w.row_of;
    c.y = static_cast<__nv_bfloat16 *>(y);
    c.T = static_cast<int>(shape->T);
    c.H = static_cast<int>(shape->H);
    c.k = shape->k;
    return cuda_status(launch_combine(c, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_ep_pack(const void *x, const float *topk_w, const moe_shape_t *shape, int32_t n_ranks,
                         int64_t capacity, void *send_rows, float *send_w, int32_t *send_counts, void *ws,
                         size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (n_ranks < 1 || shape->E % n_ranks != 0 || capacity < 1) return MOE_ERR_INVALID_ARG;
    if (capacity * n_ranks >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (send_rows == nullptr || send_w == nullptr || send_counts == nullptr || !aligned16(send_rows) ||
        (reinterpret_cast<uintptr_t>(send_w) & 3u) || (reinterpret_cast<uintptr_t>(send_counts) & 3u))
        return MOE_ERR_INVALID_ARG;
    if (shape->T == 0)      // nothing to send: every count is zero
        return cuda_status(cudaMemsetAsync(send_counts, 0, 4 * static_cast<size_t>(shape->E),
                                           static_cast<cudaStream_t>(stream)));
    if (x == nullptr || topk_w == nullptr || !aligned16(x) || (reinterpret_cast<uintptr_t>(topk_w) & 3u))
        return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *shape);
    EpPackLaunch p;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.topk_w = topk_w;
    p.row_of = w.row_of;
    p.counts = w.counts;
    p.offsets = w.offsets;
    p.T = static_cast<int>(shape->T);
    p.k = shape->k;
    p.H = shape->H;
    p.E = static_cast<int>(shape->E);
    p.E_loc = static_cast<int>(shape->E / n_ranks);
    p.C = capacity;
    p.send_rows = static_cast<__nv_bfloat16 *>(send_rows);
    p.send_w = send_w;
    p.send_counts = send_counts;
    p.err = w.err;
    return cuda_status(launch_ep_pack(p, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_ep_receive_metadata(const int32_t *recv_counts, int32_t n_ranks, int64_t capacity,
                                     const moe_shape_t *recv_shape, void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(recv_shape);
    if (r != MOE_OK) return r;
    if (n_ranks < 1 || capacity < 1 || recv_shape->k != 1 || recv_shape->T != n_ranks * capacity)
        return MOE_ERR_INVALID_ARG;
    if (recv_counts == nullptr || (reinterpret_cast<uintptr_t>(recv_counts) & 3u)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*recv_shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *recv_shape);
    EpRecvLaunch p;
    p.recv = recv_counts;
    p.P = n_ranks;
    p.E_loc = static_cast<int>(recv_shape->E);
    p.C = capacity;
    p.n_tiles = static_cast<int>((recv_shape->H + kBN - 1) / kBN);
    p.counts = w.counts;
    p.offsets = w.offsets;
    p.mt_prefix = w.mt_prefix;
    p.perm_slot = w.perm_slot;
    p.row_of = w.row_of;
    p.ccnt = w.combine;
    p.err = w.err;
    return cuda_status(launch_ep_receive_metadata(p, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_ep_combine(const void *back_rows, const moe_shape_t *shape, int32_t n_ranks, int64_t capacity,
                            void *y, void *ws, size_t ws_bytes, void *stream) {
    moe_status_t r = check_shape(shape);
    if (r != MOE_OK) return r;
    if (n_ranks < 1 || shape->E % n_ranks != 0 || capacity < 1) return MOE_ERR_INVALID_ARG;
    if (shape->T == 0) return MOE_OK;
    if (back_rows == nullptr || y == nullptr || !aligned16(back_rows) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    if ((r = check_ws(*shape, ws, ws_bytes)) != MOE_OK) return r;
    DeviceState *d = nullptr;
    if ((r = device_state(&d)) != MOE_OK) return r;
    const Ws w = carve(ws, *shape);
    EpCombineLaunch p;
    p.back = static_cast<const __nv_bfloat16 *>(back_rows);
    p.row_of = w.row_of;
    p.offsets = w.offsets;
    p.T = static_cast<int>(shape->T);
    p.k = shape->k;
    p.H = static_cast<int>(shape->H);
    p.E = static_cast<int>(shape->E);
    p.E_loc = static_cast<int>(shape->E / n_ranks);
    p.C = capacity;
    p.y = static_cast<__nv_bfloat16 *>(y);
    return cuda_status(launch_ep_combine(p, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_get_device_error(void *ws, int32_t *code, void *stream) {
    if (ws == nullptr || code == nullptr) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    *code = v;
    if (v == 0) return MOE_OK;
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_ERR_DEVICE_FLAGGED;
}

const char *moe_status_string(moe_status_t status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported shape, configuration or device";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_DEVICE_FLAGGED: return "device error word set";
    }
    return "unknown status";
}

uint64_t moe_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
