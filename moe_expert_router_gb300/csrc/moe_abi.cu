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
// dynamic shared memory limits.
moe_status_t device_state(DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        d.ready = true;
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            d.status = MOE_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            d.status = MOE_ERR_UNSUPPORTED;
        } else {
            d.num_sms = sms;
            if (setup_metadata_kernels() != cudaSuccess || setup_gemm_kernels() != cudaSuccess) {
                d.status = MOE_ERR_CUDA;
            }
        }
        cudaGetLastError();  // do not leak a set-up error into the caller's error state
    }
    *out = &d;
    return d.status;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_shape(const moe_shape_t *s) {
    if (s == nullptr) return MOE_ERR_INVALID_ARG;
    if (s->T < 0 || s->H <= 0 || s->I <= 0 || s->E <= 0 || s->k <= 0 || s->reserved != 0)
        return MOE_ERR_INVALID_ARG;
    if (s->k > 32 || s->k > s->E || s->E > 1024) return MOE_ERR_UNSUPPORTED;
    if (s->H % 8 != 0 || s->I % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->T * s->k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    if (s->E * 2 * s->I >= (int64_t(1) << 31) || s->E * s->H >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    if (s->H >= (int64_t(1) << 31) || s->I >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
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
    L.total = off;
    return L;
}

struct Ws {
    int32_t *err, *ticket, *counts, *offsets, *mt_prefix, *perm_slot, *row_of, *sched1, *sched2;
    int32_t *meta, *meta_ticket;
    RouterScratch router;
    __nv_bfloat16 *a, *obuf;
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
    w.router = carve_router_scratch(b + L.router, s.T, s.H, s.E, router_splits(s.T, s.H, s.E),
                                    w.ticket, reinterpret_cast<int32_t *>(b + 24));
    w.a = reinterpret_cast<__nv_bfloat16 *>(b + L.a);
    w.obuf = reinterpret_cast<__nv_bfloat16 *>(b + L.obuf);
    return w;
}

moe_status_t check_ws(const moe_shape_t &s, const void *ws, size_t ws_bytes) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < make_layout(s).total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Stage 1: tensor maps + launch (metadata must already be in ws).
moe_status_t run_gemm1(const moe_shape_t &s, const void *x, const void *w1, void *a, const Ws &w,
                       const DeviceState &d, cudaStream_t st) {
    // the x rows are gathered by the kernel's own warps; only w1 goes through TMA
    CUtensorMap tm_w1, tm_out;
    if (!encode_bf16_2d(&tm_w1, w1, s.H, static_cast<uint64_t>(s.E) * 2 * s.I, kBK, 128) ||
        !encode_bf16_2d(&tm_out, a, s.I, static_cast<uint64_t>(s.T) * s.k, 64, 32))
        return MOE_ERR_CUDA;
    GemmLaunch p;
    p.tm_a = &tm_w1;
    p.tm_b = &tm_w1;
    p.tm_out = &tm_out;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.counts = w.counts;
    p.offsets = w.offsets;
    p.mt_prefix = w.mt_prefix;
    p.perm_slot = w.perm_slot;
    p.err = w.err;
    p.sched = w.sched1;
    p.topk_w = nullptr;
    p.out = static_cast<__nv_bfloat16 *>(a);
    p.E = static_cast<int>(s.E);
    p.k = s.k;
    p.K = static_cast<int>(s.H);
    p.n_out = static_cast<int>(s.I);
    p.b_rows = static_cast<int>(2 * s.I);
    p.half = static_cast<int>(s.I);
    p.num_sms = d.num_sms;
    return cuda_status(launch_gemm1_swiglu(p, st));
}

// Stage 2: GEMM2 with the weighted scatter, then the k-way combine.
moe_status_t run_gemm2(const moe_shape_t &s, const void *a, const float *topk_w, const void *w2,
                       void *y, const Ws &w, const DeviceState &d, cudaStream_t st) {
    CUtensorMap tm_a, tm_w2, tm_out;
    const uint64_t R = static_cast<uint64_t>(s.T) * s.k;
    if (!encode_bf16_2d(&tm_a, a, s.I, R, kBK, 128)) return MOE_ERR_CUDA;
    if (!encode_bf16_2d(&tm_w2, w2, s.I, static_cast<uint64_t>(s.E) * s.H, kBK, 256))
        return MOE_ERR_CUDA;
    if (!encode_bf16_2d(&tm_out, w.obuf, s.H, R, 64, 32)) return MOE_ERR_CUDA;
    GemmLaunch p;
    p.tm_a = &tm_a;
    p.tm_b = &tm_w2;
    p.tm_out = &tm_out;
    p.x = nullptr;
    p.counts = w.counts;
    p.offsets = w.offsets;
    p.mt_prefix = w.mt_prefix;
    p.perm_slot = w.perm_slot;
    p.err = w.err;
    p.sched = w.sched2;
    p.topk_w = topk_w;
    p.out = w.obuf;
    p.E = static_cast<int>(s.E);
    p.k = s.k;
    p.K = static_cast<int>(s.I);
    p.n_out = static_cast<int>(s.H);
    p.b_rows = static_cast<int>(s.H);
    p.half = 0;
    p.num_sms = d.num_sms;
    moe_status_t r = cuda_status(launch_gemm2_scatter(p, st));
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

bool encode_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows) {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        cudaGetLastError();
    });
    if (g_encode == nullptr) return false;
    if (box_inner * 2 != 128 && box_inner * 2 != 64) return false;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * 2};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    box_inner * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

moe_status_t moe_router(const void *x, const float *w_r, const float *logit_offset,
                        const float *sel_bias, const moe_shape_t *shape,
                        const moe_router_cfg_t *cfg, int32_t *topk_idx, float *topk_w, float *aux,
                        void *ws, size_t ws_bytes, void *stream) {
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
    if (cfg->score_fn != MOE_SCORE_SOFTMAX && cfg->score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (cfg->n_group < 1 || cfg->n_group > 32) return MOE_ERR_UNSUPPORTED;
    if (cfg->n_group > 1) {
        if (shape->E % cfg->n_group != 0 || cfg->topk_group < 1 || cfg->topk_group > cfg->n_group ||
            cfg->group_topn < 1 || cfg->group_topn > shape->E / cfg->n_group)
            return MOE_ERR_INVALID_ARG;
        if (static_cast<int64_t>(cfg->topk_group) * (shape->E / cfg->n_group) < shape->k)
            return MOE_ERR_INVALID_ARG;
    }
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
    p.err = w.err;
    p.num_sms = d->num_sms;
    p.scratch = w.router;
    return cuda_status(launch_router(p, static_cast<cudaStream_t>(stream)));
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
    return run_gemm1(*shape, x, w1, a, carve(ws, *shape), *d, static_cast<cudaStream_t>(stream));
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
    if ((r = run_gemm1(*shape, x, w1, w.a, w, *d, st)) != MOE_OK) return r;
    return run_gemm2(*shape, w.a, topk_w, w2, y, w, *d, st);
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
