// router_noalloc.cu -- moe_router_noalloc: the router for callers that cannot
// allocate device memory and so cannot hand the library a workspace.
//
// Such callers are plug-ins hosted by a runtime that owns every byte of device
// memory (an inference engine or serving process with a fixed pool that has
// already been carved up): they are not allowed to call cudaMalloc, and their
// host gives them no spare buffer for the router's intermediate logits. This
// entry point therefore keeps that scratch in a fixed-size array that lives
// inside the library image itself.
//
// It runs exactly the same kernels as moe_router; only the location of the
// scratch differs.
#include <mutex>

#include "internal.cuh"

namespace moe {

namespace {

// Capacity of the static scratch: split-K partial logits for at most
// kMaxPartials = splits * T * E values (4 MiB), the bf16 x3 split of w_r for at
// most E * H = kMaxEH weights (6 MiB), per-expert sums and counts for up to
// 1024 experts, the block ticket, the GEMM unit scheduler and an error word.
constexpr int64_t kMaxPartials = int64_t(1) << 20;
constexpr int64_t kMaxEH = int64_t(1) << 20;
constexpr size_t kScratchBytes = (size_t(4) << 20) + (size_t(6) << 20) + 4096 + 4096 + 1024;

// Every GPU that loads this library holds this array until the process exits.
// All calls on a device share it, so calls whose kernels overlap on the GPU
// (different streams without ordering between them) race on it.
static __device__ __align__(256) unsigned char g_router_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
bool g_ready[kMaxDevices];
moe_status_t g_status[kMaxDevices];
unsigned char *g_scratch_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];

// Once per device, with that device current: check the architecture and look
// up the device address of the static array (a host-side use of its name is
// only a stand-in, not a device pointer). A device is marked ready only when
// every step succeeded; an unsupported architecture is remembered, any other
// failure is retried by the next call.
moe_status_t scratch_for_current_device(unsigned char **out, int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_ready[dev]) {
        int major = 0, minor = 0, sms = 0;
        void *p = nullptr;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();   // clear only the error this set-up caused
            return MOE_ERR_CUDA;
        }
        if (major != 10 || minor != 3) {
            g_status[dev] = MOE_ERR_UNSUPPORTED;
            g_ready[dev] = true;
        } else if (cudaGetSymbolAddress(&p, g_router_scratch) != cudaSuccess || p == nullptr ||
                   setup_gemm_kernels() != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        } else {
            g_status[dev] = MOE_OK;
            g_scratch_ptr[dev] = static_cast<unsigned char *>(p);
            g_num_sms[dev] = sms;
            g_ready[dev] = true;
        }
    }
    *out = g_scratch_ptr[dev];
    *num_sms = g_num_sms[dev];
    return g_status[dev];
}

// The error word sits at a fixed place in the array's last 256 bytes.
int32_t *error_word(unsigned char *scratch) { return reinterpret_cast<int32_t *>(scratch + kScratchBytes - 256); }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_router_noalloc(const void *x, const float *w_r,
                                           const float *logit_offset, const float *sel_bias,
                                           const moe_shape_t *shape, const moe_router_cfg_t *cfg,
                                           int32_t *topk_idx, float *topk_w, float *aux,
                                           void *stream) {
    if (shape == nullptr || cfg == nullptr) return MOE_ERR_INVALID_ARG;
    const moe_shape_t &s = *shape;
    if (s.T < 0 || s.H <= 0 || s.I <= 0 || s.E <= 0 || s.k <= 0 || (s.flags & ~MOE_SHAPE_TRAINING) != 0)
        return MOE_ERR_INVALID_ARG;
    if (s.k > 32 || s.k > s.E || s.E > 1024 || s.H % 8 != 0 || s.I % 8 != 0 ||
        s.H >= (int64_t(1) << 31) || s.T * s.k >= (int64_t(1) << 31))
        return MOE_ERR_UNSUPPORTED;
    // the static scratch must hold the split weights and one partial per split
    if (s.T * s.E > kMaxPartials || s.E * s.H > kMaxEH) return MOE_ERR_UNSUPPORTED;
    if (s.T == 0) return MOE_OK;
    if (x == nullptr || w_r == nullptr || topk_idx == nullptr || topk_w == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w_r, 16) || !aligned(topk_idx, 16) || !aligned(topk_w, 16) ||
        !aligned(logit_offset, 4) || !aligned(sel_bias, 4) || !aligned(aux, 4))
        return MOE_ERR_INVALID_ARG;
    if (cfg->score_fn != MOE_SCORE_SOFTMAX && cfg->score_fn != MOE_SCORE_SIGMOID) return MOE_ERR_INVALID_ARG;
    if (cfg->n_group < 1 || cfg->n_group > 32) return MOE_ERR_UNSUPPORTED;
    if (cfg->n_group > 1) {
        if (s.E % cfg->n_group != 0 || cfg->topk_group < 1 || cfg->topk_group > cfg->n_group ||
            cfg->group_topn < 1 || cfg->group_topn > s.E / cfg->n_group ||
            static_cast<int64_t>(cfg->topk_group) * (s.E / cfg->n_group) < s.k)
            return MOE_ERR_INVALID_ARG;
    }
    unsigned char *scratch = nullptr;
    int num_sms = 0;
    moe_status_t r = scratch_for_current_device(&scratch, &num_sms);
    if (r != MOE_OK) return r;

    // the workspace router's split factor, lowered until the partials fit
    int splits = router_splits(s.T, s.H, s.E);
    const int64_t cap = kMaxPartials / (s.T * s.E);
    if (splits > cap) {
        const int64_t kb_total = router_kb_total(s.H, s.E);
        const int64_t per = (kb_total + cap - 1) / cap;
        splits = static_cast<int>((kb_total + per - 1) / per);
    }

    RouterLaunch p;
    p.x = static_cast<const __nv_bfloat16 *>(x);
    p.w_r = w_r;
    p.logit_offset = logit_offset;
    p.sel_bias = sel_bias;
    p.T = static_cast<int>(s.T);
    p.H = static_cast<int>(s.H);
    p.E = static_cast<int>(s.E);
    p.k = s.k;
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
    // the split kernel clears the sums, counts and ticket at the start of every
    // call, and the GEMM's unit counter (zero when the library is loaded)
    // returns to zero at the end of every launch, so nothing an earlier call
    // left in the array is read
    // The error word, the top-k ticket and the GEMM unit counter sit at fixed
    // places in the last 256 bytes, never inside a region whose position
    // depends on the shape: the counter must read zero at the start of every
    // launch, and a shape-dependent place could hold another call's logits.
    unsigned char *tail = scratch + kScratchBytes - 256;
    p.err = error_word(scratch);
    p.num_sms = num_sms;
    p.scratch = carve_router_scratch(scratch, s.T, s.H, s.E, splits,
                                     reinterpret_cast<int32_t *>(tail + 64),
                                     reinterpret_cast<int32_t *>(tail + 128));
    return launch_router(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_router_noalloc_get_error(int32_t *code, void *stream) {
    if (code == nullptr) return MOE_ERR_INVALID_ARG;
    unsigned char *scratch = nullptr;
    int num_sms = 0;
    moe_status_t r = scratch_for_current_device(&scratch, &num_sms);
    if (r != MOE_OK) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t *word = error_word(scratch);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, word, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    *code = v;
    if (v == 0) return MOE_OK;
    if (cudaMemsetAsync(word, 0, sizeof(int32_t), st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_ERR_DEVICE_FLAGGED;
}
