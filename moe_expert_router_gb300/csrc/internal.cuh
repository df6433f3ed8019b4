// internal.cuh -- declarations shared by the CUDA translation units of libmoe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Rows (routed tokens) per GEMM tile; the routing metadata counts row tiles in
// these units, so every grouped GEMM uses the same value.
constexpr int kBM = 128;

// Workspace header: int32 error word at byte 0, int32 router ticket at byte 4.
constexpr size_t kWsHeaderBytes = 256;

struct RouterScratch {
    float *logits;      // [T, E]
    float *score_sum;   // [E]  sum over tokens of the full score vector
    int32_t *counts;    // [E]  rows the router sent to each expert
    int32_t *ticket;    // blocks of the top-k kernel that have finished
};

struct RouterLaunch {
    const __nv_bfloat16 *x;
    const float *w_r;
    const float *logit_offset;  // may be null
    const float *sel_bias;      // may be null
    int T, H, E, k;
    int score_fn, normalize;
    float scale;
    int n_group, topk_group, group_topn;
    int32_t *topk_idx;
    float *topk_w;
    float *aux;                 // may be null
    RouterScratch scratch;
};

struct MetadataLaunch {
    const int32_t *topk_idx;
    int R, E;
    int32_t *counts, *offsets, *mt_prefix, *perm_slot, *row_of, *err;
};

// One grouped GEMM launch: stage 1 (SwiGLU epilogue) or stage 2 (weighted scatter).
struct GemmLaunch {
    const CUtensorMap *tm_a;    // host-encoded tensor maps (copied into the launch)
    const CUtensorMap *tm_b;
    const int32_t *counts, *offsets, *mt_prefix, *perm_slot;
    int32_t *err;
    const float *topk_w;        // stage 2 only
    __nv_bfloat16 *out;         // a [R, I] (stage 1) or obuf [R, H] (stage 2)
    int E, k, K, n_out, b_rows, half;
    int num_sms;
};

struct CombineLaunch {
    const __nv_bfloat16 *obuf;
    const int32_t *row_of;
    __nv_bfloat16 *y;
    int T, H, k;
};

cudaError_t launch_router(const RouterLaunch &p, cudaStream_t st);
cudaError_t launch_routing_metadata(const MetadataLaunch &p, cudaStream_t st);
cudaError_t launch_gemm1_swiglu(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_gemm2_scatter(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_combine(const CombineLaunch &p, cudaStream_t st);

// Per-device one-time kernel attribute set-up (dynamic shared memory limits).
cudaError_t setup_router_kernels();
cudaError_t setup_metadata_kernels();
cudaError_t setup_gemm_kernels();

// Statistics: kernels launched by this library.
void note_launches(int n);

}  // namespace moe
