// backward.cu -- the light kernels of the backward around the grouped GEMMs:
// the routing-weight gradient, the router backward (logit gradient and dW_r)
// and the per-token sum that gives dX.
//
// Router backward (the router of the MegaMoE guide's opening section, taken
// through the weights; the selection is piecewise constant and passes no
// gradient). With K the chosen experts of a token, w their weights, dw the
// gradient of w and l the logits:
//   softmax, normalised: dl_i = w_i dw_i - (w_i / scale) sum_K w_j dw_j   (i in K)
//   softmax, plain:      dl_e = scale s_e ([e in K] dw_e - sum_K s_j dw_j) (all e)
//   sigmoid, normalised: dl_i = s_i (1 - s_i) / S (scale dw_i - sum_K w_j dw_j), S = sum_K s
//   sigmoid, plain:      dl_i = scale s_i (1 - s_i) dw_i
// then dX += dl . W_r and dW_r = dl^T . x (fp32).
#include <math.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

__global__ void __launch_bounds__(256)
dtw_reduce_kernel(const float *__restrict__ part, int n_part, int R, const int32_t *__restrict__ row_of,
                  float *__restrict__ dtopk_w, int64_t slots) {
    griddep_wait();
    for (int64_t s = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; s < slots;
         s += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int r = row_of[s];
        float acc = 0.0f;
        if (r >= 0)
            for (int n = 0; n < n_part; ++n) acc += part[static_cast<int64_t>(n) * R + r];
        dtopk_w[s] = acc;
    }
}

// One warp per token; lane j < k owns slot j.
__global__ void __launch_bounds__(256)
router_dlogits_kernel(const RouterBwdLaunch p) {
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= p.T) return;
    const float *lrow = p.logits + static_cast<int64_t>(t) * p.E;
    float *dl = p.dl + static_cast<int64_t>(t) * p.E;
    const bool mine = lane < p.k;
    const int e = mine ? p.topk_idx[static_cast<int64_t>(t) * p.k + lane] : -1;
    const bool ok = mine && e >= 0 && e < p.E;
    const float w = ok ? p.topk_w[static_cast<int64_t>(t) * p.k + lane] : 0.0f;
    const float dw = ok ? p.dtopk_w[static_cast<int64_t>(t) * p.k + lane] : 0.0f;
    // products rounded on their own (no fused multiply-add), so that where the
    // normalisation makes a weight constant (k = 1: w = scale) its terms cancel
    // exactly and the logit gradient is exactly 0
    const float sum_wdw = warp_sum(__fmul_rn(w, dw));
    if (p.score_fn == MOE_SCORE_SOFTMAX && !p.normalize) {
        float m = -INFINITY;
        for (int i = lane; i < p.E; i += 32) m = fmaxf(m, lrow[i]);
        m = warp_max(m);
        float z = 0.0f;
        for (int i = lane; i < p.E; i += 32) z += expf(lrow[i] - m);
        z = warp_sum(z);
        const float inv_z = 1.0f / z;
        const float s_own = ok ? expf(lrow[e] - m) * inv_z : 0.0f;
        const float sum_sdw = warp_sum(s_own * dw);
        for (int i = lane; i < p.E; i += 32) dl[i] = -p.scale * expf(lrow[i] - m) * inv_z * sum_sdw;
        __syncwarp();
        if (ok) atomicAdd(&dl[e], p.scale * s_own * dw);
        return;
    }
    for (int i = lane; i < p.E; i += 32) dl[i] = 0.0f;
    __syncwarp();
    if (p.score_fn == MOE_SCORE_SOFTMAX) {
        if (ok) atomicAdd(&dl[e], __fmul_rn(w, dw) - __fmul_rn(w / p.scale, sum_wdw));
        return;
    }
    const float s = ok ? 1.0f / (1.0f + expf(-lrow[e])) : 0.0f;
    if (p.normalize) {
        const float S = warp_sum(s);
        if (ok) atomicAdd(&dl[e], s * (1.0f - s) / S * (__fmul_rn(p.scale, dw) - sum_wdw));
    } else {
        if (ok) atomicAdd(&dl[e], p.scale * s * (1.0f - s) * dw);
    }
}

// True when slot j of token t is the first of the token's slots on expert e
// (a token's logit gradient for e is counted once however often e repeats).
__device__ __forceinline__ bool first_slot(const int32_t *__restrict__ idx_t, int j, int e) {
    for (int jj = 0; jj < j; ++jj)
        if (idx_t[jj] == e) return false;
    return true;
}

// Partial dW_r: block (e, 1024-column chunk, row segment) sums, for its thread's
// 8 columns, the rows of the batches of 128 rows numbered segment, segment +
// kDwrSegments, ... Sparse modes walk the expert's routed rows; the dense mode
// (plain softmax) walks every token. Each thread first resolves one row's token
// and logit gradient into shared memory; then every thread accumulates the
// batch's x rows, eight row loads in flight at a time.
constexpr int kDwrThreads = 128;

__global__ void __launch_bounds__(kDwrThreads)
router_dwr_part_kernel(const RouterBwdLaunch p, int chunks, int dense) {
    griddep_wait();
    __shared__ int tok_sh[kDwrThreads];
    __shared__ float coef_sh[kDwrThreads];
    const int e = blockIdx.x / chunks;
    const int seg = blockIdx.y;
    const int c = ((blockIdx.x - e * chunks) * kDwrThreads + threadIdx.x) * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const int n = dense ? p.T : p.counts[e];
    const int r0 = dense ? 0 : p.offsets[e];
    for (int b0 = seg * kDwrThreads; b0 < n; b0 += kDwrSegments * kDwrThreads) {
        const int i = b0 + threadIdx.x;
        int t = -1;
        float coef = 0.0f;
        if (i < n) {
            if (dense) {
                t = i;
            } else {
                const int s = p.perm_slot[r0 + i];
                t = s / p.k;
                if (!first_slot(p.topk_idx + static_cast<int64_t>(t) * p.k, s - t * p.k, e)) t = -1;
            }
            if (t >= 0) coef = p.dl[static_cast<int64_t>(t) * p.E + e];
        }
        __syncthreads();                    // the previous batch is consumed
        tok_sh[threadIdx.x] = t;
        coef_sh[threadIdx.x] = coef;
        __syncthreads();
        if (c < p.H) {
            const int m = min(kDwrThreads, n - b0);
            for (int j0 = 0; j0 < m; j0 += 8) {
                uint4 v[8];
                float cf[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int tj = (j0 + jj < m) ? tok_sh[j0 + jj] : -1;
                    cf[jj] = tj >= 0 ? coef_sh[j0 + jj] : 0.0f;
                    v[jj] = tj >= 0 ? __ldg(reinterpret_cast<const uint4 *>(p.x + static_cast<int64_t>(tj) * p.H + c))
                                    : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const uint32_t wv[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = fmaf(cf[jj], __uint_as_float(wv[q] << 16), acc[2 * q]);
                        acc[2 * q + 1] = fmaf(cf[jj], __uint_as_float(wv[q] & 0xffff0000u), acc[2 * q + 1]);
                    }
                }
            }
        }
    }
    if (c < p.H) {
        float4 *dst = reinterpret_cast<float4 *>(p.dwr_part + (static_cast<int64_t>(seg) * p.E + e) * p.H + c);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}

// dW_r[e, h] = sum over the segments, in segment order, of the partial sums.
__global__ void __launch_bounds__(256)
router_dwr_sum_kernel(const float *__restrict__ part, int64_t n4, float *__restrict__ dw_r) {
    griddep_wait();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float4 a = __ldcg(reinterpret_cast<const float4 *>(part) + i);
#pragma unroll
        for (int s = 1; s < kDwrSegments; ++s) {
            const float4 b = __ldcg(reinterpret_cast<const float4 *>(part) + s * n4 + i);
            a.x += b.x;
            a.y += b.y;
            a.z += b.z;
            a.w += b.w;
        }
        reinterpret_cast<float4 *>(dw_r)[i] = a;
    }
}

// dX[t, :] = sum over t's slots of the dX rows (slot order), plus the router
// term sum_e dl[t, e] w_r[e, :] (expert order for the dense form, slot order
// over first occurrences otherwise). Block (64-token group, 256-column slice):
// each warp walks 8 of the group's tokens over the slice, lane l owning columns
// 8 l .. 8 l + 7, so the w_r rows of the slice (E x 1 KB) are re-read from L1 by
// the block's tokens rather than from L2 by every token. Lane j < k holds slot
// j's row and, for the sparse router term, its expert and logit gradient.
constexpr int kCbTokens = 64;                 // tokens per block (8 per warp)

__global__ void __launch_bounds__(256)
combine_bwd_kernel(const CombineBwdLaunch p) {
    griddep_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = blockIdx.y * 32 + lane;               // 8-column group of this lane
    const bool live = g < (p.H >> 3);
    const int c = g * 8;
    const int t_end = min(p.T, (blockIdx.x + 1) * kCbTokens);
    for (int t = blockIdx.x * kCbTokens + warp; t < t_end; t += 8) {
        const int32_t *idx_t = p.topk_idx + static_cast<int64_t>(t) * p.k;
        const float *dl_t = p.dl != nullptr ? p.dl + static_cast<int64_t>(t) * p.E : nullptr;
        const int my_row = lane < p.k ? __ldg(&p.row_of[static_cast<int64_t>(t) * p.k + lane]) : -1;
        int my_e = -1;
        float my_d = 0.0f;
        if (dl_t != nullptr && !p.dense && lane < p.k) {
            const int e = idx_t[lane];
            if (e >= 0 && e < p.E && first_slot(idx_t, lane, e)) {
                my_e = e;
                my_d = dl_t[e];
            }
        }
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < p.k; j0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int r = __shfl_sync(0xffffffffu, my_row, (j0 + jj) & 31);
                v[jj] = (live && j0 + jj < p.k && r >= 0)
                            ? __ldg(reinterpret_cast<const uint4 *>(p.xbuf + static_cast<int64_t>(r) * p.H + c))
                            : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const uint32_t wv[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] += __uint_as_float(wv[q] << 16);
                    acc[2 * q + 1] += __uint_as_float(wv[q] & 0xffff0000u);
                }
            }
        }
        if (dl_t != nullptr) {
            const int n = p.dense ? p.E : p.k;
            for (int j = 0; j < n; ++j) {
                int e = j;
                float d;
                if (p.dense) {
                    d = dl_t[e];
                } else {
                    e = __shfl_sync(0xffffffffu, my_e, j & 31);
                    d = __shfl_sync(0xffffffffu, my_d, j & 31);
                    if (e < 0) continue;
                }
                if (!live) continue;
                const float4 *wr = reinterpret_cast<const float4 *>(p.w_r + static_cast<int64_t>(e) * p.H + c);
                const float4 a = __ldg(wr), b = __ldg(wr + 1);
                acc[0] = fmaf(d, a.x, acc[0]);
                acc[1] = fmaf(d, a.y, acc[1]);
                acc[2] = fmaf(d, a.z, acc[2]);
                acc[3] = fmaf(d, a.w, acc[3]);
                acc[4] = fmaf(d, b.x, acc[4]);
                acc[5] = fmaf(d, b.y, acc[5]);
                acc[6] = fmaf(d, b.z, acc[6]);
                acc[7] = fmaf(d, b.w, acc[7]);
            }
        }
        if (live)
            *reinterpret_cast<uint4 *>(p.dx + static_cast<int64_t>(t) * p.H + c) =
                make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                           pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
}

// Rows [offsets[E], R) of dH and w a belong to no expert (slots dropped for an
// index outside [0, E)) and are never written by the dA GEMM; the weight-
// gradient GEMMs still read them as the K tail of the last expert (times
// zero-filled partners), so they must hold finite values: zeros.
__global__ void __launch_bounds__(256)
zero_tail_rows_kernel(__nv_bfloat16 *__restrict__ dh, __nv_bfloat16 *__restrict__ aw,
                      const int32_t *__restrict__ routed_rows, int R, int I) {
    griddep_wait();
    const int r0 = *routed_rows;
    const int64_t per_row = 3 * static_cast<int64_t>(I) / 8;   // 16-byte chunks: 2I of dH, I of w a
    const int64_t total = static_cast<int64_t>(R - r0) * per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = r0 + i / per_row;
        const int64_t c = (i % per_row) * 8;
        uint4 *dst = (c < 2 * I) ? reinterpret_cast<uint4 *>(dh + r * 2 * I + c)
                                 : reinterpret_cast<uint4 *>(aw + r * I + (c - 2 * I));
        *dst = make_uint4(0u, 0u, 0u, 0u);
    }
}

int grid_for(int64_t items, int per_block) {
    int64_t b = (items + per_block - 1) / per_block;
    if (b > 152 * 16) b = 152 * 16;
    return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_dtw_reduce(const DtwReduceLaunch &p, cudaStream_t st) {
    const int64_t slots = static_cast<int64_t>(p.T) * p.k;
    if (slots == 0) return cudaSuccess;
    const cudaError_t e = launch_dep(dtw_reduce_kernel, dim3(grid_for(slots, 256)), dim3(256), 0, st, p.dtw_part,
                                     p.n_part, p.R, p.row_of, p.dtopk_w, slots);
    note_launches(1);
    return e;
}

cudaError_t launch_zero_tail_rows(__nv_bfloat16 *dh, __nv_bfloat16 *aw, const int32_t *routed_rows, int R,
                                  int I, cudaStream_t st) {
    const cudaError_t e = launch_dep(zero_tail_rows_kernel, dim3(32), dim3(256), 0, st, dh, aw, routed_rows, R, I);
    note_launches(1);
    return e;
}

cudaError_t launch_router_dlogits(const RouterBwdLaunch &p, cudaStream_t st) {
    if (p.T == 0) return cudaSuccess;
    const cudaError_t e = launch_dep(router_dlogits_kernel, dim3((p.T + 7) / 8), dim3(256), 0, st, p);
    note_launches(1);
    return e;
}

cudaError_t launch_router_dwr(const RouterBwdLaunch &p, cudaStream_t st) {
    const int chunks = (p.H + 8 * kDwrThreads - 1) / (8 * kDwrThreads);
    const int dense = (p.score_fn == MOE_SCORE_SOFTMAX && !p.normalize) ? 1 : 0;
    cudaError_t e = launch_dep(router_dwr_part_kernel, dim3(p.E * chunks, kDwrSegments), dim3(kDwrThreads), 0, st, p,
                               chunks, dense);
    const int64_t n4 = static_cast<int64_t>(p.E) * p.H / 4;
    if (e == cudaSuccess)
        e = launch_dep(router_dwr_sum_kernel, dim3(grid_for(n4, 256)), dim3(256), 0, st,
                       static_cast<const float *>(p.dwr_part), n4, p.dw_r);
    note_launches(2);
    return e;
}

cudaError_t launch_combine_bwd(const CombineBwdLaunch &p, cudaStream_t st) {
    if (p.T == 0 || p.H == 0) return cudaSuccess;
    // 64-token groups x 256-column slices
    const dim3 grid((p.T + kCbTokens - 1) / kCbTokens, (p.H / 8 + 31) / 32);
    const cudaError_t e = launch_dep(combine_bwd_kernel, grid, dim3(256), 0, st, p);
    note_launches(1);
    return e;
}

}  // namespace moe
