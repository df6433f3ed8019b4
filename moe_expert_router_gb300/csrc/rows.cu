// rows.cu -- the row movements of expert parallelism across devices (MegaMoE
// guide, opening section: dispatch_grouped_gemm fuses the token dispatch
// all-to-all, grouped_gemm_combine the combine all-to-all). With the exchange
// done by the caller's collective, the device work on each side is a row
// gather into routed order (the send buffer of the dispatch) and, after the
// return exchange, the k-way sum of the returned rows (the combine).
#include "internal.cuh"

namespace moe {

namespace {

// rows[r, :] = x[perm_slot[r] / k, :] for r < *routed; with row_w, also
// row_w[r] = topk_w[perm_slot[r]]. One warp per row (grid-stride over rows),
// 16-byte chunks, eight loads in flight per lane.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ perm_slot,
                   const int32_t *__restrict__ routed, int k, int64_t H, __nv_bfloat16 *__restrict__ rows,
                   const float *__restrict__ topk_w, float *__restrict__ row_w) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int n = *routed;
    const int chunks = static_cast<int>(H / 8);
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); r < n; r += warps) {
        const int s = __ldg(&perm_slot[r]);
        const uint4 *src = reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(s / k) * H);
        uint4 *dst = reinterpret_cast<uint4 *>(rows + r * H);
        int c = lane;
        for (; c + 224 < chunks; c += 256) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __ldg(src + c + 32 * j);
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[c + 32 * j] = v[j];
        }
        for (; c < chunks; c += 32) dst[c] = __ldg(src + c);
        if (row_w != nullptr && lane == 0) row_w[r] = topk_w[s];
    }
}

}  // namespace

cudaError_t launch_gather_rows(const __nv_bfloat16 *x, const int32_t *perm_slot, const int32_t *routed, int k,
                               int64_t R, int64_t H, __nv_bfloat16 *rows, const float *topk_w, float *row_w,
                               cudaStream_t st) {
    if (R == 0 || H == 0) return cudaSuccess;
    int64_t grid = (R + 7) / 8;                     // eight rows (warps) per block
    if (grid > 152 * 8) grid = 152 * 8;
    const cudaError_t e = launch_dep(gather_rows_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, x, perm_slot,
                                     routed, k, H, rows, topk_w, row_w);
    note_launches(1);
    return e;
}

}  // namespace moe
