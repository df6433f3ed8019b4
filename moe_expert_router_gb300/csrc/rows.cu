// rows.cu -- the row movements of expert parallelism across devices (MegaMoE
// guide, opening section: dispatch_grouped_gemm fuses the token dispatch
// all-to-all, grouped_gemm_combine the combine all-to-all). With the exchange
// done by the caller's collective, the device work on each side is a row
// gather into routed order (the send buffer of the dispatch) and, after the
// return exchange, the k-way sum of the returned rows (the combine).
#include "internal.cuh"

namespace moe {

namespace {

// rows[r, :] = x[perm_slot[r] / k, :] for r < *routed (16-byte chunks); with
// row_w, also row_w[r] = topk_w[perm_slot[r]].
__global__ void __launch_bounds__(256)
gather_rows_kernel(const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ perm_slot,
                   const int32_t *__restrict__ routed, int k, int64_t H, __nv_bfloat16 *__restrict__ rows,
                   const float *__restrict__ topk_w, float *__restrict__ row_w) {
    const int64_t per_row = H / 8;
    const int64_t total = static_cast<int64_t>(*routed) * per_row;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / per_row;
        const int64_t c = (i - r * per_row) * 8;
        const int64_t s = perm_slot[r];
        *reinterpret_cast<uint4 *>(rows + r * H + c) = __ldg(reinterpret_cast<const uint4 *>(x + (s / k) * H + c));
        if (row_w != nullptr && c == 0) row_w[r] = topk_w[s];
    }
}

}  // namespace

cudaError_t launch_gather_rows(const __nv_bfloat16 *x, const int32_t *perm_slot, const int32_t *routed, int k,
                               int64_t R, int64_t H, __nv_bfloat16 *rows, const float *topk_w, float *row_w,
                               cudaStream_t st) {
    const int64_t total = R * (H / 8);
    if (total == 0) return cudaSuccess;
    int64_t grid = (total + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    gather_rows_kernel<<<static_cast<int>(grid), 256, 0, st>>>(x, perm_slot, routed, k, H, rows, topk_w, row_w);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
