// rows.cu -- the row movements of expert parallelism across devices (MegaMoE
// guide, opening section: dispatch_grouped_gemm fuses the token dispatch
// all-to-all, grouped_gemm_combine the combine all-to-all). With the exchange
// done by the caller's collective, the device work on each side is a copy of
// the token rows into routed order (the send buffer of the dispatch; on one
// device, the A rows of stage 1) and, after the return exchange, the k-way sum
// of the returned rows (the combine).
#include "internal.cuh"

namespace moe {

namespace {

// The dispatch copy: rows[row_of[t k + j], :] = x[t, :] for every slot (t, j)
// with row_of >= 0 (dropped slots have none), and with row_w also
// row_w[row_of[s]] = topk_w[s]. One warp per token (grid-stride over tokens):
// the token's row is read once, eight 16-byte chunks per lane at a time, and
// stored to each of its k routed rows, so x is read T H times rather than
// T k H times (a gather by routed row would load the row once per slot).
__global__ void __launch_bounds__(256)
dispatch_rows_kernel(const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ row_of, int T, int k,
                     int64_t H, __nv_bfloat16 *__restrict__ rows, const float *__restrict__ topk_w,
                     float *__restrict__ row_w) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int chunks = static_cast<int>(H / 8);
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const int my_row = lane < k ? __ldg(&row_of[t * k + lane]) : -1;
        if (row_w != nullptr && my_row >= 0) row_w[my_row] = topk_w[t * k + lane];
        const uint4 *src = reinterpret_cast<const uint4 *>(x + t * H);
        for (int cb = 0; cb < chunks; cb += 256) {    // the same passes on every lane (shuffles below)
            const int c0 = cb + lane;
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = (c0 + 32 * j < chunks) ? __ldg(src + c0 + 32 * j) : make_uint4(0u, 0u, 0u, 0u);
            for (int j2 = 0; j2 < k; ++j2) {
                const int r = __shfl_sync(0xffffffffu, my_row, j2);
                if (r < 0) continue;                       // a dropped slot (the same for the whole warp)
                uint4 *dst = reinterpret_cast<uint4 *>(rows + static_cast<int64_t>(r) * H);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (c0 + 32 * j < chunks) dst[c0 + 32 * j] = v[j];
            }
        }
    }
}

}  // namespace

cudaError_t launch_dispatch_rows(const __nv_bfloat16 *x, const int32_t *row_of, int64_t T, int k, int64_t H,
                                 __nv_bfloat16 *rows, const float *topk_w, float *row_w, cudaStream_t st) {
    if (T == 0 || H == 0) return cudaSuccess;
    int64_t grid = (T + 7) / 8;                     // eight tokens (warps) per block
    if (grid > 152 * 8) grid = 152 * 8;
    const cudaError_t e = launch_dep(dispatch_rows_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, x, row_of,
                                     static_cast<int>(T), k, H, rows, topk_w, row_w);
    note_launches(1);
    return e;
}

}  // namespace moe
