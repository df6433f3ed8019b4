// grouped_gemm_mx.cu -- the MXFP8 expert precision (MegaMoE guide, section
// "Expert precision": mxfp8 runs the two expert stages in MXFP8): the
// quantization kernel (bf16 -> E4M3 codes + E8M0 scales per 32 elements) and
// the MXFP8 instantiations of the grouped-GEMM kernel (block-scaled tcgen05
// MMAs, kind::mxf8f6f4, scale factors staged in tensor memory per stage).
#include "gemm_kernel.cuh"

namespace moe {

namespace {

// One thread per 32-element block; block b of a row-major [rows, cols] matrix
// (cols % 32 == 0) is elements [32 b, 32 b + 32) and scale b.
__global__ void __launch_bounds__(256)
mx_quantize_kernel(const __nv_bfloat16 *__restrict__ in, int64_t blocks, uint8_t *__restrict__ codes,
                   uint8_t *__restrict__ scales) {
    griddep_wait();
    for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < blocks;
         b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 *src = reinterpret_cast<const uint4 *>(in + b * 32);
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 w = __ldg(src + q);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * q + 2 * j] = bf16_lo(u[j]);
                v[8 * q + 2 * j + 1] = bf16_hi(u[j]);
            }
        }
        uint32_t qw[8];
        const uint32_t sc = mx_quantize32(v, qw);
        uint4 *dst = reinterpret_cast<uint4 *>(codes + b * 32);
        dst[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
        dst[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
        scales[b] = static_cast<uint8_t>(sc);
    }
}

// The dispatch of the MXFP8 path, fused into the quantization of x: routed
// row r (r < *routed) is token perm_slot[r] / k, quantized into row r of
// codes [R, cols] and scales [R, cols / 32], so stage 1 reads its A tiles with
// plain TMA copies.
__global__ void __launch_bounds__(256)
mx_quantize_dispatch_kernel(const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ perm_slot,
                            const int32_t *__restrict__ routed, int k, int64_t cols, uint8_t *__restrict__ codes,
                            uint8_t *__restrict__ scales) {
    griddep_wait();
    const int64_t per_row = cols / 32;
    const int64_t blocks = static_cast<int64_t>(*routed) * per_row;
    for (int64_t b = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < blocks;
         b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = b / per_row;
        const int64_t c = b - r * per_row;
        const int64_t t = perm_slot[r] / k;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + t * cols + c * 32);
        float v[32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 w = __ldg(src + q);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * q + 2 * j] = bf16_lo(u[j]);
                v[8 * q + 2 * j + 1] = bf16_hi(u[j]);
            }
        }
        uint32_t qw[8];
        const uint32_t sc = mx_quantize32(v, qw);
        uint4 *dst = reinterpret_cast<uint4 *>(codes + b * 32);
        dst[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
        dst[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
        scales[b] = static_cast<uint8_t>(sc);
    }
}

}  // namespace

cudaError_t launch_mx_quantize_dispatch(const __nv_bfloat16 *x, const int32_t *perm_slot, const int32_t *routed,
                                        int k, int64_t R, int64_t cols, uint8_t *codes, uint8_t *scales,
                                        cudaStream_t st) {
    const int64_t blocks = R * (cols / 32);
    if (blocks == 0) return cudaSuccess;
    int64_t grid = (blocks + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    const cudaError_t e = launch_dep(mx_quantize_dispatch_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, x,
                                     perm_slot, routed, k, cols, codes, scales);
    note_launches(1);
    return e;
}

cudaError_t setup_mx_gemm_kernels() {
    cudaError_t e = set_gemm_smem<kStage1Mx>();
    if (e == cudaSuccess) e = set_gemm_smem<kStage2Mx>();
    return e;
}

cudaError_t launch_mx_quantize(const __nv_bfloat16 *in, int64_t rows, int64_t cols, uint8_t *codes,
                               uint8_t *scales, cudaStream_t st) {
    const int64_t blocks = rows * (cols / 32);
    if (blocks == 0) return cudaSuccess;
    int64_t grid = (blocks + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    const cudaError_t e = launch_dep(mx_quantize_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, in, blocks,
                                     codes, scales);
    note_launches(1);
    return e;
}

cudaError_t launch_gemm1_mx(const GemmLaunch &p, cudaStream_t st) {
    return launch_tc_gemm<kStage1Mx>(maps_of(p), grouped_args(p), p.num_sms, st);
}

cudaError_t launch_gemm2_mx(const GemmLaunch &p, cudaStream_t st) {
    return launch_tc_gemm<kStage2Mx>(maps_of(p), grouped_args(p), p.num_sms, st);
}

}  // namespace moe
