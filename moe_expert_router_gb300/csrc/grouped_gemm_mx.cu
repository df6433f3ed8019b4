// grouped_gemm_mx.cu -- the MXFP8 expert precision (MegaMoE guide, section
// "Expert precision": mxfp8 runs the two expert stages in MXFP8): the
// quantization kernel (bf16 -> E4M3 codes + E8M0 scales per 32 elements) and
// the MXFP8 instantiations of the grouped-GEMM kernel (block-scaled tcgen05
// MMAs, kind::mxf8f6f4, scale factors staged in tensor memory per stage).
#include "gemm_kernel.cuh"

namespace moe {

namespace {

// Byte of block c (columns 32 c .. 32 c + 31) of row r in k-block-major scales
// over sf_rows rows: byte c % 4 of the 32-bit word [c / 4][r], one word per row
// and 128-column k-block of the block-scaled MMA.
__device__ __forceinline__ int64_t kmajor_scale_byte(int64_t r, int64_t c, int64_t sf_rows) {
    return (((c >> 2) * sf_rows + r) << 2) + (c & 3);
}

// Quantizes the 32 bf16 values at src into E4M3 codes at dst (32 bytes) and
// returns their E8M0 scale code.
__device__ __forceinline__ uint32_t quantize_block32(const __nv_bfloat16 *src, uint8_t *dst) {
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    float v[32];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint4 w = __ldg(s4 + q);
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * q + 2 * j] = bf16_lo(u[j]);
            v[8 * q + 2 * j + 1] = bf16_hi(u[j]);
        }
    }
    uint32_t qw[8];
    const uint32_t sc = mx_quantize32(v, qw);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    d4[0] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    d4[1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    return sc;
}

// Both quantizers give a warp 8 rows x one 128-column k-block per step: lane
// (i, j) = (lane / 4, lane % 4) quantizes block 4 kb + j of row 8 g + i, so the
// warp reads and writes 8 runs of 256 / 128 contiguous bytes and its 32 scale
// bytes are the 8 consecutive words [kb][8 g .. 8 g + 7], one 32-byte sector.

// A row-major [rows, cols] matrix (cols % 128 == 0): codes [rows, cols], scales
// k-block-major over sf_rows (rows rounded up to 4) rows.
__global__ void __launch_bounds__(256)
mx_quantize_kernel(const __nv_bfloat16 *__restrict__ in, int64_t rows, int64_t cols, int64_t sf_rows,
                   uint8_t *__restrict__ codes, uint8_t *__restrict__ scales) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t kbs = cols / 128;
    const int64_t steps = (rows + 7) / 8 * kbs;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); w < steps; w += warps) {
        const int64_t grp = w / kbs, kb = w - grp * kbs;
        const int64_t r = grp * 8 + (lane >> 2);
        const int64_t c = kb * 4 + (lane & 3);
        if (r < rows) {
            const uint32_t sc = quantize_block32(in + r * cols + c * 32, codes + r * cols + c * 32);
            scales[kmajor_scale_byte(r, c, sf_rows)] = static_cast<uint8_t>(sc);
        }
    }
}

// The dispatch of the MXFP8 path, fused into the quantization of x: routed
// row r (r < *routed) is token perm_slot[r] / k, quantized into row r of
// codes [R, cols] and of the k-block-major scales over sf_rows rows (R rounded
// up to 4), so stage 1 reads its A tiles and scale words with plain TMA copies.
__global__ void __launch_bounds__(256)
mx_quantize_dispatch_kernel(const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ perm_slot,
                            const int32_t *__restrict__ routed, int k, int64_t sf_rows, int64_t cols,
                            uint8_t *__restrict__ codes, uint8_t *__restrict__ scales) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t rows = *routed;
    const int64_t kbs = cols / 128;
    const int64_t steps = (rows + 7) / 8 * kbs;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); w < steps; w += warps) {
        const int64_t grp = w / kbs, kb = w - grp * kbs;
        const int64_t r = grp * 8 + (lane >> 2);
        const int64_t c = kb * 4 + (lane & 3);
        if (r < rows) {
            const int64_t t = perm_slot[r] / k;
            const uint32_t sc = quantize_block32(x + t * cols + c * 32, codes + r * cols + c * 32);
            scales[kmajor_scale_byte(r, c, sf_rows)] = static_cast<uint8_t>(sc);
        }
    }
}

// Row offsets of the MXFP8 weight-gradient operands: expert e's rows start at
// kpad[e], a multiple of 128 (one k-block of the block-scaled MMA), so each
// expert's reduction covers whole k-blocks; kpad[e+1] - kpad[e] =
// ceil(counts[e] / 128) * 128. One warp: a running sum over the experts in
// chunks of 32.
__global__ void __launch_bounds__(32) mx_wgrad_offsets_kernel(const int32_t *__restrict__ counts, int E,
                                                              int32_t *__restrict__ kpad) {
    griddep_wait();
    const int lane = threadIdx.x;
    int base = 0;
    if (lane == 0) kpad[0] = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
        const int e = e0 + lane;
        int v = (e < E) ? (counts[e] + 127) / 128 * 128 : 0;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int o = __shfl_up_sync(0xffffffffu, v, d);
            if (lane >= d) v += o;
        }
        if (e < E) kpad[e + 1] = base + v;
        base += __shfl_sync(0xffffffffu, v, 31);
    }
}

// The operands of an MXFP8 weight gradient, quantized along the expert's routed
// rows (the GEMM's reduction dimension) and stored transposed, K-major: codes
// [C, ld], where column r of expert e's segment [kpad[e], kpad[e+1]) holds
// routed row offsets[e] + (r - kpad[e]) of the source (zero past the expert's
// count), and the scales k-block-major: word [kb][c] holds the four E8M0 codes
// of rows [128 kb, 128 kb + 128) of column c, 32 rows each, so the GEMM's
// scale-factor warps read 32 consecutive columns' words as one 128-byte line.
// Source row of routed row q: src[q, :] (row stride src_ld), or with perm_slot
// the token's row src[perm_slot[q] / k, :]. One CTA per 128-row k-block and 128
// columns: the block's rows are staged in shared memory with 16-byte loads,
// then each thread quantizes one column's four 32-value blocks and writes its
// 128 codes as one 128-byte line and its four scales as one word.
constexpr int kQtCols = 128;
constexpr int kQtRows = 128;
__global__ void __launch_bounds__(kQtCols)
mx_quantize_rows_t_kernel(const __nv_bfloat16 *__restrict__ src, int64_t src_ld, const int32_t *__restrict__ perm_slot,
                          int k, const int32_t *__restrict__ counts, const int32_t *__restrict__ offsets,
                          const int32_t *__restrict__ kpad, int E, int C, int64_t ld, uint8_t *__restrict__ codes,
                          uint8_t *__restrict__ scales) {
    extern __shared__ __align__(16) uint32_t qt_tile[];   // [kQtRows][kQtCols / 2 + 4]
    constexpr int kStride = kQtCols / 2 + 4;             // words per staged row (16-byte aligned)
    griddep_wait();
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kQtRows;   // first padded row of the k-block
    if (r0 >= kpad[E]) return;                                         // past every expert's segment
    int lo = 0, hi = E;                                                // expert with kpad[e] <= r0 < kpad[e+1]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (kpad[mid] <= r0) lo = mid; else hi = mid;
    }
    const int e = lo;
    const int local = static_cast<int>(r0 - kpad[e]);                 // row of the expert's segment
    const int c0 = blockIdx.y * kQtCols;
    const int cnt = counts[e];
    for (int i = threadIdx.x; i < kQtRows * (kQtCols / 8); i += blockDim.x) {
        const int row = i / (kQtCols / 8);
        const int cc = (i % (kQtCols / 8)) * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (local + row < cnt && c0 + cc < C) {
            const int64_t q = offsets[e] + local + row;
            const int64_t srow = perm_slot ? perm_slot[q] / k : q;
            v = __ldg(reinterpret_cast<const uint4 *>(src + srow * src_ld + c0 + cc));
        }
        *reinterpret_cast<uint4 *>(qt_tile + row * kStride + cc / 2) = v;
    }
    __syncthreads();
    const int c = c0 + threadIdx.x;
    if (c >= C) return;
    uint32_t sw = 0;
    uint4 *dst = reinterpret_cast<uint4 *>(codes + static_cast<int64_t>(c) * ld + r0);
#pragma unroll 1
    for (int b = 0; b < kQtRows / 32; ++b) {
        float v[32];
#pragma unroll
        for (int row = 0; row < 32; ++row) {
            const uint32_t w = qt_tile[(32 * b + row) * kStride + threadIdx.x / 2];
            v[row] = (threadIdx.x & 1) ? bf16_hi(w) : bf16_lo(w);
        }
        uint32_t qw[8];
        sw |= mx_quantize32(v, qw) << (8 * b);
        dst[2 * b] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
        dst[2 * b + 1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
    }
    reinterpret_cast<uint32_t *>(scales)[(r0 / kQtRows) * C + c] = sw;
}

size_t qt_smem() { return sizeof(uint32_t) * kQtRows * (kQtCols / 2 + 4); }

}  // namespace

cudaError_t launch_mx_wgrad_offsets(const int32_t *counts, int E, int32_t *kpad, cudaStream_t st) {
    const cudaError_t e = launch_dep(mx_wgrad_offsets_kernel, dim3(1), dim3(32), 0, st, counts, E, kpad);
    note_launches(1);
    return e;
}

cudaError_t launch_mx_quantize_rows_t(const __nv_bfloat16 *src, int64_t src_ld, const int32_t *perm_slot, int k,
                                      const int32_t *counts, const int32_t *offsets, const int32_t *kpad, int E,
                                      int C, int64_t ld, uint8_t *codes, uint8_t *scales, cudaStream_t st) {
    if (ld <= 0 || C <= 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>(ld / kQtRows), static_cast<unsigned>((C + kQtCols - 1) / kQtCols));
    const cudaError_t e = launch_dep(mx_quantize_rows_t_kernel, grid, dim3(kQtCols), qt_smem(), st, src, src_ld,
                                     perm_slot, k, counts, offsets, kpad, E, C, ld, codes, scales);
    note_launches(1);
    return e;
}

cudaError_t launch_wgrad_mx(const GemmLaunch &p, cudaStream_t st) {
    GemmArgs g = grouped_args(p);
    g.total_units = g.E * g.m_tiles * g.n_tiles;
    const int grid = g.total_units < p.num_sms ? g.total_units : p.num_sms;
    if (grid <= 0) return cudaSuccess;
    return launch_tc_gemm<kWgradMx>(maps_of(p), g, grid, st);
}

cudaError_t launch_mx_quantize_dispatch(const __nv_bfloat16 *x, const int32_t *perm_slot, const int32_t *routed,
                                        int k, int64_t R, int64_t cols, uint8_t *codes, uint8_t *scales,
                                        cudaStream_t st) {
    const int64_t blocks = R * (cols / 32);
    if (blocks == 0) return cudaSuccess;
    int64_t grid = (blocks + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    const cudaError_t e = launch_dep(mx_quantize_dispatch_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, x,
                                     perm_slot, routed, k, static_cast<int64_t>(mx_rows(R)), cols, codes, scales);
    note_launches(1);
    return e;
}

cudaError_t setup_mx_gemm_kernels() {
    cudaError_t e = set_gemm_smem<kStage1Mx>();
    if (e == cudaSuccess) e = set_gemm_smem<kStage2Mx>();
    if (e == cudaSuccess) e = set_gemm_smem<kWgradMx>();
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(mx_quantize_rows_t_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(qt_smem()));
    return e;
}

cudaError_t launch_mx_quantize(const __nv_bfloat16 *in, int64_t rows, int64_t cols, uint8_t *codes,
                               uint8_t *scales, cudaStream_t st) {
    const int64_t blocks = rows * (cols / 32);
    if (blocks == 0) return cudaSuccess;
    int64_t grid = (blocks + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    const cudaError_t e = launch_dep(mx_quantize_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, in, rows,
                                     cols, static_cast<int64_t>(mx_rows(rows)), codes, scales);
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
