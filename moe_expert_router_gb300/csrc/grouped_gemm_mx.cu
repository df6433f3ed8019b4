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

// The dispatch of the MXFP8 path, fused into the quantization of x, token by
// token: each x row is read and quantized once and its codes are written to the
// token's k routed rows row_of[t k + j] of codes [R, cols] (slots without a row,
// -1, are skipped), so x streams from memory once however the rows are ordered.
// A warp takes one token and 1024 columns (lane l: block l of 32 columns, a
// 2 KB read and 1 KB of codes per routed row). Routed rows are scattered, so the
// scales go row-major into sc_rows ([R][cols / 32] bytes: each warp writes 32
// consecutive bytes per row) and mx_scales_kmajor_kernel moves them to the
// k-block-major words stage 1 loads.
__global__ void __launch_bounds__(256)
mx_quantize_tokens_kernel(const __nv_bfloat16 *__restrict__ x, const int32_t *__restrict__ row_of, int k,
                          int64_t T, int64_t cols, uint8_t *__restrict__ codes, uint8_t *__restrict__ sc_rows) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t chunks = (cols + 1023) / 1024;
    const int64_t steps = T * chunks;
    const int64_t blocks = cols / 32;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); w < steps; w += warps) {
        // w is the same on every lane: the whole warp runs each iteration
        const int64_t t = w / chunks;
        const int64_t blk = (w - t * chunks) * 32 + lane;
        const bool valid = blk < blocks;                                // lanes past the row's last block idle
        const int my_row = lane < k ? row_of[t * k + lane] : -1;        // k <= 32
        uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
        uint8_t sc = 0;
        if (valid) {
            float v[32];
            const uint4 *s4 = reinterpret_cast<const uint4 *>(x + t * cols + blk * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 u4 = __ldg(s4 + q);
                const uint32_t u[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    v[8 * q + 2 * j] = bf16_lo(u[j]);
                    v[8 * q + 2 * j + 1] = bf16_hi(u[j]);
                }
            }
            uint32_t qw[8];
            sc = static_cast<uint8_t>(mx_quantize32(v, qw));
            c0 = make_uint4(qw[0], qw[1], qw[2], qw[3]);
            c1 = make_uint4(qw[4], qw[5], qw[6], qw[7]);
        }
        for (int j = 0; j < k; ++j) {
            const int r = __shfl_sync(0xffffffffu, my_row, j);
            if (r < 0 || !valid) continue;
            uint4 *d4 = reinterpret_cast<uint4 *>(codes + static_cast<int64_t>(r) * cols + blk * 32);
            d4[0] = c0;
            d4[1] = c1;
            sc_rows[static_cast<int64_t>(r) * blocks + blk] = sc;
        }
    }
}

// Scale words from row-major [R][kbs] (sc_rows of the token-order dispatch, four
// bytes of one row and k-block per word) to k-block-major [kbs][sf_rows], rows
// [0, *routed): 32 x 32 words per CTA through shared memory.
__global__ void __launch_bounds__(256)
mx_scales_kmajor_kernel(const uint32_t *__restrict__ in, const int32_t *__restrict__ routed, int64_t kbs,
                        int64_t sf_rows, uint32_t *__restrict__ out) {
    __shared__ uint32_t tile[32][33];
    griddep_wait();
    const int64_t R = *routed;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int64_t kb0 = static_cast<int64_t>(blockIdx.y) * 32;
    if (r0 >= R) return;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
#pragma unroll
    for (int i = ty; i < 32; i += 8)
        if (r0 + i < R && kb0 + tx < kbs) tile[i][tx] = in[(r0 + i) * kbs + kb0 + tx];
    __syncthreads();
#pragma unroll
    for (int i = ty; i < 32; i += 8)
        if (r0 + tx < R && kb0 + i < kbs) out[(kb0 + i) * sf_rows + r0 + tx] = tile[tx][i];
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
// columns, in three phases:
//   1. the block's 128 x 128 bf16 values are copied into shared memory with
//      16-byte cp.async copies, all sixteen of a thread's in flight at once
//      (zero-filled past the expert's rows);
//   2. each thread quantizes one column's four 32-value blocks and keeps the
//      128 codes in registers;
//   3. the codes go back into the (now free) tile, one 144-byte row per column,
//      and each warp stores four columns' 128-byte lines, so every store
//      instruction writes whole lines.
constexpr int kQtCols = 128;
constexpr int kQtRows = 128;
constexpr int kQtStride = kQtCols / 2 + 4;        // words per staged input row (272 bytes)
constexpr int kQtCodeStride = (kQtRows + 16) / 4; // words per staged code row (144 bytes)

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__global__ void __launch_bounds__(kQtCols)
mx_quantize_rows_t_kernel(const __nv_bfloat16 *__restrict__ src, int64_t src_ld, const int32_t *__restrict__ perm_slot,
                          int k, const int32_t *__restrict__ counts, const int32_t *__restrict__ offsets,
                          const int32_t *__restrict__ kpad, int E, int C, int64_t ld, uint8_t *__restrict__ codes,
                          uint8_t *__restrict__ scales) {
    extern __shared__ __align__(16) uint32_t qt_tile[];   // [kQtRows][kQtStride], later [kQtCols][kQtCodeStride]
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
    const int64_t base = offsets[e] + local;
    const int tid = threadIdx.x;

    // phase 1: thread tid copies 8 columns (16 bytes) of rows tid / 16 + 8 m
    const int cc = (tid & 15) * 8;
    const bool col_ok = c0 + cc < C;                                   // C % 8 == 0: whole chunks
    int64_t srow[kQtRows / 8];
#pragma unroll
    for (int m = 0; m < kQtRows / 8; ++m) {
        const int row = (tid >> 4) + 8 * m;
        srow[m] = -1;
        if (col_ok && local + row < cnt) srow[m] = perm_slot ? perm_slot[base + row] / k : base + row;
    }
#pragma unroll
    for (int m = 0; m < kQtRows / 8; ++m) {
        const int row = (tid >> 4) + 8 * m;
        const bool ok = srow[m] >= 0;
        const __nv_bfloat16 *p = ok ? src + srow[m] * src_ld + c0 + cc : src;
        cp_async16_zfill(smem_addr(qt_tile + row * kQtStride + cc / 2), p, ok ? 16u : 0u);
    }
    cp_async_wait_all();
    __syncthreads();

    // phase 2: column c0 + tid, four 32-row blocks
    uint32_t qw[kQtRows / 32][8];
    uint32_t sw = 0;
#pragma unroll
    for (int b = 0; b < kQtRows / 32; ++b) {
        float v[32];
#pragma unroll
        for (int row = 0; row < 32; ++row) {
            const uint32_t w = qt_tile[(32 * b + row) * kQtStride + tid / 2];
            v[row] = (tid & 1) ? bf16_hi(w) : bf16_lo(w);
        }
        sw |= mx_quantize32(v, qw[b]) << (8 * b);
    }
    __syncthreads();                                                   // the input tile is read

    // phase 3: codes through shared memory, whole 128-byte lines out
    uint32_t *crow = qt_tile + tid * kQtCodeStride;
#pragma unroll
    for (int b = 0; b < kQtRows / 32; ++b) {
        reinterpret_cast<uint4 *>(crow)[2 * b] = make_uint4(qw[b][0], qw[b][1], qw[b][2], qw[b][3]);
        reinterpret_cast<uint4 *>(crow)[2 * b + 1] = make_uint4(qw[b][4], qw[b][5], qw[b][6], qw[b][7]);
    }
    __syncthreads();
    const int part = tid & 7;
#pragma unroll
    for (int m = 0; m < kQtCols / 16; ++m) {
        const int col = (tid >> 3) + 16 * m;
        if (c0 + col < C) {
            const uint4 v = reinterpret_cast<const uint4 *>(qt_tile + col * kQtCodeStride)[part];
            reinterpret_cast<uint4 *>(codes + static_cast<int64_t>(c0 + col) * ld + r0)[part] = v;
        }
    }
    if (c0 + tid < C) reinterpret_cast<uint32_t *>(scales)[(r0 / kQtRows) * C + c0 + tid] = sw;
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

cudaError_t launch_mx_quantize_dispatch(const __nv_bfloat16 *x, const int32_t *row_of, const int32_t *routed, int k,
                                        int64_t T, int64_t cols, uint8_t *codes, uint8_t *scales, uint8_t *sc_tmp,
                                        cudaStream_t st) {
    const int64_t steps = T * ((cols + 1023) / 1024);
    if (steps == 0) return cudaSuccess;
    int64_t grid = (steps + 7) / 8;
    if (grid > 152 * 8) grid = 152 * 8;
    cudaError_t e = launch_dep(mx_quantize_tokens_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, x, row_of,
                               k, T, cols, codes, sc_tmp);
    note_launches(1);
    if (e != cudaSuccess) return e;
    const int64_t R = T * k, kbs = cols / 128;
    const dim3 tgrid(static_cast<unsigned>((R + 31) / 32), static_cast<unsigned>((kbs + 31) / 32));
    e = launch_dep(mx_scales_kmajor_kernel, tgrid, dim3(256), 0, st, reinterpret_cast<const uint32_t *>(sc_tmp),
                   routed, kbs, static_cast<int64_t>(mx_rows(R)), reinterpret_cast<uint32_t *>(scales));
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
