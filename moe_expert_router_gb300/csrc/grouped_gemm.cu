// grouped_gemm.cu -- the two expert-path grouped GEMMs of the MegaMoE layer on
// sm_103a, plus the final k-way combine.
//
//   stage 1, dispatch_grouped_gemm (MegaMoE guide, opening section; section
//   "Design: two stages", stage1 = dispatch + GEMM1): for each routed row r of
//   expert e, h = x[token(r)] . w1[e]^T and a[r] = silu(h[:I]) * h[I:]
//   (SwiGLU silu(x_glu) * x_linear, as in the "GDN <-> FLA Parity in Primus"
//   page, section B). The dispatch is a TMA row gather (tile::gather4) of x
//   driven by the routing permutation, so no permuted copy of x is made.
//
//   stage 2, grouped_gemm_combine (stage2 = GEMM2 + combine): o[r] = a[r] .
//   w2[e]^T; the epilogue scales o[r] by the routing weight of its slot and
//   scatters it to the slot's row of obuf (slot order t*k + j), and a light
//   reduction sums the k rows of every token into y.
//
// Kernel design (one CTA per SM, persistent over work units):
//   work unit  = (expert e, n-tile, 128-row tile of e's routed rows), ordered
//                expert-major, then n-tile, then row tile, so that CTAs running
//                side by side share a weight slab through L2;
//   warp 0     = TMA producer (x row gather / a tile, weight slabs) into a
//                4-stage ring of 128B-swizzled K-major tiles (BK = 64);
//   warp 1     = TMEM allocator and single-thread tcgen05.mma issuer
//                (M = 128, N = 256, K = 16 per instruction, fp32 accumulate);
//   warps 2-5  = epilogue: tcgen05.ld of the accumulator, fused SwiGLU or
//                weighted scatter, bf16 stores. Two TMEM accumulators (512
//                columns) let the epilogue of one unit overlap the next
//                unit's main loop.
// Row counts per expert are read from device memory, so any (ragged) routing
// runs without a host sync or re-launch. Rows of a tile past the expert's
// count are computed on stale or foreign data and never stored.
#include "internal.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int BM = kBM;          // 128 rows per tile (MMA M)
constexpr int BK = 64;           // 64 bf16 = one 128-byte swizzled row per stage
constexpr int BN = 256;          // accumulator columns per tile (MMA N)
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int ACC_STAGES = 2;
constexpr int TMEM_COLS = ACC_STAGES * BN;   // 512: the whole TMEM of the SM
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr uint64_t kDrainLimitNs = 10000000ull;  // 10 ms

struct __align__(1024) Smem {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full[ACC_STAGES];
    uint64_t acc_empty[ACC_STAGES];
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;  // + slack to align the base to 1024

struct GemmArgs {
    const int32_t *counts;
    const int32_t *offsets;
    const int32_t *mt_prefix;
    const int32_t *perm_slot;
    int32_t *err;
    const float *topk_w;
    __nv_bfloat16 *out;
    int E, k, K;
    int n_out;      // valid output columns (I or H)
    int n_tiles;    // n-tiles per expert
    int b_rows;     // weight rows per expert (2I or H)
    int half;       // stage 1: row offset of the up projection inside w1[e] (= I)
};

struct Unit {
    int e, n, row0, rows;
};

// Unit u -> (expert, n-tile, row tile). Units of expert e are
// [mt_prefix[e] * n_tiles, mt_prefix[e+1] * n_tiles), n-tile major.
__device__ __forceinline__ Unit decode_unit(int u, const GemmArgs &g) {
    int lo = 0, hi = g.E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (g.mt_prefix[mid] * g.n_tiles <= u) lo = mid; else hi = mid;
    }
    const int mt0 = g.mt_prefix[lo];
    const int mt_e = g.mt_prefix[lo + 1] - mt0;
    const int local = u - mt0 * g.n_tiles;
    Unit t;
    t.e = lo;
    t.n = local / mt_e;
    const int m = local - t.n * mt_e;
    t.row0 = g.offsets[lo] + m * BM;
    t.rows = min(BM, g.counts[lo] - m * BM);
    return t;
}

// Wait that ignores the abort flag and sets no error: used only to let
// in-flight copies or MMAs finish before an aborting CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kDrainLimitNs) return;
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + __expf(-g)) * u;
}

template <bool kSwiGLU>
__global__ void __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b, const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));
    volatile int *abort_flag = &sm.abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        for (int s = 0; s < ACC_STAGES; ++s) {
            mbar_init(smem_addr(&sm.acc_full[s]), 1);
            mbar_init(smem_addr(&sm.acc_empty[s]), EPI_THREADS);
        }
        mbar_init(smem_addr(&sm.drain), 1);
        sm.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sm.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;

    const int total = g.mt_prefix[g.E] * g.n_tiles;
    const int num_kb = (g.K + BK - 1) / BK;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        int stage = 0, issued = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
            const Unit t = decode_unit(u, g);
            const int brow = t.e * g.b_rows + t.n * (kSwiGLU ? BN / 2 : BN);
            int tok[4] = {0, 0, 0, 0};
            uint32_t a_bytes = A_BYTES;
            int n_gather = 0;
            if constexpr (kSwiGLU) {
                // rows 4*lane .. 4*lane+3 of the tile; rows past the count reuse row 0
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = lane * 4 + q;
                    tok[q] = g.perm_slot[t.row0 + (r < t.rows ? r : 0)] / g.k;
                }
                n_gather = (t.rows + 3) >> 2;
                a_bytes = static_cast<uint32_t>(n_gather) * 4u * BK * 2u;
            }
            for (int kb = 0; kb < num_kb; ++kb) {
                bool w_ok = true;
                if (lane == 0) w_ok = mbar_wait(smem_addr(&sm.empty[stage]), phase ^ 1u, abort_flag, g.err);
                w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
                if (!w_ok) { ok = false; break; }
                const uint32_t full = smem_addr(&sm.full[stage]);
                const uint32_t sa = smem_addr(sm.a[stage]);
                const uint32_t sb = smem_addr(sm.b[stage]);
                const int kx = kb * BK;
                if (lane == 0) mbar_arrive_expect_tx(full, a_bytes + B_BYTES);
                __syncwarp();
                if constexpr (kSwiGLU) {
                    if (lane < n_gather)
                        tma_gather4(sa + lane * 4 * (BK * 2), &tm_a, kx, tok[0], tok[1], tok[2], tok[3], full);
                    if (lane == 0) {
                        tma_load_2d(sb, &tm_b, kx, brow, full);                       // gate rows
                        tma_load_2d(sb + B_BYTES / 2, &tm_b, kx, brow + g.half, full);  // up rows
                    }
                } else {
                    if (lane == 0) {
                        tma_load_2d(sa, &tm_a, kx, t.row0, full);
                        tma_load_2d(sb, &tm_b, kx, brow, full);
                    }
                }
                __syncwarp();
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok && lane == 0) {
            // let the copies already issued land before the CTA exits
            int s = stage;
            uint32_t ph = phase;
            for (int i = 0; i < min(issued, STAGES); ++i) {
                if (--s < 0) { s = STAGES - 1; ph ^= 1u; }
                drain_wait(smem_addr(&sm.full[s]), ph);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true, any = false;
            for (int u = blockIdx.x; u < total && ok; u += gridDim.x) {
                if (!mbar_wait(smem_addr(&sm.acc_empty[acc]), acc_phase ^ 1u, abort_flag, g.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_addr(&sm.full[stage]), phase, abort_flag, g.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(sm.a[stage]);
                    const uint32_t sb = smem_addr(sm.b[stage]);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        mma_bf16(d_tmem, smem_desc_sw128(sa + kk * UMMA_K * 2),
                                 smem_desc_sw128(sb + kk * UMMA_K * 2), IDESC, (kb | kk) != 0);
                    }
                    mma_commit(smem_addr(&sm.empty[stage]));   // frees the smem stage
                    any = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(smem_addr(&sm.acc_full[acc]));      // accumulator ready
                if (++acc == ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
            }
            if (!ok && any) {
                mma_commit(smem_addr(&sm.drain));
                drain_wait(smem_addr(&sm.drain), 0);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;              // TMEM lanes this warp may access
        const int row = quad * 32 + lane;       // tile row = TMEM lane
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit t = decode_unit(u, g);
            bool ok = true;
            if (lane == 0) ok = mbar_wait(smem_addr(&sm.acc_full[acc]), acc_phase, abort_flag, g.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                  static_cast<uint32_t>(acc * BN);
            const bool valid = row < t.rows;
            if constexpr (kSwiGLU) {
                const int col0 = t.n * (BN / 2);
                __nv_bfloat16 *dst =
                    g.out + static_cast<int64_t>(t.row0 + row) * g.n_out + col0;
#pragma unroll 1
                for (int c = 0; c < BN / 2; c += 32) {
                    uint32_t gv[32], uv[32];
                    tmem_ld32(tacc + c, gv);
                    tmem_ld32(tacc + BN / 2 + c, uv);
                    tmem_wait_ld();
                    tmem_reg_fence(gv);
                    tmem_reg_fence(uv);
                    if (valid) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float a0 = silu_mul(__uint_as_float(gv[2 * i]), __uint_as_float(uv[2 * i]));
                            const float a1 = silu_mul(__uint_as_float(gv[2 * i + 1]),
                                                      __uint_as_float(uv[2 * i + 1]));
                            pk[i] = pack_bf16x2(a0, a1);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (col0 + c + j * 8 < g.n_out)
                                *reinterpret_cast<uint4 *>(dst + c + j * 8) =
                                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        }
                    }
                }
            } else {
                const int col0 = t.n * BN;
                int slot = 0;
                float w = 0.0f;
                if (valid) {
                    slot = g.perm_slot[t.row0 + row];
                    w = g.topk_w[slot];
                }
                __nv_bfloat16 *dst = g.out + static_cast<int64_t>(slot) * g.n_out + col0;
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t v[32];
                    tmem_ld32(tacc + c, v);
                    tmem_wait_ld();
                    tmem_reg_fence(v);
                    if (valid) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(w * __uint_as_float(v[2 * i]), w * __uint_as_float(v[2 * i + 1]));
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (col0 + c + j * 8 < g.n_out)
                                *reinterpret_cast<uint4 *>(dst + c + j * 8) =
                                    make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&sm.acc_empty[acc]));
            if (++acc == ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// y[t, :] = sum over the token's k slots of obuf[slot, :] (already weighted);
// dropped slots (row_of < 0) are skipped. fp32 sum, bf16 result.
__global__ void __launch_bounds__(256)
combine_kernel(const __nv_bfloat16 *__restrict__ obuf, const int32_t *__restrict__ row_of,
               __nv_bfloat16 *__restrict__ y, int T, int H, int k) {
    const int groups = H >> 3;
    const int64_t total = static_cast<int64_t>(T) * groups;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(i / groups);
        const int c = static_cast<int>(i - static_cast<int64_t>(t) * groups) * 8;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const int64_t s = static_cast<int64_t>(t) * k + j;
            if (row_of[s] < 0) continue;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(obuf + s * H + c));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[2 * q] += __uint_as_float(w[q] << 16);
                acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
            }
        }
        *reinterpret_cast<uint4 *>(y + static_cast<int64_t>(t) * H + c) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                       pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    }
}

GemmArgs make_args(const GemmLaunch &p, int n_tiles) {
    GemmArgs g;
    g.counts = p.counts;
    g.offsets = p.offsets;
    g.mt_prefix = p.mt_prefix;
    g.perm_slot = p.perm_slot;
    g.err = p.err;
    g.topk_w = p.topk_w;
    g.out = p.out;
    g.E = p.E;
    g.k = p.k;
    g.K = p.K;
    g.n_out = p.n_out;
    g.n_tiles = n_tiles;
    g.b_rows = p.b_rows;
    g.half = p.half;
    return g;
}

}  // namespace

cudaError_t setup_gemm_kernels() {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(grouped_gemm_kernel<false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SMEM_BYTES));
}

cudaError_t launch_gemm1_swiglu(const GemmLaunch &p, cudaStream_t st) {
    const GemmArgs g = make_args(p, (p.n_out + BN / 2 - 1) / (BN / 2));
    grouped_gemm_kernel<true><<<p.num_sms, NUM_THREADS, SMEM_BYTES, st>>>(*p.tm_a, *p.tm_b, g);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_gemm2_scatter(const GemmLaunch &p, cudaStream_t st) {
    const GemmArgs g = make_args(p, (p.n_out + BN - 1) / BN);
    grouped_gemm_kernel<false><<<p.num_sms, NUM_THREADS, SMEM_BYTES, st>>>(*p.tm_a, *p.tm_b, g);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_combine(const CombineLaunch &p, cudaStream_t st) {
    const int64_t total = static_cast<int64_t>(p.T) * (p.H / 8);
    if (total == 0) return cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    combine_kernel<<<static_cast<int>(blocks), 256, 0, st>>>(p.obuf, p.row_of, p.y, p.T, p.H, p.k);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
