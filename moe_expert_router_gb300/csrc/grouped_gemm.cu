// grouped_gemm.cu -- the tensor-core GEMMs of the MegaMoE expert path on
// sm_103a, plus the final k-way combine.
//
//   stage 1, dispatch_grouped_gemm (MegaMoE guide, opening section; section
//   "Design: two stages", stage1 = dispatch + GEMM1): for each routed row r of
//   expert e, h = x[token(r)] . w1[e]^T and a[r] = silu(h[:I]) * h[I:]
//   (SwiGLU silu(x_glu) * x_linear, as in the "GDN <-> FLA Parity in Primus"
//   page, section B). The dispatch is fused: dedicated warps gather the
//   routed x rows straight into the shared-memory A tiles, driven by the
//   routing permutation, so no permuted copy of x is ever written.
//
//   stage 2, grouped_gemm_combine (stage2 = GEMM2 + combine): o[r] = a[r] .
//   w2[e]^T; the epilogue scales o[r] by the routing weight of its slot and
//   writes it to row r of obuf; the combine then gathers the k rows of every
//   token through row_of and sums them into y.
//
//   router GEMM (the fused router's score function, MegaMoE guide opening
//   section): partial fp32 logits of x . w_r^T with w_r split exactly into
//   three bf16 matrices hi + mid + lo (Henry, Tang and Heinecke 2019,
//   "Leveraging the bfloat16 artificial intelligence datatype for higher-
//   precision computations"); x is bf16, so every product is exact and the
//   fp32 accumulation matches an fp32 dot product. Split-K partials are
//   summed in a fixed order by the top-k kernel.
//
// Kernel design (one CTA per SM, persistent):
//   work unit  = (expert e, n-tile, 256-row tile of e's routed rows) for the
//                grouped stages, (256-row tile, n-tile, k split) for the
//                router. The 256 rows are two 128-row halves that share every
//                weight tile, which halves the weight bytes each SM loads per
//                flop against a 128-row tile; an empty second half is neither
//                loaded nor multiplied. Grouped units are numbered
//                expert-major, then n-tile, then row tile; CTAs take the next
//                unit from a global counter, so CTAs running side by side work
//                on neighbouring units and share each weight slab through L2.
//   warp 0     = scheduler + TMA producer: claims units, publishes them to an
//                in-CTA queue and fills a ring of swizzled K-major tiles (per
//                stage: two 128 x BK A halves and one 256 x BK B tile; six
//                32 KB stages at BK = 32, three 64 KB stages at BK = 64).
//   warp 1     = TMEM allocator and single-thread tcgen05.mma issuer: per
//                16-deep k-step one M=128 N=256 MMA per half into two fp32
//                TMEM accumulators (all 512 columns).
//   warps 2-9  = epilogue, one TMEM lane quadrant of one half each:
//                tcgen05.ld, then fused SwiGLU, weighted scatter or fp32 store.
// Row counts are read from device memory, so ragged routing never needs a
// host sync or a re-launch. Rows of a tile past the expert's count are
// computed on stale or foreign data and never stored.
#include "internal.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int BM = kBM;                      // rows per MMA / per accumulator
constexpr int UM = kUnitM;                   // rows per work unit (two halves)
constexpr int BK = kBK;
constexpr int BN = kBN;
constexpr int UMMA_K = 16;
constexpr int ROW_BYTES = BK * 2;            // bytes of one K-major tile row per stage
constexpr int STAGES = (BK == 64) ? 3 : 6;
constexpr int A_HALF_BYTES = BM * BK * 2;    // 16 KB (BK 64) or 8 KB (BK 32)
constexpr int A_BYTES = 2 * A_HALF_BYTES;    // 32 KB
constexpr int B_BYTES = BN * BK * 2;         // 32 KB or 16 KB
constexpr int TMEM_COLS = 2 * BN;            // two accumulators: all 512 columns
constexpr int EPI_WARPS = 8;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int GATHER_WARPS = 4;              // stage 1: x row gather into the A tiles
constexpr int GATHER_THREADS = GATHER_WARPS * 32;
constexpr int UQ = 4;                        // depth of the in-CTA unit queue
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
constexpr uint64_t kDrainLimitNs = 10000000ull;  // 10 ms

enum Mode : int { kStage1 = 0, kStage2 = 1, kRouter = 2 };

// warps: 0 scheduler + TMA producer, 1 MMA issuer, 2..9 epilogue, and in
// stage 1 also 10..13 gathering the routed x rows
template <int MODE>
constexpr int kNumThreads = 64 + EPI_THREADS + (MODE == kStage1 ? GATHER_THREADS : 0);

struct __align__(1024) Smem {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    uint8_t stage_out[EPI_WARPS][32 * 128];  // per epilogue warp: a 32 x 64 bf16 output box
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t uq_full[UQ];
    uint64_t uq_empty[UQ];
    uint64_t drain;
    int unit_q[UQ];
    uint32_t tmem_base;
    int abort;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;  // + slack to align the base to 1024

struct GemmArgs {
    const int32_t *counts;
    const int32_t *offsets;
    const int32_t *mt_prefix;
    const int32_t *perm_slot;
    const __nv_bfloat16 *x;  // stage 1: token rows [T, K]
    int32_t *err;
    int32_t *sched;          // [0] next unit, [1] CTAs finished
    const float *topk_w;
    __nv_bfloat16 *out;
    float *logits_part;      // router
    int E, k, K;
    int n_out;               // valid output columns (I, H or E)
    int n_tiles;             // n-tiles per expert (grouped) or per row tile (router)
    int b_rows;              // weight rows per expert (2I or H)
    int half;                // stage 1: row offset of the up projection inside w1[e] (= I)
    int T, splits, kb_per_split, kb_total, kb_h;   // router
    int total_units;         // router: known on the host; grouped: -1 (read from the device)
};

struct Unit {
    int e, n, row0, rows, kb0, kb1, split;
};

template <int MODE>
__device__ __forceinline__ Unit decode_unit(int u, const GemmArgs &g) {
    Unit t;
    if constexpr (MODE == kRouter) {
        const int per_m = g.n_tiles * g.splits;
        const int m = u / per_m;
        const int rem = u - m * per_m;
        t.n = rem / g.splits;
        t.split = rem - t.n * g.splits;
        t.e = 0;
        t.row0 = m * UM;
        t.rows = min(UM, g.T - t.row0);
        t.kb0 = t.split * g.kb_per_split;
        t.kb1 = min(g.kb_total, t.kb0 + g.kb_per_split);
    } else {
        // units of expert e are [mt_prefix[e] * n_tiles, mt_prefix[e+1] * n_tiles)
        int lo = 0, hi = g.E;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (g.mt_prefix[mid] * g.n_tiles <= u) lo = mid; else hi = mid;
        }
        const int mt0 = g.mt_prefix[lo];
        const int mt_e = g.mt_prefix[lo + 1] - mt0;
        const int local = u - mt0 * g.n_tiles;
        t.e = lo;
        t.n = local / mt_e;
        const int m = local - t.n * mt_e;
        t.row0 = g.offsets[lo] + m * UM;
        t.rows = min(UM, g.counts[lo] - m * UM);
        t.kb0 = 0;
        t.kb1 = (g.K + BK - 1) / BK;
        t.split = 0;
    }
    return t;
}

// Weight (B operand) coordinates of k-block kb: inner coordinate and first row.
template <int MODE>
__device__ __forceinline__ void b_coords(const GemmArgs &g, const Unit &t, int kb, int &kx, int &row) {
    if constexpr (MODE == kRouter) {
        const int seg = kb / g.kb_h;              // 0: hi, 1: mid, 2: lo
        kx = (kb - seg * g.kb_h) * BK;
        row = seg * g.E + t.n * BN;
    } else if constexpr (MODE == kStage1) {
        kx = kb * BK;
        row = t.e * g.b_rows + t.n * (BN / 2);
    } else {
        kx = kb * BK;
        row = t.e * g.b_rows + t.n * BN;
    }
}

// Wait that ignores the abort flag and sets no error: used only to let
// in-flight copies or MMAs finish before an aborting CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kDrainLimitNs) return;
    }
}

// silu(g) * u with the fast exponential and division intrinsics (a few
// instructions instead of an IEEE division); their error (a few ulp of fp32)
// is far below the bf16 rounding of the result. For g < -88 the quotient
// flushes to 0, which is the bf16 value of silu there anyway.
__device__ __forceinline__ float silu_mul(float g, float u) {
    return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// 32 output columns of this thread's row, packed to bf16: stage 1 applies the
// SwiGLU to accumulator columns [c, c+32) (gate) and [BN/2 + c, ...) (up),
// stage 2 scales accumulator columns [c, c+32) by the row's routing weight.
template <int MODE>
__device__ __forceinline__ void epilogue_piece(uint32_t tacc, int c, float w, uint32_t (&pk)[16]) {
    if constexpr (MODE == kStage1) {
        uint32_t gv[32], uv[32];
        tmem_ld32(tacc + c, gv);
        tmem_ld32(tacc + BN / 2 + c, uv);
        tmem_wait_ld();
        tmem_reg_fence(gv);
        tmem_reg_fence(uv);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(silu_mul(__uint_as_float(gv[2 * i]), __uint_as_float(uv[2 * i])),
                                silu_mul(__uint_as_float(gv[2 * i + 1]), __uint_as_float(uv[2 * i + 1])));
    } else {
        uint32_t v[32];
        tmem_ld32(tacc + c, v);
        tmem_wait_ld();
        tmem_reg_fence(v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(w * __uint_as_float(v[2 * i]), w * __uint_as_float(v[2 * i + 1]));
    }
}

template <int MODE>
__global__ void __launch_bounds__(kNumThreads<MODE>, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_out, const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));
    volatile int *abort_flag = &sm.abort;
    volatile int *unit_q = sm.unit_q;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            // stage 1: the producer's expect_tx arrival plus one per gather thread
            mbar_init(smem_addr(&sm.full[s]), MODE == kStage1 ? 1 + GATHER_THREADS : 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        mbar_init(smem_addr(&sm.acc_full), 1);
        mbar_init(smem_addr(&sm.acc_empty), EPI_THREADS);
        for (int s = 0; s < UQ; ++s) {
            mbar_init(smem_addr(&sm.uq_full[s]), 1);
            mbar_init(smem_addr(&sm.uq_empty[s]), 1 + EPI_WARPS + (MODE == kStage1 ? GATHER_WARPS : 0));
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

    if (warp == 0) {
        // ------------------------------------------------ scheduler + TMA producer
        const int total = (MODE == kRouter) ? g.total_units : g.mt_prefix[g.E] * g.n_tiles;
        int stage = 0, issued = 0, q = 0;
        uint32_t phase = 0, qphase = 0;
        bool ok = true;
        while (true) {
            int u = 0;
            if (lane == 0) u = atomicAdd(&g.sched[0], 1);
            u = __shfl_sync(0xffffffffu, u, 0);
            const bool more = u < total;
            bool w_ok = true;
            if (lane == 0) {
                w_ok = mbar_wait(smem_addr(&sm.uq_empty[q]), qphase ^ 1u, abort_flag, g.err);
                if (w_ok) {
                    unit_q[q] = more ? u : -1;
                    mbar_arrive(smem_addr(&sm.uq_full[q]));
                }
            }
            w_ok = __shfl_sync(0xffffffffu, w_ok, 0);
            if (!w_ok) { ok = false; break; }
            if (++q == UQ) { q = 0; qphase ^= 1u; }
            if (!more) break;

            const Unit t = decode_unit<MODE>(u, g);
            const bool two = t.rows > BM;            // second half present
            // stage 1: the A rows arrive through the gather warps, not TMA
            const uint32_t a_bytes = (MODE == kStage1) ? 0u : (two ? A_BYTES : A_HALF_BYTES);
            for (int kb = t.kb0; kb < t.kb1; ++kb) {
                bool e_ok = true;
                if (lane == 0) e_ok = mbar_wait(smem_addr(&sm.empty[stage]), phase ^ 1u, abort_flag, g.err);
                e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
                if (!e_ok) { ok = false; break; }
                const uint32_t full = smem_addr(&sm.full[stage]);
                const uint32_t sa = smem_addr(sm.a[stage]);
                const uint32_t sb = smem_addr(sm.b[stage]);
                int kx, brow;
                b_coords<MODE>(g, t, kb, kx, brow);
                if (lane == 0) mbar_arrive_expect_tx(full, a_bytes + B_BYTES);
                __syncwarp();
                if constexpr (MODE == kStage1) {
                    if (lane == 0) {
                        tma_load_2d(sb, &tm_b, kx, brow, full);                        // gate rows
                        tma_load_2d(sb + B_BYTES / 2, &tm_b, kx, brow + g.half, full);   // up rows
                    }
                } else {
                    if (lane == 0) {
                        tma_load_2d(sa, &tm_a, kx, t.row0, full);
                        if (two) tma_load_2d(sa + A_HALF_BYTES, &tm_a, kx, t.row0 + BM, full);
                        tma_load_2d(sb, &tm_b, kx, brow, full);
                    }
                }
                __syncwarp();
                ++issued;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
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
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, q = 0;
            uint32_t phase = 0, acc_phase = 0, qphase = 0;
            bool ok = true, any = false;
            while (true) {
                if (!mbar_wait(smem_addr(&sm.uq_full[q]), qphase, abort_flag, g.err)) { ok = false; break; }
                const int u = unit_q[q];
                mbar_arrive(smem_addr(&sm.uq_empty[q]));
                if (++q == UQ) { q = 0; qphase ^= 1u; }
                if (u < 0) break;
                const Unit t = decode_unit<MODE>(u, g);
                const bool two = t.rows > BM;
                // the epilogue must have drained both accumulators of the previous unit
                if (!mbar_wait(smem_addr(&sm.acc_empty), acc_phase ^ 1u, abort_flag, g.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    if (!mbar_wait(smem_addr(&sm.full[stage]), phase, abort_flag, g.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_addr(sm.a[stage]);
                    const uint32_t sb = smem_addr(sm.b[stage]);
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                        const uint32_t acc = (kb > t.kb0 || kk > 0) ? 1u : 0u;
                        const uint64_t bdesc = smem_desc_swizzled<ROW_BYTES>(sb + kk * UMMA_K * 2);
                        mma_bf16(tmem_base, smem_desc_swizzled<ROW_BYTES>(sa + kk * UMMA_K * 2), bdesc, IDESC, acc);
                        if (two)
                            mma_bf16(tmem_base + BN, smem_desc_swizzled<ROW_BYTES>(sa + A_HALF_BYTES + kk * UMMA_K * 2), bdesc,
                                     IDESC, acc);
                    }
                    mma_commit(smem_addr(&sm.empty[stage]));   // frees the smem stage
                    any = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit(smem_addr(&sm.acc_full));           // accumulators ready
                acc_phase ^= 1u;
            }
            if (!ok && any) {
                mma_commit(smem_addr(&sm.drain));
                drain_wait(smem_addr(&sm.drain), 0);
            }
        }
        __syncwarp();
    } else if (warp < 2 + EPI_WARPS) {
        // ------------------------------------------------ epilogue
        const int quad = warp & 3;                  // TMEM lanes this warp may access
        const int half = (warp - 2) >> 2;           // accumulator (row half) of this warp
        const int row = half * BM + quad * 32 + lane;   // unit row
        const uint32_t tacc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                              static_cast<uint32_t>(half * BN);
        int q = 0;
        uint32_t acc_phase = 0, qphase = 0;
        while (true) {
            bool ok = true;
            int u = -1;
            if (lane == 0) {
                ok = mbar_wait(smem_addr(&sm.uq_full[q]), qphase, abort_flag, g.err);
                if (ok) {
                    u = unit_q[q];
                    mbar_arrive(smem_addr(&sm.uq_empty[q]));
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            u = __shfl_sync(0xffffffffu, u, 0);
            if (++q == UQ) { q = 0; qphase ^= 1u; }
            if (!ok || u < 0) break;
            const Unit t = decode_unit<MODE>(u, g);
            const bool valid = row < t.rows;
            float w = 0.0f;                             // stage 2: routing weight of the row's slot
            if constexpr (MODE == kStage2) {
                if (valid) w = g.topk_w[g.perm_slot[t.row0 + row]];
            }
            if (lane == 0) ok = mbar_wait(smem_addr(&sm.acc_full), acc_phase, abort_flag, g.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            if (t.rows > half * BM) {                   // this half was computed
                if constexpr (MODE == kStage1 || MODE == kStage2) {
                    // output rows are the unit's routed rows t.row0 + row (a for stage 1,
                    // obuf for stage 2), columns [col0, col0 + ncols)
                    constexpr int ncols = (MODE == kStage1) ? BN / 2 : BN;
                    const int col0 = t.n * ncols;
                    const int slab0 = half * BM + quad * 32;      // first unit row of this warp
                    if (slab0 + 32 <= t.rows) {
                        // whole 32-row slab valid: stage 32 x 64 bf16 boxes in shared
                        // memory (128B-swizzled) and write each with one TMA store
                        const uint32_t buf = smem_addr(sm.stage_out[warp - 2]);
#pragma unroll 1
                        for (int cc = 0; cc < ncols; cc += 64) {
                            if (col0 + cc >= g.n_out) break;
                            if (lane == 0) bulk_wait_read<0>();   // previous box read out
                            __syncwarp();
#pragma unroll
                            for (int p = 0; p < 2; ++p) {
                                uint32_t pk[16];
                                epilogue_piece<MODE>(tacc, cc + 32 * p, w, pk);
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    const int c16 = p * 4 + j;
                                    st_shared_v4(buf + lane * 128 + ((c16 ^ (lane & 7)) << 4), pk[4 * j],
                                                 pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                                }
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&tm_out, buf, col0 + cc, t.row0 + slab0);
                                bulk_commit();
                            }
                        }
                    } else {
                        // partial slab (the expert's last rows): masked direct stores
                        __nv_bfloat16 *dst = g.out + static_cast<int64_t>(t.row0 + row) * g.n_out + col0;
#pragma unroll 1
                        for (int c = 0; c < ncols; c += 32) {
                            uint32_t pk[16];
                            epilogue_piece<MODE>(tacc, c, w, pk);
                            if (valid) {
#pragma unroll
                                for (int j = 0; j < 4; ++j) {
                                    if (col0 + c + j * 8 < g.n_out)
                                        *reinterpret_cast<uint4 *>(dst + c + j * 8) =
                                            make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                                }
                            }
                        }
                    }
                } else {
                    const int col0 = t.n * BN;
                    float *dst = g.logits_part +
                                 (static_cast<int64_t>(t.split) * g.T + t.row0 + row) * g.n_out + col0;
                    const bool vec = (g.n_out & 3) == 0;
#pragma unroll 1
                    for (int c = 0; c < BN; c += 32) {
                        uint32_t v[32];
                        tmem_ld32(tacc + c, v);
                        tmem_wait_ld();
                        tmem_reg_fence(v);
                        if (valid) {
                            if (vec) {
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    if (col0 + c + j * 4 < g.n_out)
                                        *reinterpret_cast<uint4 *>(dst + c + j * 4) =
                                            make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                                }
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j) {
                                    if (col0 + c + j < g.n_out) dst[c + j] = __uint_as_float(v[j]);
                                }
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_addr(&sm.acc_empty));
            acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait<0>();                  // every output box written
    } else {
        // ------------------------------------------------ stage 1: routed x row gather
        // The dispatch of dispatch_grouped_gemm: 128 threads copy the x rows of
        // the unit's routed tokens straight into the 128B-swizzled A tiles with
        // 16-byte cp.async (one thread per 16-byte chunk of a row slice).
        // Each thread waits for its own copies, orders them before the tensor
        // core's async-proxy reads, then arrives on the stage's full barrier,
        // one stage behind its issue so that two stages of copies are in flight.
        if constexpr (MODE == kStage1) {
            const int gt = threadIdx.x - (64 + EPI_THREADS);
            constexpr int CHUNKS = ROW_BYTES / 16;                 // per row slice
            constexpr int RSTEP = GATHER_THREADS / CHUNKS;         // rows per pass
            constexpr int NROWS = UM / RSTEP;                      // rows per thread
            const int chunk = gt % CHUNKS;
            const int rg = gt / CHUNKS;                            // rows rg + RSTEP i
            int stage = 0, q = 0, pending = -1;
            uint32_t phase = 0, qphase = 0;
            while (true) {
                bool ok = true;
                int u = -1;
                if (lane == 0) {
                    ok = mbar_wait(smem_addr(&sm.uq_full[q]), qphase, abort_flag, g.err);
                    if (ok) {
                        u = unit_q[q];
                        mbar_arrive(smem_addr(&sm.uq_empty[q]));
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                u = __shfl_sync(0xffffffffu, u, 0);
                if (++q == UQ) { q = 0; qphase ^= 1u; }
                if (!ok || u < 0) break;
                const Unit t = decode_unit<MODE>(u, g);
                int tok[NROWS];
#pragma unroll
                for (int i = 0; i < NROWS; ++i) {
                    const int r = rg + RSTEP * i;
                    tok[i] = (r < t.rows) ? g.perm_slot[t.row0 + r] / g.k : -1;
                }
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    bool e_ok = true;
                    if (lane == 0) e_ok = mbar_wait(smem_addr(&sm.empty[stage]), phase ^ 1u, abort_flag, g.err);
                    e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
                    if (!e_ok) { ok = false; break; }
                    const int col = kb * BK + chunk * 8;
                    const uint32_t nbytes = col < g.K ? 16u : 0u;   // zero-fill the K tail
                    const uint32_t sa = smem_addr(sm.a[stage]);
#pragma unroll
                    for (int i = 0; i < NROWS; ++i) {
                        if (tok[i] >= 0) {
                            const int r = rg + RSTEP * i;
                            const uint32_t dst = sa + (r >> 7) * A_HALF_BYTES +
                                                 swizzled_chunk<ROW_BYTES>(r & (BM - 1), chunk);
                            cp_async_16(dst, g.x + static_cast<int64_t>(tok[i]) * g.K + (nbytes ? col : 0), nbytes);
                        }
                    }
                    cp_async_commit();
                    if (pending >= 0) {
                        cp_async_wait<1>();
                        fence_proxy_async_smem();
                        mbar_arrive(smem_addr(&sm.full[pending]));
                    }
                    pending = stage;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (pending >= 0) {                       // signal the unit's last stage
                    cp_async_wait<0>();
                    fence_proxy_async_smem();
                    mbar_arrive(smem_addr(&sm.full[pending]));
                    pending = -1;
                }
                if (!ok) break;
            }
            cp_async_wait<0>();                           // no copy in flight at exit
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    if (threadIdx.x == 0) {
        // the last CTA to finish resets the unit counter for the next launch
        __threadfence();
        if (atomicAdd(&g.sched[1], 1) == static_cast<int>(gridDim.x) - 1) {
            atomicExch(&g.sched[0], 0);
            atomicExch(&g.sched[1], 0);
        }
    }
}

// y[t, :] = sum over the token's k slots s of obuf[row_of[s], :] (rows already
// weighted, in routed order); dropped slots (row_of < 0) are skipped. fp32 sum,
// bf16 result.
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
            const int r = row_of[s];
            if (r < 0) continue;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(obuf + static_cast<int64_t>(r) * H + c));
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

GemmArgs grouped_args(const GemmLaunch &p, int n_tiles) {
    GemmArgs g{};
    g.counts = p.counts;
    g.offsets = p.offsets;
    g.mt_prefix = p.mt_prefix;
    g.perm_slot = p.perm_slot;
    g.x = p.x;
    g.err = p.err;
    g.sched = p.sched;
    g.topk_w = p.topk_w;
    g.out = p.out;
    g.logits_part = nullptr;
    g.E = p.E;
    g.k = p.k;
    g.K = p.K;
    g.n_out = p.n_out;
    g.n_tiles = n_tiles;
    g.b_rows = p.b_rows;
    g.half = p.half;
    g.total_units = -1;
    return g;
}

}  // namespace

cudaError_t setup_gemm_kernels() {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<kStage1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(tc_gemm_kernel<kStage2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(SMEM_BYTES));
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(tc_gemm_kernel<kRouter>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SMEM_BYTES));
}

cudaError_t launch_gemm1_swiglu(const GemmLaunch &p, cudaStream_t st) {
    const GemmArgs g = grouped_args(p, (p.n_out + BN / 2 - 1) / (BN / 2));
    tc_gemm_kernel<kStage1><<<p.num_sms, kNumThreads<kStage1>, SMEM_BYTES, st>>>(*p.tm_a, *p.tm_b, *p.tm_out, g);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_gemm2_scatter(const GemmLaunch &p, cudaStream_t st) {
    const GemmArgs g = grouped_args(p, (p.n_out + BN - 1) / BN);
    tc_gemm_kernel<kStage2><<<p.num_sms, kNumThreads<kStage2>, SMEM_BYTES, st>>>(*p.tm_a, *p.tm_b, *p.tm_out, g);
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_router_gemm(const RouterGemmLaunch &p, cudaStream_t st) {
    GemmArgs g{};
    g.err = p.err;
    g.sched = p.sched;
    g.logits_part = p.logits_part;
    g.E = p.E;
    g.K = p.H;
    g.n_out = p.E;
    g.n_tiles = (p.E + BN - 1) / BN;
    g.T = p.T;
    g.kb_h = (p.H + BK - 1) / BK;
    g.kb_total = 3 * g.kb_h;
    g.splits = p.splits;
    g.kb_per_split = (g.kb_total + p.splits - 1) / p.splits;
    g.total_units = ((p.T + UM - 1) / UM) * g.n_tiles * p.splits;
    // every split must own at least one k-block: an empty split would leave its
    // accumulator unwritten
    if (p.splits < 1 || (p.splits - 1) * g.kb_per_split >= g.kb_total) return cudaErrorInvalidValue;
    const int grid = g.total_units < p.num_sms ? g.total_units : p.num_sms;
    tc_gemm_kernel<kRouter><<<grid, kNumThreads<kRouter>, SMEM_BYTES, st>>>(*p.tm_x, *p.tm_w3, *p.tm_w3, g);
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
