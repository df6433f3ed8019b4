// gemm_kernel.cuh -- the persistent tcgen05 grouped-GEMM kernel template of the
// MegaMoE expert path on sm_103a, shared by the forward (grouped_gemm.cu) and
// the backward (grouped_gemm_bwd.cu) translation units.
//
// Forward modes (MegaMoE guide, opening section; section "Design: two stages"):
//   kStage1  dispatch_grouped_gemm: for routed row r of expert e,
//            h = x[token(r)] . w1[e]^T, a[r] = silu(h[:I]) * h[I:] (SwiGLU
//            silu(x_glu) * x_linear, "GDN <-> FLA Parity in Primus" page,
//            section B). The routed x rows were dispatched into routed order
//            beforehand (a copy kernel; the MXFP8 quantization in kStage1Mx), so
//            the A tiles are plain TMA loads. kStage1SaveH also stores h (gate
//            and up halves, bf16) for the backward.
//   kStage2  grouped_gemm_combine: o[r] = a[r] . w2[e]^T, scaled by the slot's
//            routing weight and stored to row r of obuf (combined afterwards).
//   kRouter  partial fp32 logits of x . w_r^T with w_r split exactly into three
//            bf16 matrices (Henry, Tang and Heinecke 2019, "Leveraging the
//            bfloat16 artificial intelligence datatype for higher-precision
//            computations"); split-K partials are summed in a fixed order later.
//
// Backward modes (the guide's stage order: stage 2's backward yields dW2, then
// stage 1's yields dW1; everything else is the chain rule of the forward):
//   kBwdDA   dA_u[r] = dY[token(r)] . w2[e] (dY rows dispatched into routed order
//            like x in stage 1, w2[e] read MN-major). The epilogue applies the SwiGLU backward with
//            the saved h: dA = w dA_u, dU = dA silu(g), dG = dA u silu'(g), and
//            stores dH = [dG | dU], the weighted activations w a (for dW2) and
//            per-tile partial sums of dA_u . a (the routing-weight gradient).
//   kBwdDX   dXr[r] = dH[r] . w1[e] (w1[e] read MN-major), unweighted rows in
//            routed order, summed per token afterwards.
//   kBwdDW2  dW2[e] = sum over e's rows of dY[token(r)]^T (w a)[r]: M = H,
//            N = I, K = the expert's rows; dispatched dY rows read MN-major.
//   kBwdDW1  dW1[e] = sum over e's rows of dH[r]^T x[token(r)]: M = 2I, N = H,
//            K = the expert's rows; dispatched x rows read MN-major.
//
// MXFP8 modes (the guide's section "Expert precision"): kStage1Mx and kStage2Mx
// run the two expert stages, kWgradMx the dW1 / dW2 weight gradients (operands
// transposed and quantized along the routed rows beforehand), as
// kind::mxf8f6f4.block_scale MMAs on E4M3 operands with E8M0 scales per 32
// K-elements. The scales are k-block-major 32-bit words; each stage's words
// arrive by TMA on a barrier of their own and the helper warps copy them into
// tensor memory.
//
// Kernel design (one CTA per SM, persistent):
//   work unit  = (expert e, n-tile, 256-row tile of e's routed rows) for the
//                row-grouped modes, (256-row tile, n-tile, k split) for the
//                router, (expert e, 256-row m-tile, n-tile) for the weight
//                gradients. The 256 rows are two 128-row halves that share every
//                B tile; an empty second half is neither loaded nor multiplied.
//                Units are numbered expert-major, so CTAs running side by side
//                share each expert's operands through L2; CTAs take the next
//                unit from a global counter.
//   warp 0     = scheduler + TMA producer: claims units, publishes them to an
//                in-CTA queue and fills a ring of swizzled tiles (per stage two
//                128-row A halves and one 256-row B tile).
//   warp 1     = TMEM allocator and single-thread tcgen05.mma issuer: per
//                16-deep k-step one M=128 N=256 MMA per half into two fp32
//                TMEM accumulators (all 512 columns).
//   warps 2-9  = epilogue, one TMEM lane quadrant of one half each.
//   warps 10-13 (weight gradients) = zero the K rows past the expert's count in
//                the last k-block; (MXFP8) = the scale factors of every stage.
// Operands are K-major (rows of K contiguous, 128- or 64-byte swizzle) or
// MN-major (K rows of 64-element, 128-byte swizzled MN atoms; the atoms of one
// tile are BK * 128 bytes apart, 8-row K groups 1024 bytes apart).
// Row counts are read from device memory, so ragged routing never needs a
// host sync or a re-launch.
#pragma once

#include "internal.cuh"
#include "mx.cuh"
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
constexpr int MN_ATOM_BYTES = BK * 128;      // one 64-wide MN atom over the stage's BK rows
constexpr int TMEM_COLS = 2 * BN;            // two accumulators: all 512 columns
constexpr int EPI_WARPS = 8;
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int HELPER_WARPS = 4;
constexpr int HELPER_THREADS = HELPER_WARPS * 32;
constexpr int UQ = 4;                        // depth of the in-CTA unit queue
constexpr uint64_t kDrainLimitNs = 10000000ull;  // 10 ms
// Stages 1 and 2 hold their stages in a byte ring over the A and B arrays (192 KB)
// with slots sized to the unit: 64 KB for a 256-row unit, 48 KB for a 128-row
// one. A k-block's refill only starts once its slot has been consumed, so the
// number of slots in flight sets how much load latency is covered: a 256-row
// unit's three slots keep the tensor pipe fed, a 128-row unit gets four. At
// most kRingSlots slots are in flight.
constexpr int kRingSlots = 6;
constexpr uint32_t kRingBytes = 3u * 64u * 1024u;

enum Mode : int {
    kStage1 = 0, kStage2 = 1, kRouter = 2,
    kBwdDA = 3, kBwdDX = 4, kBwdDW2 = 5, kBwdDW1 = 6,
    kStage1SaveH = 7,           // stage 1 that also stores h for the backward
    kStage1Mx = 8,              // stage 1 in MXFP8: E4M3 x and w1, a quantized in the epilogue
    kStage2Mx = 9,              // stage 2 in MXFP8: E4M3 a and w2
    kWgradMx = 10               // MXFP8 weight gradient: operands quantized along the expert's routed rows
};

template <int MODE> constexpr bool kIsMx = MODE == kStage1Mx || MODE == kStage2Mx || MODE == kWgradMx;
template <int MODE> constexpr bool kIsStage1 = MODE == kStage1 || MODE == kStage1SaveH || MODE == kStage1Mx;
template <int MODE> constexpr bool kRing = MODE == kStage1 || MODE == kStage2;
template <int MODE> constexpr bool kAMn = MODE == kBwdDW2 || MODE == kBwdDW1;
template <int MODE> constexpr bool kBMn = MODE >= kBwdDA && MODE <= kBwdDW1;
template <int MODE> constexpr bool kWeightGrad = MODE == kBwdDW2 || MODE == kBwdDW1;
// units (expert, m-tile, n-tile) reducing over the expert's rows, written per expert
template <int MODE> constexpr bool kPerExpertOut = kWeightGrad<MODE> || MODE == kWgradMx;
// warps 10..13: the reduction-tail zeroing of the weight gradients, and in the
// MXFP8 modes the scale factors
template <int MODE> constexpr bool kHelpers = kWeightGrad<MODE> || kIsMx<MODE>;
// accumulator columns of one 128-row half (a unit's output columns): 2 x 96
// (gate, up) in stage 1 MXFP8, 224 in stage 2 MXFP8, else 256; the MXFP8 modes
// keep the rest of tensor memory for per-stage scale factors
template <int MODE> constexpr int kUnitN = MODE == kStage1Mx ? 192 : ((MODE == kStage2Mx || MODE == kWgradMx) ? 224 : BN);
// K elements per pipeline stage (128-byte rows either way)
template <int MODE> constexpr int kStageK = kIsMx<MODE> ? 128 : BK;
template <int MODE> constexpr int kElemBytes = kIsMx<MODE> ? 1 : 2;
// scale factors of stage s: columns kSfBase + 16 s + [0, 4) A rows 0..127,
// [4, 8) A rows 128..255, [8, 8 + N/32) B rows
template <int MODE> constexpr int kSfBase = 2 * kUnitN<MODE>;
constexpr int kSfStride = 16;
static_assert(2 * 224 + STAGES * kSfStride <= 512, "MXFP8 scale factors must fit in tensor memory");
static_assert(BK == 64, "the MXFP8 modes share the 128-byte stage rows of BK = 64");
// MXFP8: each stage's scale words arrive by TMA with its operands, into the tail
// of the stage's B slot (past the widest MXFP8 B tile, 224 rows x 128 bytes).
// The scales are k-block-major 32-bit words (one per row and 128-deep k-block),
// so a stage needs one word per A row and per B row. An A box starts at the
// unit's first row rounded down to 4 words (a TMA copy starts on a 16-byte
// boundary) and holds 132 words, so it covers the 128 rows of one half.
constexpr uint32_t kSfSmemOff = 224 * 128;
constexpr int kSfBoxA = kSfBoxRowsA;         // words per A box (132)
constexpr uint32_t kSfA1 = 640;              // second half's A box (bytes from kSfSmemOff)
constexpr uint32_t kSfB0 = 1280;             // B words: stage 1 gate rows, else all rows
constexpr uint32_t kSfB1 = kSfB0 + 96 * 4;   // stage 1: up rows
static_assert(kSfA1 >= kSfBoxA * 4 && kSfB0 >= kSfA1 + kSfBoxA * 4, "MXFP8 scale boxes overlap");
static_assert(kSfSmemOff + kSfB0 + 224 * 4 <= static_cast<uint32_t>(B_BYTES), "MXFP8 scale words must fit the B slot");
// bytes of one stage's scale boxes
__host__ __device__ constexpr uint32_t sf_stage_bytes(int mode, bool two) {
    return (two ? 2u : 1u) * kSfBoxA * 4u + (mode == kStage1Mx ? 2u * 96u * 4u : 224u * 4u);
}

// warps: 0 scheduler + TMA producer, 1 MMA issuer, 2..9 epilogue, 10..13 helpers
template <int MODE>
constexpr int kNumThreads = 64 + EPI_THREADS + (kHelpers<MODE> ? HELPER_THREADS : 0);

template <int MODE>
constexpr uint32_t kIdesc = idesc_bf16_f32(BM, BN) | (kAMn<MODE> ? (1u << 15) : 0u) |
                            (kBMn<MODE> ? (1u << 16) : 0u);

struct __align__(1024) Smem {
    uint8_t a[STAGES][A_BYTES];
    uint8_t b[STAGES][B_BYTES];
    uint8_t stage_out[EPI_WARPS][32 * 128];  // per epilogue warp: one 32 x 64 or two 32 x 32 bf16 boxes
    uint64_t full[STAGES > kRingSlots ? STAGES : kRingSlots];   // stages, or ring slots (stages 1 / 2)
    uint64_t empty[STAGES > kRingSlots ? STAGES : kRingSlots];
    uint64_t sf_full[STAGES];                // MXFP8: the stage's scale words have landed (TMA)
    uint64_t sf_ready[STAGES];               // MXFP8: ... and are in tensor memory (one arrival per helper warp)
    uint64_t acc_full;
    uint64_t acc_empty;
    uint64_t uq_full[UQ];
    uint64_t uq_empty[UQ];
    uint64_t drain;
    uint64_t tail_ready;                     // weight gradients: the MMA issuer saw a partial k-block land
    uint64_t tail_fixed;                     // ... and the helpers zeroed its rows past the expert's count
    int unit_q[UQ];
    uint32_t tmem_base;
    int abort;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;  // + slack to align the base to 1024
static_assert(STAGES * (A_BYTES + B_BYTES) == kRingBytes && offsetof(Smem, b) == STAGES * A_BYTES,
              "the stage arrays must form one contiguous ring");

// Tensor maps of one launch (unused ones are copies of a used one).
struct GemmMaps {
    CUtensorMap a;     // A operand (TMA-loaded modes)
    CUtensorMap b;     // B operand
    CUtensorMap out;   // primary output
    CUtensorMap out2;  // kStage1SaveH: h gate half; dA: dH up half
    CUtensorMap out3;  // kStage1SaveH: h up half;   dA: w a
    CUtensorMap sfa;   // MXFP8: k-block-major scale words of the A rows (32-bit, [K / 128][rows])
    CUtensorMap sfb;   // MXFP8: ... of the B rows
};

struct GemmArgs {
    const int32_t *counts;
    const int32_t *offsets;
    const int32_t *mt_prefix;
    const int32_t *perm_slot;
    const __nv_bfloat16 *h;     // dA: saved pre-activation [R, 2I]
    int32_t *err;
    int32_t *sched;             // [0] next unit, [1] CTAs finished
    const float *topk_w;
    const int32_t *row_of;      // stage 2, fused combine: routed row of each slot (-1: dropped)
    __nv_bfloat16 *y;           // stage 2, fused combine: y [T, H]
    int32_t *ccnt;              // stage 2, fused combine: counters [T, n_tiles], or null (combine kernel)
    __nv_bfloat16 *out;         // masked direct stores of partial row slabs
    __nv_bfloat16 *out2, *out3; // kStage1SaveH: h gate / up halves; dA: dH up half, w a
    float *logits_part;         // router
    float *dtw_part;            // dA: [n_tiles, R] partial routing-weight gradients
    uint8_t *out_sf;            // stage 1 MXFP8: scales of a, k-block-major over sf_rows rows
    int64_t sf_rows;            // stage 1 MXFP8: rows of the scale arrays of x and a (T k rounded up to 4)
    int E, k, K;
    int n_out;                  // valid output columns
    int n_tiles;                // n-tiles per expert (grouped) or per row tile (router)
    int m_total, m_tiles;       // weight gradients: output rows per expert, 256-row tiles
    int b_rows;                 // weight rows per expert (stage 1: 2I)
    int half;                   // stage 1: row offset of the up projection (= I); dA: I
    int out_ld;                 // row stride (elements) of out / out2 / out3
    int R;                      // routed rows
    int T, splits, kb_per_split, kb_total;         // router
    int n_mma;                  // router: N of its MMAs and rows of its weight tile (E rounded up to 32, <= 256;
                                //   3 router_seg with the parts fused)
    int router_seg;             // router: accumulator columns of each of the hi / mid / lo parts when one
                                //   MMA covers all three (E <= 64), else 0
    const int32_t *kpad;        // MXFP8 weight gradients: [E+1] start of each expert's rows in the
                                //   quantized operands, a multiple of 128 (rows padded to whole k-blocks)
    const uint8_t *bpack;       // stage 1 / 2: the tile-packed weights (pack.cu), or null for the TMA views
    int kb_tiles;               // K tiles per packed weight slab
    int total_units;            // router / weight gradients: known on the host; else -1
};

struct Unit {
    int e, n, row0, rows, kb0, kb1, split;
    int koff, kcount;           // weight gradients: the expert's routed rows
};

template <int MODE>
__device__ __forceinline__ Unit decode_unit(int u, const GemmArgs &g) {
    Unit t;
    t.koff = 0;
    t.kcount = 0;
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
    } else if constexpr (MODE == kWgradMx) {
        // K runs over the expert's rows in the quantized operands: k-blocks of 128
        // rows from kpad[e] (a multiple of 128), rows past the count are zero codes
        const int per_e = g.m_tiles * g.n_tiles;
        t.e = u / per_e;
        const int rem = u - t.e * per_e;
        const int m = rem / g.n_tiles;
        t.n = rem - m * g.n_tiles;
        t.row0 = m * UM;
        t.rows = min(UM, g.m_total - t.row0);
        t.kcount = g.counts[t.e];
        t.kb0 = g.kpad[t.e] / kStageK<MODE>;
        t.kb1 = t.kb0 + (t.kcount + kStageK<MODE> - 1) / kStageK<MODE>;
        t.split = 0;
    } else if constexpr (kWeightGrad<MODE>) {
        const int per_e = g.m_tiles * g.n_tiles;
        t.e = u / per_e;
        const int rem = u - t.e * per_e;
        const int m = rem / g.n_tiles;
        t.n = rem - m * g.n_tiles;
        t.row0 = m * UM;
        t.rows = min(UM, g.m_total - t.row0);
        t.koff = g.offsets[t.e];
        t.kcount = g.counts[t.e];
        t.kb0 = 0;
        t.kb1 = (t.kcount + BK - 1) / BK;
        t.split = 0;
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
        t.kb1 = (g.K + kStageK<MODE> - 1) / kStageK<MODE>;
        t.split = 0;
    }
    return t;
}

// Descriptor of an MN-major bf16 operand: 64-element (128-byte) swizzled MN
// atoms MN_ATOM_BYTES apart (leading byte offset), 8-row K groups 1024 bytes
// apart (stride byte offset), version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(MN_ATOM_BYTES >> 4) << 16;
    d |= static_cast<uint64_t>(1024 >> 4) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

template <bool MN>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int kk) {
    if constexpr (MN) return smem_desc_mn(base + kk * UMMA_K * 128);
    else return smem_desc_swizzled<ROW_BYTES>(base + kk * UMMA_K * 2);
}

// Wait that ignores the abort flag and sets no error: used only to let
// in-flight copies or MMAs finish before an aborting CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kDrainLimitNs) return;
    }
}

// silu(g) * u for the SwiGLU epilogues of stage 1, through the identity
// silu(g) = g sigmoid(g) = h (1 + tanh(h)) with h = g / 2: one hardware tanh
// approximation (tanh.approx.f32) and two FMA-pipe operations per element,
// where 1 / (1 + exp(-g)) costs two special-function operations and more
// instructions -- the epilogue holds the accumulator while this runs (mid
// stage 1: 0.248 -> 0.243 ms). The approximation's error is a few times 1e-4
// of |h|, below the bf16 rounding of a; the GPU tests bound a's relative error
// against the fp64 oracle at 5e-3 (the general output bound is 1e-2).
__device__ __forceinline__ float sigmoid_tanh(float g) {
    // sigmoid(g) = (1 + tanh(g / 2)) / 2, for the SwiGLU backward of dA
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(0.5f * g));
    return fmaf(0.5f, t, 0.5f);
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    const float h = 0.5f * g;
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(h));
    return fmaf(h, t, h) * u;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Bytes of A a stage of unit t holds: two 128-row halves or one.
__device__ __forceinline__ uint32_t unit_a_bytes(const Unit &t) { return t.rows > BM ? A_BYTES : A_HALF_BYTES; }

// Write 16 packed words (32 bf16 of one row) into a 32 x 32 box staged with the
// 64-byte swizzle (what a TMA store of a 64-byte-wide box expects).
__device__ __forceinline__ void stage_row32(uint32_t buf, int lane, const uint32_t (&pk)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        st_shared_v4(buf + swizzled_chunk<64>(lane, j), pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
}

// Masked direct store of 32 bf16 columns of one row (partial row slabs).
__device__ __forceinline__ void store_row32(__nv_bfloat16 *dst, int cols_left, const uint32_t (&pk)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
        if (j * 8 < cols_left)
            *reinterpret_cast<uint4 *>(dst + j * 8) = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
}

// ---------------------------------------------------------------- fused combine (stage 2)

// The k-way sum of grouped_gemm_combine, fused into stage 2's epilogue. Each
// weighted expert row r (token t) is first stored to obuf; then the warp counts
// it in cnt[t, n] (n: the unit's 256-column tile), which the routing metadata
// set to the token's number of dropped slots. The lane whose row brings the
// counter to k owns the sum: the warp reads the token's k rows of that tile back
// (L2) and writes y[t, tile] = sum_j obuf[row_of[t k + j], tile] in fp32, in
// slot order, rounded to bf16 once -- the same arithmetic, in the same order,
// as combine_kernel, wherever and whenever the last row lands. It then resets
// the counter, so the metadata serve a later stage-2 call as well.
// Call with the warp converged, after this thread's rows of the unit are
// stored and visible (a generic store, or a completed bulk store followed by
// fence_proxy_async_global); `valid` and `tok` describe this lane's row.
__device__ __forceinline__ void fused_combine(const GemmArgs &g, int n, int col0, bool valid, int tok, int lane) {
    __threadfence();                                   // release: this row before the count
    bool last = false;
    if (valid) last = atomicAdd(&g.ccnt[static_cast<int64_t>(tok) * g.n_tiles + n], 1) == g.k - 1;
    unsigned done = __ballot_sync(0xffffffffu, last);
    if (done == 0u) return;
    __threadfence();                                   // acquire: the token's other rows
    const int c = col0 + 8 * lane;                     // 8 columns per lane, 256 per warp
    const bool live = c < g.n_out;
    while (done != 0u) {
        const int src = __ffs(done) - 1;
        done &= done - 1u;
        const int t = __shfl_sync(0xffffffffu, tok, src);
        const int my_row = lane < g.k ? __ldg(&g.row_of[static_cast<int64_t>(t) * g.k + lane]) : -1;
        const int n_valid = __popc(__ballot_sync(0xffffffffu, my_row >= 0));
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < g.k; j0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int r = __shfl_sync(0xffffffffu, my_row, (j0 + jj) & 31);
                v[jj] = (live && j0 + jj < g.k && r >= 0)
                            ? ld_cg_v4(g.out + static_cast<int64_t>(r) * g.n_out + c)
                            : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const uint32_t w[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] += bf16_lo(w[q]);
                    acc[2 * q + 1] += bf16_hi(w[q]);
                }
            }
        }
        if (live)
            *reinterpret_cast<uint4 *>(g.y + static_cast<int64_t>(t) * g.n_out + c) =
                make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                           pack_bf16x2(acc[6], acc[7]));
        if (lane == src) g.ccnt[static_cast<int64_t>(t) * g.n_tiles + n] = g.k - n_valid;
    }
}

// Tokens whose every slot was dropped get no row, so no count: their y rows are
// zeroed here (threads first, first + stride, ... over the tokens).
__device__ __forceinline__ void zero_dropped_tokens(const GemmArgs &g, int first, int stride) {
    for (int t = first; t < g.T; t += stride) {
        bool any = false;
        for (int j = 0; j < g.k; ++j) any |= __ldg(&g.row_of[static_cast<int64_t>(t) * g.k + j]) >= 0;
        if (any) continue;
        uint4 *dst = reinterpret_cast<uint4 *>(g.y + static_cast<int64_t>(t) * g.n_out);
        for (int c = 0; c < g.n_out / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// ---------------------------------------------------------------- epilogue pieces

// Stage 1: the SwiGLU of accumulator columns [c, c+32) (gate) and
// [BN/2 + c, ...) (up), packed to bf16.
__device__ __forceinline__ void swiglu_piece(uint32_t tacc, int c, uint32_t (&pk)[16]) {
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
}

// 64 accumulator columns [c, c+64) scaled by w, packed to bf16: both loads in
// flight before the one wait.
__device__ __forceinline__ void scaled_piece2(uint32_t tacc, int c, float w, uint32_t (&pk0)[16],
                                              uint32_t (&pk1)[16]) {
    uint32_t v0[32], v1[32];
    tmem_ld32(tacc + c, v0);
    tmem_ld32(tacc + c + 32, v1);
    tmem_wait_ld();
    tmem_reg_fence(v0);
    tmem_reg_fence(v1);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        pk0[i] = pack_bf16x2(w * __uint_as_float(v0[2 * i]), w * __uint_as_float(v0[2 * i + 1]));
        pk1[i] = pack_bf16x2(w * __uint_as_float(v1[2 * i]), w * __uint_as_float(v1[2 * i + 1]));
    }
}

// dA: the saved h of one row's columns [col, col+32): gate words into hg, the
// matching up words (half columns further on) into hu; zeros past n_out or for
// a row past the unit's count.
__device__ __forceinline__ void load_h_piece(const __nv_bfloat16 *hrow, int half, int col, int n_out, bool valid,
                                             uint32_t (&hg)[16], uint32_t (&hu)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint4 gq = make_uint4(0u, 0u, 0u, 0u), uq = gq;
        if (valid && col + 8 * j < n_out) {
            gq = __ldg(reinterpret_cast<const uint4 *>(hrow + col + 8 * j));
            uq = __ldg(reinterpret_cast<const uint4 *>(hrow + half + col + 8 * j));
        }
        hg[4 * j] = gq.x; hg[4 * j + 1] = gq.y; hg[4 * j + 2] = gq.z; hg[4 * j + 3] = gq.w;
        hu[4 * j] = uq.x; hu[4 * j + 1] = uq.y; hu[4 * j + 2] = uq.z; hu[4 * j + 3] = uq.w;
    }
}

// 32 accumulator columns [c, c+32) scaled by w, packed to bf16.
__device__ __forceinline__ void scaled_piece(uint32_t tacc, int c, float w, uint32_t (&pk)[16]) {
    uint32_t v[32];
    tmem_ld32(tacc + c, v);
    tmem_wait_ld();
    tmem_reg_fence(v);
#pragma unroll
    for (int i = 0; i < 16; ++i)
        pk[i] = pack_bf16x2(w * __uint_as_float(v[2 * i]), w * __uint_as_float(v[2 * i + 1]));
}

// One stage's scale words, from the tail of its B slot, in the tensor-memory
// columns the block-scaled MMA reads: column j < 8 = A row 32 j + lane (j >= 4:
// the second half), column 8 + j = B row 32 j + lane (stage 1: j < 3 the gate
// rows, 3..5 the matching up rows). Each word holds the four E8M0 codes of the
// stage's K steps. Rows past the unit's rows or past n_out get 0 (2^-127), so
// nothing outside the unit enters its accumulators' valid part.
template <int MODE>
__device__ __forceinline__ void stage_scale_words(uint32_t sf_smem, const Unit &t, int rem, int n0, int n_out,
                                                  int lane, uint32_t (&r)[16]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int row = 32 * j + lane;
        const uint32_t off = (j < 4 ? 0u : kSfA1) + 4u * static_cast<uint32_t>(rem + (row & 127));
        r[j] = row < t.rows ? ld_shared_u32(sf_smem + off) : 0u;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        r[8 + j] = 0u;
        if constexpr (MODE == kStage1Mx) {
            const int c = 32 * (j % 3) + lane;
            if (j < 6 && n0 + c < n_out) r[8 + j] = ld_shared_u32(sf_smem + (j < 3 ? kSfB0 : kSfB1) + 4u * c);
        } else {
            const int c = 32 * j + lane;
            if (j < 7 && n0 + c < n_out) r[8 + j] = ld_shared_u32(sf_smem + kSfB0 + 4u * c);
        }
    }
}

// ---------------------------------------------------------------- the kernel

template <int MODE>
__global__ void __launch_bounds__(kNumThreads<MODE>, 1)
tc_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs g) {
    // every CTA is resident from the start (one per SM), so the next kernel may
    // be scheduled right away; it waits for this grid in its own griddep_wait
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw + ((1024u - (raw & 1023u)) & 1023u));
    volatile int *abort_flag = &sm.abort;
    volatile int *unit_q = sm.unit_q;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < (STAGES > kRingSlots ? STAGES : kRingSlots); ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_addr(&sm.sf_full[s]), 1);
            mbar_init(smem_addr(&sm.sf_ready[s]), HELPER_WARPS);
        }
        mbar_init(smem_addr(&sm.acc_full), 1);
        mbar_init(smem_addr(&sm.acc_empty), EPI_THREADS);
        for (int s = 0; s < UQ; ++s) {
            mbar_init(smem_addr(&sm.uq_full[s]), 1);
            mbar_init(smem_addr(&sm.uq_empty[s]), 1 + EPI_WARPS + (kHelpers<MODE> ? HELPER_WARPS : 0));
        }
        mbar_init(smem_addr(&sm.drain), 1);
        mbar_init(smem_addr(&sm.tail_ready), 1);
        mbar_init(smem_addr(&sm.tail_fixed), HELPER_THREADS);
        sm.abort = 0;
        fence_mbar_init();
        tma_prefetch_desc(&maps.a);
        tma_prefetch_desc(&maps.b);
        if constexpr (kIsMx<MODE>) {
            tma_prefetch_desc(&maps.sfa);
            tma_prefetch_desc(&maps.sfb);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sm.tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = sm.tmem_base;
    griddep_wait();     // shared memory and tensor memory are set up; now the inputs

    if (warp == 0) {
        // ------------------------------------------------ scheduler + TMA producer
        const int total = (MODE == kRouter || kPerExpertOut<MODE>) ? g.total_units : g.mt_prefix[g.E] * g.n_tiles;
        int stage = 0, issued = 0, q = 0;
        uint32_t phase = 0, qphase = 0;
        bool ok = true;
        // ring modes: slots rrel .. rj - 1 are in flight; slot m uses barrier pair
        // m % kRingSlots and the bytes [rstart, rend) recorded under that index
        const uint32_t ring0 = smem_addr(sm.a[0]);
        uint32_t rhead = 0, rstart[kRingSlots], rend[kRingSlots];
        int rj = 0, rrel = 0;
#pragma unroll
        for (int i = 0; i < kRingSlots; ++i) rstart[i] = rend[i] = 0;
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
            // one or two 128-row halves of A (K-major rows or MN-major atoms) and the B tile
            const uint32_t a_bytes = unit_a_bytes(t);
            const uint32_t tx_bytes = a_bytes + (MODE == kRouter ? g.n_mma : kUnitN<MODE>) * 128;
            for (int kb = t.kb0; kb < t.kb1; ++kb) {
                uint32_t full, sa, sb;
                if constexpr (kRing<MODE>) {
                    // a slot: the unit's A rows, then its B tile, contiguous; a slot that
                    // would pass the end of the ring starts at its beginning
                    const uint32_t bytes = a_bytes + B_BYTES;
                    const uint32_t base = (rhead + bytes > kRingBytes) ? 0u : rhead;
                    // the newest in-flight slot that must be consumed first: one whose
                    // bytes the new slot reuses, or the one whose barrier pair it takes
                    int need = rj - kRingSlots;
#pragma unroll
                    for (int i = 0; i < kRingSlots; ++i) {
                        const int m = rj - kRingSlots + ((i - (rj - kRingSlots)) % kRingSlots + kRingSlots) % kRingSlots;
                        if (m >= rrel && m >= 0 && rstart[i] < base + bytes && base < rend[i] && m > need) need = m;
                    }
                    if (need >= rrel) {
                        bool e_ok = true;
                        if (lane == 0)
                            e_ok = mbar_wait(smem_addr(&sm.empty[need % kRingSlots]),
                                             static_cast<uint32_t>(need / kRingSlots) & 1u, abort_flag, g.err);
                        e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
                        if (!e_ok) { ok = false; break; }
                        rrel = need + 1;
                    }
                    const int slot = rj % kRingSlots;
#pragma unroll
                    for (int i = 0; i < kRingSlots; ++i)
                        if (i == slot) { rstart[i] = base; rend[i] = base + bytes; }
                    rhead = base + bytes;
                    full = smem_addr(&sm.full[slot]);
                    sa = ring0 + base;
                    sb = sa + a_bytes;
                    ++rj;
                } else {
                    bool e_ok = true;
                    if (lane == 0) e_ok = mbar_wait(smem_addr(&sm.empty[stage]), phase ^ 1u, abort_flag, g.err);
                    e_ok = __shfl_sync(0xffffffffu, e_ok, 0);
                    if (!e_ok) { ok = false; break; }
                    full = smem_addr(&sm.full[stage]);
                    sa = smem_addr(sm.a[stage]);
                    sb = smem_addr(sm.b[stage]);
                }
                if (lane == 0) {
                    if constexpr (kIsMx<MODE>) {
                        // first the stage's scale words (their own barrier, so that the
                        // helper warps can move them into tensor memory while the
                        // operand tiles are still in flight): k-block kb of the unit's A
                        // rows (from the first row rounded down to 4 words) and B rows
                        const uint32_t sff = smem_addr(&sm.sf_full[stage]);
                        const uint32_t sfs = sb + kSfSmemOff;
                        const int ax = t.row0 & ~3;
                        mbar_arrive_expect_tx(sff, sf_stage_bytes(MODE, two));
                        tma_load_2d(sfs, &maps.sfa, ax, kb, sff);
                        if (two) tma_load_2d(sfs + kSfA1, &maps.sfa, ax + BM, kb, sff);
                        if constexpr (MODE == kStage1Mx) {
                            const int row = t.e * g.b_rows + t.n * (kUnitN<MODE> / 2);
                            tma_load_2d(sfs + kSfB0, &maps.sfb, row, kb, sff);              // gate rows
                            tma_load_2d(sfs + kSfB1, &maps.sfb, row + g.half, kb, sff);     // up rows
                        } else {
                            tma_load_2d(sfs + kSfB0, &maps.sfb, t.e * g.b_rows + t.n * kUnitN<MODE>, kb, sff);
                        }
                    }
                    mbar_arrive_expect_tx(full, tx_bytes);
                    if constexpr (kIsStage1<MODE>) {
                        constexpr int hn = kUnitN<MODE> / 2;                                 // gate (= up) rows
                        const int row = t.e * g.b_rows + t.n * hn;
                        const int kx = kb * kStageK<MODE>;
                        tma_load_2d(sa, &maps.a, kx, t.row0, full);                         // dispatched x rows
                        if (two) tma_load_2d(sa + A_HALF_BYTES, &maps.a, kx, t.row0 + BM, full);
                        if (MODE == kStage1 && g.bpack != nullptr) {                        // packed gate + up slab
                            bulk_load(sb, g.bpack + ((static_cast<int64_t>(t.e) * g.n_tiles + t.n) * g.kb_tiles + kb) *
                                                        B_BYTES, B_BYTES, full);
                        } else {
                            tma_load_2d(sb, &maps.b, kx, row, full);                        // gate rows
                            tma_load_2d(sb + hn * 128, &maps.b, kx, row + g.half, full);    // up rows
                        }
                    } else if constexpr (MODE == kWgradMx) {
                        // rows of the m-tile / n-tile of the two quantized operands, K = the
                        // k-block's 128 rows of the expert (absolute column of the operands)
                        const int kx = kb * kStageK<MODE>;
                        tma_load_2d(sa, &maps.a, kx, t.row0, full);
                        if (two) tma_load_2d(sa + A_HALF_BYTES, &maps.a, kx, t.row0 + BM, full);
                        tma_load_2d(sb, &maps.b, kx, t.n * kUnitN<MODE>, full);
                    } else if constexpr (MODE == kStage2 || MODE == kStage2Mx) {
                        const int kx = kb * kStageK<MODE>;
                        tma_load_2d(sa, &maps.a, kx, t.row0, full);
                        if (two) tma_load_2d(sa + A_HALF_BYTES, &maps.a, kx, t.row0 + BM, full);
                        if (MODE == kStage2 && g.bpack != nullptr)                          // packed slab
                            bulk_load(sb, g.bpack + ((static_cast<int64_t>(t.e) * g.n_tiles + t.n) * g.kb_tiles + kb) *
                                                        B_BYTES, B_BYTES, full);
                        else
                            tma_load_2d(sb, &maps.b, kx, t.e * g.b_rows + t.n * kUnitN<MODE>, full);
                    } else if constexpr (MODE == kRouter) {
                        if (g.router_seg) {
                            // one x tile, then the hi, mid and lo rows of w_r, router_seg rows apart
                            const int kx = kb * BK;
                            tma_load_2d(sa, &maps.a, kx, t.row0, full);
                            if (two) tma_load_2d(sa + A_HALF_BYTES, &maps.a, kx, t.row0 + BM, full);
                            for (int part = 0; part < 3; ++part)
                                tma_load_2d(sb + part * g.router_seg * ROW_BYTES, &maps.b, kx, part * g.E, full);
                        } else {
                            // the hi, mid and lo parts of one x k-block in consecutive
                            // k-blocks: the x tile's second and third copies hit L2
                            const int kh = kb / 3;
                            const int seg = kb - 3 * kh;              // 0: hi, 1: mid, 2: lo
                            const int kx = kh * BK;
                            tma_load_2d(sa, &maps.a, kx, t.row0, full);
                            if (two) tma_load_2d(sa + A_HALF_BYTES, &maps.a, kx, t.row0 + BM, full);
                            tma_load_2d(sb, &maps.b, kx, seg * g.E + t.n * BN, full);
                        }
                    } else if constexpr (MODE == kBwdDA || MODE == kBwdDX) {
                        // dA: dispatched dY rows; dX: dH rows
                        tma_load_2d(sa, &maps.a, kb * BK, t.row0, full);
                        if (two) tma_load_2d(sa + A_HALF_BYTES, &maps.a, kb * BK, t.row0 + BM, full);
                        // weight slab of expert e, MN-major: K rows kb*BK.., four 64-wide atoms
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_3d(sb + j * MN_ATOM_BYTES, &maps.b, t.n * BN + 64 * j, kb * BK, t.e, full);
                    } else {
                        // weight gradients, MN-major over K = the expert's routed rows:
                        // A = the m-tile's columns of the dispatched dY rows (dW2) or of
                        // dH (dW1), B = the n-tile's columns of w a (dW2) or of the
                        // dispatched x rows (dW1)
                        const int na = two ? 4 : 2;
                        for (int j = 0; j < na; ++j)
                            tma_load_2d(sa + j * MN_ATOM_BYTES, &maps.a, t.row0 + 64 * j, t.koff + kb * BK, full);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            tma_load_2d(sb + j * MN_ATOM_BYTES, &maps.b, t.n * BN + 64 * j, t.koff + kb * BK, full);
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
            if constexpr (kRing<MODE>) {
                for (int m = rrel; m < rj; ++m)
                    drain_wait(smem_addr(&sm.full[m % kRingSlots]), static_cast<uint32_t>(m / kRingSlots) & 1u);
            } else {
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < min(issued, STAGES); ++i) {
                    if (--s < 0) { s = STAGES - 1; ph ^= 1u; }
                    drain_wait(smem_addr(&sm.full[s]), ph);
                    if constexpr (kIsMx<MODE>) drain_wait(smem_addr(&sm.sf_full[s]), ph);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0, q = 0;
            uint32_t phase = 0, acc_phase = 0, qphase = 0, tail_phase = 0;
            bool ok = true, any = false;
            const uint32_t ring0 = smem_addr(sm.a[0]);
            uint32_t mhead = 0;                 // ring modes: the producer's slot sequence, replayed
            int mj = 0;
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
                const uint32_t a_bytes = unit_a_bytes(t);
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    uint32_t full_bar, empty_bar, fparity, ring_sa = 0;
                    if constexpr (kRing<MODE>) {
                        const uint32_t bytes = a_bytes + B_BYTES;
                        const uint32_t base = (mhead + bytes > kRingBytes) ? 0u : mhead;
                        mhead = base + bytes;
                        full_bar = smem_addr(&sm.full[mj % kRingSlots]);
                        empty_bar = smem_addr(&sm.empty[mj % kRingSlots]);
                        fparity = static_cast<uint32_t>(mj / kRingSlots) & 1u;
                        ring_sa = ring0 + base;
                        ++mj;
                    } else {
                        full_bar = smem_addr(&sm.full[stage]);
                        empty_bar = smem_addr(&sm.empty[stage]);
                        fparity = phase;
                    }
                    if (!mbar_wait(full_bar, fparity, abort_flag, g.err)) {
                        ok = false;
                        break;
                    }
                    if constexpr (kIsMx<MODE>) {
                        // ... and the helper warps have put its scale factors in tensor memory
                        if (!mbar_wait(smem_addr(&sm.sf_ready[stage]), fparity, abort_flag, g.err)) {
                            ok = false;
                            break;
                        }
                    }
                    tc_fence_after();
                    if constexpr (kWeightGrad<MODE>) {
                        if (kb == t.kb1 - 1 && t.kcount % BK != 0) {
                            // the helpers zero this block's K rows past the expert's count first
                            mbar_arrive(smem_addr(&sm.tail_ready));
                            if (!mbar_wait(smem_addr(&sm.tail_fixed), tail_phase, abort_flag, g.err)) {
                                ok = false;
                                break;
                            }
                            tail_phase ^= 1u;
                            tc_fence_after();
                        }
                    }
                    const uint32_t sa = kRing<MODE> ? ring_sa : smem_addr(sm.a[stage]);
                    const uint32_t sb = kRing<MODE> ? ring_sa + a_bytes : smem_addr(sm.b[stage]);
                    if constexpr (kIsMx<MODE>) {
                        // four K = 32 steps; the scale words of this stage hold one byte per step
                        const uint32_t sf = tmem_base + kSfBase<MODE> + stage * kSfStride;
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint32_t acc = (kb > t.kb0 || kk > 0) ? 1u : 0u;
                            const uint32_t idesc = idesc_mxf8(BM, kUnitN<MODE>, kk);
                            const uint64_t bdesc = smem_desc_swizzled<128>(sb + kk * 32);
                            mma_mxf8(tmem_base, smem_desc_swizzled<128>(sa + kk * 32), bdesc, idesc, sf, sf + 8, acc);
                            if (two)
                                mma_mxf8(tmem_base + kUnitN<MODE>, smem_desc_swizzled<128>(sa + A_HALF_BYTES + kk * 32),
                                         bdesc, idesc, sf + 4, sf + 8, acc);
                        }
                    } else {
                        // the router's N follows E; the expert GEMMs use the full 256
                        const uint32_t idesc = MODE == kRouter ? idesc_bf16_f32(BM, g.n_mma) : kIdesc<MODE>;
#pragma unroll
                        for (int kk = 0; kk < BK / UMMA_K; ++kk) {
                            const uint32_t acc = (kb > t.kb0 || kk > 0) ? 1u : 0u;
                            const uint64_t bdesc = operand_desc<kBMn<MODE>>(sb, kk);
                            mma_bf16(tmem_base, operand_desc<kAMn<MODE>>(sa, kk), bdesc, idesc, acc);
                            if (two)
                                mma_bf16(tmem_base + BN, operand_desc<kAMn<MODE>>(sa + A_HALF_BYTES, kk), bdesc,
                                         idesc, acc);
                        }
                    }
                    mma_commit(empty_bar);                     // frees the smem stage (or slot)
                    any = true;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                // accumulators ready (with no k-block, at once: the epilogue then
                // writes zeros without reading them)
                mma_commit(smem_addr(&sm.acc_full));
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
                              static_cast<uint32_t>(half * kUnitN<MODE>);
        const uint32_t buf = smem_addr(sm.stage_out[warp - 2]);
        uint32_t boxes = 0;                         // 32 x 32 boxes stored so far (ping-pong halves)
        int q = 0;
        uint32_t acc_phase = 0, qphase = 0;
        if constexpr (MODE == kStage2) {
            if (g.ccnt != nullptr)
                zero_dropped_tokens(g, blockIdx.x * EPI_THREADS + (threadIdx.x - 64), gridDim.x * EPI_THREADS);
        }
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
            float w = 1.0f;                             // routing weight of the row's slot
            int tok = -1;                               // stage 2: the row's token (fused combine)
            if constexpr (MODE == kStage2 || MODE == kBwdDA || MODE == kStage2Mx) {
                const int slot = valid ? g.perm_slot[t.row0 + row] : 0;
                w = valid ? g.topk_w[slot] : 0.0f;
                tok = valid ? slot / g.k : -1;
            }
            // dA: the saved h (gate and up) of the row's first 32 columns, loaded while
            // the unit's MMAs still run; each later piece's h is loaded before the
            // previous piece's stores, so the epilogue rarely waits for global memory
            uint32_t hg[16], hu[16];
            const __nv_bfloat16 *hrow = nullptr;
            if constexpr (MODE == kBwdDA) {
                hrow = g.h + (valid ? static_cast<int64_t>(t.row0 + row) : 0) * (2 * static_cast<int64_t>(g.half));
                load_h_piece(hrow, g.half, t.n * BN, g.n_out, valid, hg, hu);
            }
            if (lane == 0) ok = mbar_wait(smem_addr(&sm.acc_full), acc_phase, abort_flag, g.err);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after();
            bool released = false;                      // this thread's acc_empty arrival done
            const int slab0 = half * BM + quad * 32;    // first unit row of this warp
            const bool full_slab = slab0 + 32 <= t.rows;
            if (t.rows > half * BM) {                   // this half was computed
                if constexpr (MODE == kStage1Mx) {
                    // per 32 output columns: SwiGLU of the gate / up columns, then the
                    // MXFP8 quantization of that block of a (32 E4M3 codes, one E8M0
                    // scale). The accumulator is released as soon as the last piece has
                    // been read from tensor memory, before that piece's arithmetic.
                    const int col0 = t.n * (kUnitN<MODE> / 2);
                    const int np = min(kUnitN<MODE> / 64, (g.n_out - col0 + 31) / 32);   // pieces inside n_out
                    const int64_t r = t.row0 + row;
#pragma unroll 1
                    for (int p = 0; p < np; ++p) {
                        const int c = 32 * p;
                        uint32_t gv[32], uv[32];
                        tmem_ld32(tacc + c, gv);
                        tmem_ld32(tacc + kUnitN<MODE> / 2 + c, uv);
                        tmem_wait_ld();
                        tmem_reg_fence(gv);
                        tmem_reg_fence(uv);
                        if (p == np - 1) {
                            tc_fence_before();
                            mbar_arrive(smem_addr(&sm.acc_empty));
                            released = true;
                        }
                        if (g.out2 != nullptr && valid) {
                            // training: the pre-activation h (gate and up halves, bf16) for the backward
                            uint32_t pg[16], pu[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                pg[i] = pack_bf16x2(__uint_as_float(gv[2 * i]), __uint_as_float(gv[2 * i + 1]));
                                pu[i] = pack_bf16x2(__uint_as_float(uv[2 * i]), __uint_as_float(uv[2 * i + 1]));
                            }
                            store_row32(g.out2 + r * g.out_ld + col0 + c, g.n_out - col0 - c, pg);
                            store_row32(g.out3 + r * g.out_ld + col0 + c, g.n_out - col0 - c, pu);
                        }
                        float av[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) av[i] = silu_mul(__uint_as_float(gv[i]), __uint_as_float(uv[i]));
                        uint32_t q[8];
                        const uint32_t sc = mx_quantize32(av, q);
                        if (valid) {
                            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(g.out) + r * g.n_out + col0 + c);
                            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
                            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
                            // k-block-major scales: byte (col / 32) % 4 of word [col / 128][r]
                            const int col = col0 + c;
                            g.out_sf[((static_cast<int64_t>(col >> 7) * g.sf_rows + r) << 2) + ((col >> 5) & 3)] =
                                static_cast<uint8_t>(sc);
                        }
                    }
                } else if constexpr (MODE == kStage2Mx) {
                    // weighted rows into obuf, 32 x 32 boxes (the unit is 224 columns wide)
                    constexpr int NP = kUnitN<MODE> / 32;
                    const int col0 = t.n * kUnitN<MODE>;
                    const int y = t.row0 + slab0;
                    if (full_slab) {
                        // the first two boxes are staged at once (both staging halves), the
                        // rest of the row read into packed bf16 registers; then the
                        // accumulator is released and the stores overlap the next unit's MMAs
                        uint32_t pks[NP][16];
                        scaled_piece2(tacc, 0, w, pks[0], pks[1]);
                        if (lane == 0) bulk_wait_read<0>();       // the previous unit's boxes are read out
                        __syncwarp();
                        stage_row32(buf, lane, pks[0]);
                        stage_row32(buf + 2048, lane, pks[1]);
#pragma unroll
                        for (int p = 2; p + 1 < NP; p += 2) scaled_piece2(tacc, 32 * p, w, pks[p], pks[p + 1]);
                        if constexpr (NP % 2 == 1) scaled_piece(tacc, 32 * (NP - 1), w, pks[NP - 1]);
                        tc_fence_before();
                        mbar_arrive(smem_addr(&sm.acc_empty));
                        released = true;
                        fence_proxy_async_smem();
                        __syncwarp();
#pragma unroll
                        for (int p = 0; p < NP; ++p) {
                            const int col = col0 + 32 * p;
                            if (col >= g.n_out) break;
                            const uint32_t b2 = buf + (p & 1) * 2048;
                            if (p >= 2) {
                                if (lane == 0) bulk_wait_read<1>();   // the box two boxes ago is read out
                                __syncwarp();
                                stage_row32(b2, lane, pks[p]);
                                fence_proxy_async_smem();
                                __syncwarp();
                            }
                            if (lane == 0) {
                                tma_store_2d(&maps.out, b2, col, y);
                                bulk_commit();
                            }
                        }
                    } else {
                        // partial slab: masked direct stores, piece by piece
                        __nv_bfloat16 *dst = g.out + static_cast<int64_t>(t.row0 + row) * g.n_out;
#pragma unroll 1
                        for (int c = 0; c < kUnitN<MODE>; c += 32) {
                            const int col = col0 + c;
                            if (col >= g.n_out) break;
                            uint32_t pk[16];
                            scaled_piece(tacc, c, w, pk);
                            if (valid) store_row32(dst + col, g.n_out - col, pk);
                        }
                    }
                } else if constexpr (kIsStage1<MODE> || MODE == kStage2 || MODE == kBwdDX) {
                    // row-grouped outputs: rows t.row0 + row, columns [col0, col0 + ncols)
                    constexpr int ncols = kIsStage1<MODE> ? BN / 2 : BN;
                    const int col0 = t.n * ncols;
                    const int y = t.row0 + slab0;
                    if constexpr (MODE == kStage1SaveH) {
                        // a, h gate and h up in 32 x 32 boxes (two staging halves)
                        const int64_t r = t.row0 + row;
#pragma unroll 1
                        for (int c = 0; c < ncols; c += 32) {
                            if (col0 + c >= g.n_out) break;
                            uint32_t gv[32], uv[32];
                            tmem_ld32(tacc + c, gv);
                            tmem_ld32(tacc + BN / 2 + c, uv);
                            tmem_wait_ld();
                            tmem_reg_fence(gv);
                            tmem_reg_fence(uv);
                            uint32_t pg[16], pu[16], pa[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                pg[i] = pack_bf16x2(__uint_as_float(gv[2 * i]), __uint_as_float(gv[2 * i + 1]));
                                pu[i] = pack_bf16x2(__uint_as_float(uv[2 * i]), __uint_as_float(uv[2 * i + 1]));
                            }
                            if (full_slab) {
                                if (lane == 0) bulk_wait_read<0>();
                                __syncwarp();
                                stage_row32(buf, lane, pg);
                                stage_row32(buf + 2048, lane, pu);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_2d(&maps.out2, buf, col0 + c, y);
                                    tma_store_2d(&maps.out3, buf + 2048, col0 + c, y);
                                    bulk_commit();
                                }
                            } else if (valid) {
                                store_row32(g.out2 + r * g.out_ld + col0 + c, g.n_out - col0 - c, pg);
                                store_row32(g.out3 + r * g.out_ld + col0 + c, g.n_out - col0 - c, pu);
                            }
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pa[i] = pack_bf16x2(
                                    silu_mul(__uint_as_float(gv[2 * i]), __uint_as_float(uv[2 * i])),
                                    silu_mul(__uint_as_float(gv[2 * i + 1]), __uint_as_float(uv[2 * i + 1])));
                            if (full_slab) {
                                if (lane == 0) bulk_wait_read<0>();
                                __syncwarp();
                                stage_row32(buf, lane, pa);
                                fence_proxy_async_smem();
                                __syncwarp();
                                if (lane == 0) {
                                    tma_store_2d(&maps.out, buf, col0 + c, y);
                                    bulk_commit();
                                }
                            } else if (valid) {
                                store_row32(g.out + r * g.n_out + col0 + c, g.n_out - col0 - c, pa);
                            }
                        }
                    } else if (full_slab) {
                        // whole 32-row slab valid: stage 32 x 64 bf16 boxes in shared
                        // memory (128B-swizzled) and write each with one TMA store. The
                        // row's first box is staged at once and the rest is converted
                        // into packed bf16 registers, so the accumulator is released
                        // before the stores: their shared-memory waits overlap the
                        // next unit's MMAs.
                        constexpr int NPIECE = ncols / 32;
                        uint32_t pk[NPIECE][16];
#pragma unroll
                        for (int p = 0; p < NPIECE; ++p) {
                            if constexpr (MODE == kStage1) swiglu_piece(tacc, 32 * p, pk[p]);
                            else if (p % 2 == 0) scaled_piece2(tacc, 32 * p, w, pk[p], pk[p + 1]);
                            if (p == 1) {                     // box 0 complete: stage it
                                if (lane == 0) bulk_wait_read<0>();   // previous box read out
                                __syncwarp();
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const uint32_t *q = &pk[j >> 2][4 * (j & 3)];
                                    st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), q[0], q[1], q[2],
                                                 q[3]);
                                }
                            }
                        }
                        tc_fence_before();
                        mbar_arrive(smem_addr(&sm.acc_empty));
                        released = true;
#pragma unroll
                        for (int b = 0; b < NPIECE / 2; ++b) {
                            if (col0 + 64 * b >= g.n_out) break;
                            if (b > 0) {
                                if (lane == 0) bulk_wait_read<0>();   // previous box read out
                                __syncwarp();
#pragma unroll
                                for (int j = 0; j < 8; ++j) {
                                    const uint32_t *q = &pk[2 * b + (j >> 2)][4 * (j & 3)];
                                    st_shared_v4(buf + lane * 128 + ((j ^ (lane & 7)) << 4), q[0], q[1], q[2],
                                                 q[3]);
                                }
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                // stage 2's weighted rows are read again by the combine: keep
                                // them in L2 ahead of the weight stream
                                if constexpr (MODE == kStage2)
                                    tma_store_2d_hint(&maps.out, buf, col0 + 64 * b, y, l2_policy_evict_last());
                                else
                                    tma_store_2d(&maps.out, buf, col0 + 64 * b, y);
                                bulk_commit();
                            }
                        }
                        if constexpr (MODE == kStage2) {
                            if (g.ccnt != nullptr) {
                                if (lane == 0) {
                                    bulk_wait<0>();                 // the slab's rows are in global memory
                                    fence_proxy_async_global();
                                }
                                __syncwarp();
                                fused_combine(g, t.n, col0, valid, tok, lane);
                            }
                        }
                    } else {
                        // partial slab (the expert's last rows): masked direct stores. Stage 2
                        // first reads the row's columns into packed registers, as its full-slab
                        // path does, and releases the accumulator before storing (a unit's
                        // release waits for its slowest warp); in stage 1 and dX the extra
                        // registers spill and cost more than they save.
                        __nv_bfloat16 *dst = g.out + static_cast<int64_t>(t.row0 + row) * g.n_out + col0;
                        if constexpr (MODE == kStage2) {
                            constexpr int NPIECE = ncols / 32;
                            uint32_t pk[NPIECE][16];
#pragma unroll
                            for (int p = 0; p < NPIECE; p += 2) scaled_piece2(tacc, 32 * p, w, pk[p], pk[p + 1]);
                            tc_fence_before();
                            mbar_arrive(smem_addr(&sm.acc_empty));
                            released = true;
                            if (valid) {
#pragma unroll
                                for (int p = 0; p < NPIECE; ++p)
                                    if (col0 + 32 * p < g.n_out) store_row32(dst + 32 * p, g.n_out - col0 - 32 * p, pk[p]);
                            }
                            if (g.ccnt != nullptr) {
                                __syncwarp();
                                fused_combine(g, t.n, col0, valid, tok, lane);
                            }
                        } else {
#pragma unroll 1
                            for (int c = 0; c < ncols; c += 32) {
                                if (col0 + c >= g.n_out) break;
                                uint32_t pk[16];
                                if constexpr (MODE == kStage1) swiglu_piece(tacc, c, pk);
                                else scaled_piece(tacc, c, w, pk);
                                if (valid) store_row32(dst + c, g.n_out - col0 - c, pk);
                            }
                        }
                    }
                } else if constexpr (MODE == kBwdDA) {
                    // SwiGLU backward: dG, dU (dH halves) and w a, plus sum_i dA_u a
                    const int col0 = t.n * BN;
                    const int y = t.row0 + slab0;
                    const int64_t r = t.row0 + row;
                    float dtw = 0.0f;
#pragma unroll 1
                    for (int c = 0; c < BN; c += 32) {
                        const int col = col0 + c;
                        if (col >= g.n_out) break;
                        uint32_t v[32];
                        tmem_ld32(tacc + c, v);
                        tmem_wait_ld();
                        tmem_reg_fence(v);
                        uint32_t pdg[16], pdu[16], paw[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float og[2], ou[2], oa[2];
#pragma unroll
                            for (int e2 = 0; e2 < 2; ++e2) {
                                const float gv = e2 ? bf16_hi(hg[i]) : bf16_lo(hg[i]);
                                const float uv = e2 ? bf16_hi(hu[i]) : bf16_lo(hu[i]);
                                const float d = __uint_as_float(v[2 * i + e2]);
                                const float sg = sigmoid_tanh(gv);
                                const float silu = gv * sg;
                                const float a = silu * uv;
                                dtw = fmaf(d, a, dtw);
                                const float dA = w * d;
                                ou[e2] = dA * silu;
                                og[e2] = dA * uv * sg * fmaf(gv, 1.0f - sg, 1.0f);
                                oa[e2] = w * a;
                            }
                            pdg[i] = pack_bf16x2(og[0], og[1]);
                            pdu[i] = pack_bf16x2(ou[0], ou[1]);
                            paw[i] = pack_bf16x2(oa[0], oa[1]);
                        }
                        if (c + 32 < BN && col + 32 < g.n_out)          // the next piece's h
                            load_h_piece(hrow, g.half, col + 32, g.n_out, valid, hg, hu);
                        if (full_slab) {
                            if (lane == 0) bulk_wait_read<0>();
                            __syncwarp();
                            stage_row32(buf, lane, pdg);
                            stage_row32(buf + 2048, lane, pdu);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&maps.out, buf, col, y);
                                tma_store_2d(&maps.out2, buf + 2048, col, y);
                                bulk_commit();
                                bulk_wait_read<0>();
                            }
                            __syncwarp();
                            stage_row32(buf, lane, paw);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_2d(&maps.out3, buf, col, y);
                                bulk_commit();
                            }
                        } else if (valid) {
                            store_row32(g.out + r * g.out_ld + col, g.n_out - col, pdg);
                            store_row32(g.out2 + r * g.out_ld + col, g.n_out - col, pdu);
                            store_row32(g.out3 + r * g.n_out + col, g.n_out - col, paw);
                        }
                    }
                    if (valid) g.dtw_part[static_cast<int64_t>(t.n) * g.R + r] = dtw;
                } else if constexpr (MODE == kWgradMx) {
                    // as stage 2 in MXFP8: dW rows t.row0 + row of expert e through a 3-D
                    // map (rows past m_total and columns past n_out clipped by the store);
                    // the first two 32 x 32 boxes staged at once, the rest of the row in
                    // packed registers, then the accumulator released (a unit reduces over
                    // only its expert's rows, so its MMAs are short and its stores are
                    // better spent under the next unit's)
                    constexpr int NP = kUnitN<MODE> / 32;
                    const int col0 = t.n * kUnitN<MODE>;
                    const bool empty = t.kb1 == t.kb0;  // expert without rows: zeros
                    if (slab0 < t.rows && empty) {
                        // expert without rows: zero boxes, the accumulator untouched
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) pk[i] = 0u;
#pragma unroll 1
                        for (int p = 0; p < NP; ++p) {
                            const int col = col0 + 32 * p;
                            if (col >= g.n_out) break;
                            // the first box: the previous unit's last box may be in either half
                            if (lane == 0) {
                                if (p == 0) bulk_wait_read<0>();
                                else bulk_wait_read<1>();
                            }
                            __syncwarp();
                            const uint32_t b2 = buf + (p & 1) * 2048;
                            stage_row32(b2, lane, pk);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_3d(&maps.out, b2, col, t.row0 + slab0, t.e);
                                bulk_commit();
                            }
                        }
                    } else if (slab0 < t.rows) {
                        uint32_t pks[NP][16];
                        scaled_piece2(tacc, 0, 1.0f, pks[0], pks[1]);
                        if (lane == 0) bulk_wait_read<0>();       // the previous unit's boxes are read out
                        __syncwarp();
                        stage_row32(buf, lane, pks[0]);
                        stage_row32(buf + 2048, lane, pks[1]);
#pragma unroll
                        for (int p = 2; p + 1 < NP; p += 2) scaled_piece2(tacc, 32 * p, 1.0f, pks[p], pks[p + 1]);
                        if constexpr (NP % 2 == 1) scaled_piece(tacc, 32 * (NP - 1), 1.0f, pks[NP - 1]);
                        tc_fence_before();
                        mbar_arrive(smem_addr(&sm.acc_empty));
                        released = true;
                        fence_proxy_async_smem();
                        __syncwarp();
#pragma unroll
                        for (int p = 0; p < NP; ++p) {
                            const int col = col0 + 32 * p;
                            if (col >= g.n_out) break;
                            const uint32_t b2 = buf + (p & 1) * 2048;
                            if (p >= 2) {
                                if (lane == 0) bulk_wait_read<1>();   // the box two boxes ago is read out
                                __syncwarp();
                                stage_row32(b2, lane, pks[p]);
                                fence_proxy_async_smem();
                                __syncwarp();
                            }
                            if (lane == 0) {
                                tma_store_3d(&maps.out, b2, col, t.row0 + slab0, t.e);
                                bulk_commit();
                            }
                        }
                    }
                } else if constexpr (kPerExpertOut<MODE>) {
                    // dW rows t.row0 + row of expert e, 32 x 32 boxes through a 3-D map
                    // (rows past m_total and columns past n_out are clipped by the store),
                    // staged in the two halves of the warp's buffer in turn, so staging a
                    // box waits only for the one two boxes back to be read out
                    constexpr int NC = kUnitN<MODE>;
                    const int col0 = t.n * NC;
                    const bool empty = t.kb1 == t.kb0;  // expert without rows: zeros
                    if (slab0 < t.rows) {
#pragma unroll 1
                        for (int c = 0; c < NC; c += 32) {
                            if (col0 + c >= g.n_out) break;
                            uint32_t pk[16];
                            if (empty) {
#pragma unroll
                                for (int i = 0; i < 16; ++i) pk[i] = 0u;
                            } else {
                                scaled_piece(tacc, c, 1.0f, pk);
                            }
                            if (lane == 0) bulk_wait_read<1>();
                            __syncwarp();
                            const uint32_t b2 = buf + (boxes++ & 1u) * 2048;
                            stage_row32(b2, lane, pk);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                tma_store_3d(&maps.out, b2, col0 + c, t.row0 + slab0, t.e);
                                bulk_commit();
                            }
                        }
                    }
                } else {
                    const int col0 = t.n * BN;
                    float *dst = g.logits_part +
                                 (static_cast<int64_t>(t.split) * g.T + t.row0 + row) * g.n_out + col0;
                    const bool vec = (g.n_out & 3) == 0;
                    const int ncols = g.router_seg ? g.router_seg : g.n_mma;
#pragma unroll 1
                    for (int c = 0; c < ncols; c += 32) {
                        uint32_t v[32];
                        tmem_ld32(tacc + c, v);
                        if (g.router_seg) {
                            // logits = (hi + mid) + lo, each part's partial sum from its own columns
                            uint32_t vm[32], vl[32];
                            tmem_ld32(tacc + g.router_seg + c, vm);
                            tmem_ld32(tacc + 2 * g.router_seg + c, vl);
                            tmem_wait_ld();
                            tmem_reg_fence(v);
                            tmem_reg_fence(vm);
                            tmem_reg_fence(vl);
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                v[j] = __float_as_uint((__uint_as_float(v[j]) + __uint_as_float(vm[j])) +
                                                       __uint_as_float(vl[j]));
                        }
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
            if (!released) {
                tc_fence_before();
                mbar_arrive(smem_addr(&sm.acc_empty));
            }
            acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait<0>();                  // every output box written
    } else {
        // ------------------------------------------------ helpers
        // Weight gradients: the reduction runs over the expert's routed rows, so
        // the tiles of its last, partial k-block also hold rows past its count
        // (the next expert's rows, or rows never written). When the MMA issuer
        // has seen such a block land it signals tail_ready; these 128 threads
        // then zero the block's K rows >= count in the dispatched operand (dY
        // rows: dW2's A; x rows: dW1's B) and signal tail_fixed. The other
        // operand's rows there are finite (dH and w a have their dropped-slot
        // rows zeroed), so the padding adds nothing.
        // MXFP8 modes: each stage's scale factors into tensor memory.
        const int ht = threadIdx.x - (64 + EPI_THREADS);
        int stage = 0, q = 0;
        uint32_t phase = 0, qphase = 0, tail_phase = 0;
        bool ok = true;
        while (ok) {
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
            if constexpr (kWeightGrad<MODE>) {
                const int nkb = t.kb1 - t.kb0;
                const int rem = t.kcount % BK;
                if (nkb > 0 && rem != 0) {
                    if (lane == 0) ok = mbar_wait(smem_addr(&sm.tail_ready), tail_phase, abort_flag, g.err);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    tail_phase ^= 1u;
                    const int tail = (stage + nkb - 1) % STAGES;
                    const uint32_t base = smem_addr(MODE == kBwdDW2 ? sm.a[tail] : sm.b[tail]);
                    const int atoms = (MODE == kBwdDW2 && t.rows <= BM) ? 2 : 4;
                    const int per_atom = (BK - rem) * (128 / 16);          // 16-byte chunks of rows rem..BK-1
                    for (int i = ht; i < atoms * per_atom; i += HELPER_THREADS) {
                        const int at = i / per_atom;
                        st_shared_v4(base + at * MN_ATOM_BYTES + rem * 128 + (i - at * per_atom) * 16, 0u, 0u, 0u,
                                     0u);
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(smem_addr(&sm.tail_fixed));
                }
                stage = (stage + nkb) % STAGES;
            } else if constexpr (kIsMx<MODE>) {
                // A, B and their scale words arrive through TMA, the scale words on
                // their own barrier; these warps move them into tensor memory and
                // then release the stage's scale factors to the MMA issuer
                const int rem = t.row0 & 3;                 // the A boxes start 16-byte aligned
                const int n0 = t.n * (MODE == kStage1Mx ? kUnitN<MODE> / 2 : kUnitN<MODE>);
                const uint32_t sf_lane = tmem_base + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kSfBase<MODE>;
                for (int kb = t.kb0; kb < t.kb1; ++kb) {
                    const uint32_t sff = smem_addr(&sm.sf_full[stage]);
                    if (lane == 0) ok = mbar_wait(sff, phase, abort_flag, g.err);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) break;
                    // the phase is complete (the stage cannot be refilled before this
                    // warp's release below); every lane observes it before reading
                    (void)mbar_try_wait(sff, phase);
                    uint32_t sfw[16];
                    stage_scale_words<MODE>(smem_addr(sm.b[stage]) + kSfSmemOff, t, rem, n0, g.n_out, lane, sfw);
                    tc_fence_after();
                    tmem_st16(sf_lane + stage * kSfStride, sfw);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();           // every lane's stores are complete: one arrival per warp
                    if (lane == 0) mbar_arrive(smem_addr(&sm.sf_ready[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
            }
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

// Grouped-mode arguments shared by every launcher.
inline GemmArgs grouped_args(const GemmLaunch &p) {
    GemmArgs g{};
    g.counts = p.counts;
    g.offsets = p.offsets;
    g.mt_prefix = p.mt_prefix;
    g.perm_slot = p.perm_slot;
    g.h = p.h;
    g.err = p.err;
    g.sched = p.sched;
    g.topk_w = p.topk_w;
    g.row_of = p.row_of;
    g.y = p.y;
    g.ccnt = p.ccnt;
    g.T = p.T;
    g.out = p.out;
    g.out2 = p.out2;
    g.out3 = p.out3;
    g.dtw_part = p.dtw_part;
    g.out_sf = p.out_sf;
    g.sf_rows = p.sf_rows;
    g.bpack = p.bpack;
    g.kpad = p.kpad;
    g.kb_tiles = (p.K + BK - 1) / BK;
    g.E = p.E;
    g.k = p.k;
    g.K = p.K;
    g.n_out = p.n_out;
    g.n_tiles = (p.n_out + p.n_tile - 1) / p.n_tile;
    g.m_total = p.m_total;
    g.m_tiles = (p.m_total + UM - 1) / UM;
    g.b_rows = p.b_rows;
    g.half = p.half;
    g.out_ld = p.out_ld;
    g.R = p.R;
    g.total_units = -1;
    return g;
}

inline GemmMaps maps_of(const GemmLaunch &p) {
    GemmMaps m;
    m.a = *(p.tm_a ? p.tm_a : p.tm_b);
    m.b = *p.tm_b;
    m.out = *p.tm_out;
    m.out2 = *(p.tm_out2 ? p.tm_out2 : p.tm_out);
    m.out3 = *(p.tm_out3 ? p.tm_out3 : p.tm_out);
    m.sfa = *(p.tm_sfa ? p.tm_sfa : p.tm_b);
    m.sfb = *(p.tm_sfb ? p.tm_sfb : p.tm_b);
    return m;
}

template <int MODE>
cudaError_t set_gemm_smem() {
    return cudaFuncSetAttribute(tc_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(SMEM_BYTES));
}

template <int MODE>
cudaError_t launch_tc_gemm(const GemmMaps &maps, const GemmArgs &g, int grid, cudaStream_t st) {
    const cudaError_t e = launch_dep(tc_gemm_kernel<MODE>, dim3(grid), dim3(kNumThreads<MODE>), SMEM_BYTES, st, maps, g);
    note_launches(1);
    return e;
}

}  // namespace

}  // namespace moe
