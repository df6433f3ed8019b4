// internal.cuh -- declarations shared by the CUDA translation units of libmoe.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "moe.h"

namespace moe {

// Rows per MMA (one TMEM accumulator holds 128 rows). A GEMM work unit spans
// kUnitM = 2 * kBM rows that share every weight tile; the routing metadata
// counts row tiles in units of kUnitM, so every grouped GEMM uses that value.
constexpr int kBM = 128;
constexpr int kUnitM = 256;
// MXFP8: words of a TMA box of one 128-row half's scale words (128 rows plus up
// to 3 before them, the box starting at the half's first row rounded down to 4)
constexpr int kSfBoxRowsA = kBM + 4;
// Reduction depth of one pipeline stage: 32 bf16 = 64-byte rows with the 64-byte
// swizzle (six 32 KB stages), or 64 = 128-byte rows with the 128-byte swizzle
// (three 64 KB stages).
#ifndef MOE_STAGE_BK
#define MOE_STAGE_BK 64
#endif
constexpr int kBK = MOE_STAGE_BK;
static_assert(kBK == 32 || kBK == 64, "stage depth must be 32 or 64");
constexpr int kBN = 256;    // accumulator columns of one tile

// Workspace header (zeroed by moe_workspace_init):
//   byte 0  int32 device error word
//   byte 4  int32 router top-k block ticket
//   byte 8  int32[2] stage-1 unit scheduler (next unit, finished CTAs)
//   byte 16 int32[2] stage-2 unit scheduler
//   byte 24 int32[2] router-GEMM unit scheduler
//   byte 32 int32    routing-metadata block ticket
constexpr size_t kWsHeaderBytes = 256;

// Slots per CTA of the routing-metadata kernels (one histogram row each).
constexpr int kMetaChunk = 1024;

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Router GEMM layout (logits = x . w_r^T with w_r split into three bf16 parts). With E <= 64 one MMA of N = 3 * router_seg(E) multiplies
// an x tile by the hi, mid and lo parts of w_r at once (each part's rows padded
// to router_seg(E) accumulator columns), so x is loaded once per k-block;
// otherwise the three parts are separate k-blocks of the reduction, the three
// of one x k-block consecutive.
inline int router_seg(int64_t E) { return E <= 32 ? 32 : (E <= 64 ? 64 : 0); }
inline int64_t router_kb_total(int64_t H, int64_t E) {
    const int64_t kb_h = (H + kBK - 1) / kBK;
    return router_seg(E) ? kb_h : 3 * kb_h;
}

inline int router_splits(int64_t T, int64_t H, int64_t E) {
    // Split-K count of the router GEMM: the one that minimises an estimated time,
    // whole waves of units over the 152 SMs times the k-blocks of a unit (~0.6 us
    // each), plus writing and re-reading one more [T, E] fp32 partial (~6 TB/s)
    // per split. Every split owns at least one k-block.
    const int64_t tiles = ((T + kUnitM - 1) / kUnitM) * ((E + kBN - 1) / kBN);
    const int64_t kb_total = router_kb_total(H, E);
    const int64_t smax = kb_total < 32 ? kb_total : 32;
    int best = 1;
    double best_cost = 0.0;
    for (int64_t s = 1; s <= smax; ++s) {
        const int64_t per = (kb_total + s - 1) / s;
        const int64_t splits = (kb_total + per - 1) / per;
        const int64_t waves = (tiles * splits + 151) / 152;
        const double cost = 0.6 * static_cast<double>(waves * per) + 8.0 * static_cast<double>(splits * T * E) / 6.0e6;
        if (s == 1 || cost < best_cost) {
            best_cost = cost;
            best = static_cast<int>(splits);
        }
    }
    return best;
}

// N of the router GEMM's MMAs and rows of its weight tile: E rounded up to a
// whole 32-column TMEM load, at most one 256-column tile.
inline int router_n_mma(int64_t E) { return E >= kBN ? kBN : static_cast<int>((E + 31) / 32 * 32); }

// Bytes of router scratch for a shape and split factor.
inline size_t router_scratch_bytes(int64_t T, int64_t H, int64_t E, int splits) {
    return align256(4 * static_cast<size_t>(splits) * T * E) +   // partial logits
           align256(2 * 3 * static_cast<size_t>(E) * H) +         // bf16 x3 split of w_r
           align256(4 * static_cast<size_t>(E)) +                 // score sums
           align256(4 * static_cast<size_t>(E)) +                 // counts
           256;                                                   // ticket + scheduler
}

struct RouterScratch {
    float *logits_part;       // [splits, T, E] partial fp32 logits
    __nv_bfloat16 *w3;        // [3, E, H]: hi, mid, lo parts of w_r
    float *score_sum;         // [E]  sum over tokens of the full score vector
    int32_t *counts;          // [E]  rows the router sent to each expert
    int32_t *ticket;          // top-k blocks that have finished
    int32_t *sched;           // [2] router-GEMM unit scheduler
    int splits;
};

// Carve router scratch out of `base` (256-byte aligned).
inline RouterScratch carve_router_scratch(unsigned char *base, int64_t T, int64_t H, int64_t E,
                                          int splits, int32_t *ticket, int32_t *sched) {
    RouterScratch r;
    size_t off = 0;
    r.logits_part = reinterpret_cast<float *>(base + off);
    off += align256(4 * static_cast<size_t>(splits) * T * E);
    r.w3 = reinterpret_cast<__nv_bfloat16 *>(base + off);
    off += align256(2 * 3 * static_cast<size_t>(E) * H);
    r.score_sum = reinterpret_cast<float *>(base + off);
    off += align256(4 * static_cast<size_t>(E));
    r.counts = reinterpret_cast<int32_t *>(base + off);
    off += align256(4 * static_cast<size_t>(E));
    r.ticket = ticket ? ticket : reinterpret_cast<int32_t *>(base + off);
    r.sched = sched ? sched : reinterpret_cast<int32_t *>(base + off + 64);
    r.splits = splits;
    return r;
}

struct RouterLaunch {
    const __nv_bfloat16 *x;
    const float *w_r;
    const float *logit_offset;  // may be null
    const float *sel_bias;      // may be null
    int T, H, E, k;
    int score_fn, normalize;
    float scale;
    int n_group, topk_group, group_topn;
    int32_t *topk_idx;
    float *topk_w;
    float *aux;                 // may be null
    float *logits;              // [T, E] saved fp32 logits for the backward, may be null
    int32_t *err;
    int num_sms;
    RouterScratch scratch;
};

// Counters of stage 2's fused k-way combine: int32 [T, n_tiles], n_tiles =
// ceil(H / 256) output tiles per row; the metadata sets each to the number of
// the token's dropped slots (cnt may be null: no counters).
struct CombineCounters {
    int32_t *cnt;
    int T, k, n_tiles;
};

struct MetadataLaunch {
    const int32_t *topk_idx;
    int R, E;
    int32_t *counts, *offsets, *mt_prefix, *perm_slot, *row_of, *err;
    int32_t *block_hist;        // [ceil(R / kMetaChunk), E]
    int32_t *ticket;
    CombineCounters combine;
};

// One grouped GEMM launch (forward stages 1 and 2, backward dA / dX / dW2 / dW1).
struct GemmLaunch {
    const uint8_t *bpack;       // stage 1 / 2: tile-packed weights (pack.cu) instead of tm_b, or null
    const int32_t *kpad;        // MXFP8 weight gradients: [E+1] padded row offsets of the quantized operands
    const CUtensorMap *tm_a;    // host-encoded tensor maps (copied into the launch);
    const CUtensorMap *tm_b;    // tm_a, tm_out2 and tm_out3 may be null when unused
    const CUtensorMap *tm_out;
    const CUtensorMap *tm_out2;
    const CUtensorMap *tm_out3;
    const int32_t *counts, *offsets, *mt_prefix, *perm_slot;
    const __nv_bfloat16 *h;     // backward dA: saved pre-activation [R, 2I]
    int32_t *err;
    int32_t *sched;             // [2] unit scheduler of this launch
    const float *topk_w;        // stage 2 and dA
    const int32_t *row_of;      // stage 2 with the fused combine: routed row of each slot
    __nv_bfloat16 *y;           // stage 2 with the fused combine: y [T, H]
    int32_t *ccnt;              // stage 2 with the fused combine: counters [T, ceil(H / 256)], or null
    int T;
    __nv_bfloat16 *out;         // row-grouped output (masked stores of partial slabs)
    __nv_bfloat16 *out2, *out3; // stage 1 with h: h gate / up halves; dA: dH up half, w a
    float *dtw_part;            // dA: [ceil(I / 256), R]
    const CUtensorMap *tm_sfa;  // MXFP8: k-block-major scale words of the A rows, box 132 x 1
    const CUtensorMap *tm_sfb;  // MXFP8: ... of the B rows, box 96 x 1 (stage 1) or 224 x 1
    uint8_t *out_sf;            // stage 1 MXFP8: E8M0 scales of a, k-block-major [I / 128][sf_rows] words
    int64_t sf_rows;            // stage 1 MXFP8: rows of the scale arrays of x and a (T k rounded up to 4)
    int E, k;
    int K;                      // reduction length of the row-grouped modes
    int n_out;                  // output columns
    int n_tile;                 // output columns per unit (128 for stage 1, else 256)
    int m_total;                // weight gradients: output rows per expert
    int b_rows, half;           // stage 1: 2I and I; dA: half = I
    int out_ld;                 // row stride of out / out2 where it differs from n_out
    int R;                      // routed rows (T * k)
    int save_h;                 // stage 1: also store h
    int num_sms;
};

// The router GEMM: partial logits [splits, T, E] of x . w3^T.
struct RouterGemmLaunch {
    const CUtensorMap *tm_x;    // x [T, H], box 64 x 128
    const CUtensorMap *tm_w3;   // w3 [3E, H], box 64 x router_n_mma(E)
    float *logits_part;
    int32_t *err;
    int32_t *sched;
    int T, H, E, splits;
    int num_sms;
};

struct CombineLaunch {
    const __nv_bfloat16 *obuf;
    const int32_t *row_of;
    __nv_bfloat16 *y;
    int T, H, k;
};

cudaError_t launch_router(const RouterLaunch &p, cudaStream_t st);
// The router's selection stage alone, from caller-given fp32 logits [T, E]
// (p.x and p.w_r unused).
cudaError_t launch_route_logits(const RouterLaunch &p, const float *logits, cudaStream_t st);
cudaError_t launch_routing_metadata(const MetadataLaunch &p, cudaStream_t st);
cudaError_t launch_gemm1_swiglu(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_gemm2_scatter(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_router_gemm(const RouterGemmLaunch &p, cudaStream_t st);
// Tile-packed forward weights (pack.cu): tile counts and the packing copies.
int64_t packed_w1_tiles(int64_t E, int64_t H, int64_t I);
int64_t packed_w2_tiles(int64_t E, int64_t H, int64_t I);
cudaError_t launch_pack_w1(const __nv_bfloat16 *w1, int64_t E, int64_t H, int64_t I, void *w1p, cudaStream_t st);
cudaError_t launch_pack_w2(const __nv_bfloat16 *w2, int64_t E, int64_t H, int64_t I, void *w2p, cudaStream_t st);
cudaError_t launch_combine(const CombineLaunch &p, cudaStream_t st);
// The dispatch copy: rows[row_of[s], :] = x[s / k, :] for every slot s with
// row_of[s] >= 0, and with row_w row_w[row_of[s]] = topk_w[s] (rows.cu).
cudaError_t launch_dispatch_rows(const __nv_bfloat16 *x, const int32_t *row_of, int64_t T, int k, int64_t H,
                                 __nv_bfloat16 *rows, const float *topk_w, float *row_w, cudaStream_t st);

// Routing-weight gradient: dtopk_w[s] = sum_n dtw_part[n, row_of[s]] (0 if dropped).
struct DtwReduceLaunch {
    const float *dtw_part;      // [n_part, R]
    int n_part, R, T, k;
    const int32_t *row_of;
    float *dtopk_w;             // [T, k]
};

// Router backward: logit gradient, then dW_r (and the dX term in the combine).
struct RouterBwdLaunch {
    const float *logits;        // [T, E] fp32 logits of the forward (offset included)
    const int32_t *topk_idx;
    const float *topk_w, *dtopk_w;
    int T, H, E, k, score_fn, normalize;
    float scale;
    float *dl;                  // [T, E] logit gradient (output)
    const __nv_bfloat16 *x;     // [T, H]
    const int32_t *offsets, *counts, *perm_slot;
    float *dw_r;                // [E, H] (output)
    float *dwr_part;            // [kDwrSegments, E, H] partial sums (workspace)
};
// Row segments of the dW_r reduction (partial sums per segment, then a fixed-order sum).
constexpr int kDwrSegments = 8;

// dX = sum over the token's slots of the dX rows (routed order) + dlogits . W_r.
struct CombineBwdLaunch {
    const __nv_bfloat16 *xbuf;  // [R, H]
    const int32_t *row_of, *topk_idx;
    const float *dl;            // [T, E] or null (no router term)
    const float *w_r;           // [E, H] or null
    int dense;                  // dl may be non-zero outside the chosen experts
    __nv_bfloat16 *dx;
    int T, H, E, k;
};

// Expert parallelism with fixed-size exchange buffers (ep.cu): P ranks, E_loc
// experts each, C rows per (sender, receiver) block.
struct EpPackLaunch {
    const __nv_bfloat16 *x;
    const float *topk_w;
    const int32_t *row_of, *counts, *offsets;
    int T, k;
    int64_t H;
    int E, E_loc;
    int64_t C;
    __nv_bfloat16 *send_rows;   // [P * C, H]
    float *send_w;              // [P * C]
    int32_t *send_counts;       // [P, E_loc] (= [E])
    int32_t *err;
};
struct EpRecvLaunch {
    const int32_t *recv;        // [P, E_loc] rows received per (source, local expert)
    int P, E_loc;
    int64_t C;
    int n_tiles;                // ceil(H / 256): combine counters per received row
    int32_t *counts, *offsets, *mt_prefix, *perm_slot, *row_of, *ccnt, *err;
};
struct EpCombineLaunch {
    const __nv_bfloat16 *back;  // [P * C, H] returned rows, in the send buffer's places
    const int32_t *row_of, *offsets;
    int T, k, H, E, E_loc;
    int64_t C;
    __nv_bfloat16 *y;
};
cudaError_t launch_ep_pack(const EpPackLaunch &p, cudaStream_t st);
cudaError_t launch_ep_receive_metadata(const EpRecvLaunch &p, cudaStream_t st);
cudaError_t launch_ep_combine(const EpCombineLaunch &p, cudaStream_t st);

cudaError_t launch_dtw_reduce(const DtwReduceLaunch &p, cudaStream_t st);
// Zero rows [*routed_rows, R) of dH [R, 2I] and w a [R, I] (rows of dropped slots).
cudaError_t launch_zero_tail_rows(__nv_bfloat16 *dh, __nv_bfloat16 *aw, const int32_t *routed_rows, int R,
                                  int I, cudaStream_t st);
cudaError_t launch_router_dlogits(const RouterBwdLaunch &p, cudaStream_t st);
cudaError_t launch_router_dwr(const RouterBwdLaunch &p, cudaStream_t st);
cudaError_t launch_combine_bwd(const CombineBwdLaunch &p, cudaStream_t st);

// MXFP8 (grouped_gemm_mx.cu): quantization of a bf16 [rows, cols] matrix along its
// rows (cols % 128 == 0) into E4M3 codes [rows, cols] and E8M0 block scales as
// k-block-major 32-bit words [cols / 128][rows rounded up to 4]; the two MXFP8
// expert stages (stage 1: out = a codes, out_sf = a scales; stage 2 as kStage2).
cudaError_t launch_mx_quantize(const __nv_bfloat16 *in, int64_t rows, int64_t cols, uint8_t *codes,
                               uint8_t *scales, cudaStream_t st);
// The MXFP8 dispatch: quantize each token's x row once into its routed rows
// row_of[t k + j] of codes [R = T k, cols] and of the k-block-major scale words
// [cols / 128][R rounded up to 4] (rows [0, *routed)); sc_tmp holds R * cols / 32
// bytes of row-major scales in between (two launches).
cudaError_t launch_mx_quantize_dispatch(const __nv_bfloat16 *x, const int32_t *row_of, const int32_t *routed, int k,
                                        int64_t T, int64_t cols, uint8_t *codes, uint8_t *scales, uint8_t *sc_tmp,
                                        cudaStream_t st);
// MXFP8 weight gradients: padded row offsets kpad [E+1] of the quantized operands
// (each expert's rows rounded up to whole 128-row k-blocks), the quantization of
// an operand along the routed rows into transposed codes [C, ld] and k-block-major
// scale words [ld / 128, C] (four E8M0 bytes each; rows of routed row q: src[q]
// or, with perm_slot, src[perm_slot[q] / k]), and the block-scaled GEMM.
cudaError_t launch_mx_wgrad_offsets(const int32_t *counts, int E, int32_t *kpad, cudaStream_t st);
cudaError_t launch_mx_quantize_rows_t(const __nv_bfloat16 *src, int64_t src_ld, const int32_t *perm_slot, int k,
                                      const int32_t *counts, const int32_t *offsets, const int32_t *kpad, int E,
                                      int C, int64_t ld, uint8_t *codes, uint8_t *scales, cudaStream_t st);
cudaError_t launch_wgrad_mx(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_gemm1_mx(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_gemm2_mx(const GemmLaunch &p, cudaStream_t st);
cudaError_t setup_mx_gemm_kernels();

// MXFP8 scale words ([k_blocks][rows] 32-bit words, k-block-major; rows a
// multiple of 4), boxes of box_rows words of one k-block, unswizzled.
bool encode_sf_words(CUtensorMap *map, const void *base, uint64_t rows, uint64_t k_blocks, uint32_t box_rows);
// Rows of the k-block-major MXFP8 scale array of a matrix with `rows` rows
// (rounded up to 4, so that each k-block's words start 16-byte aligned).
inline uint64_t mx_rows(uint64_t rows) { return (rows + 3) & ~static_cast<uint64_t>(3); }
// uint8 tensor [rows, inner] (e.g. E4M3 codes) with a box_inner x box_rows box,
// 128-byte swizzle (box_inner = 128).
bool encode_u8_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                  uint32_t box_rows);

// Backward GEMMs (grouped_gemm_bwd.cu).
cudaError_t launch_bwd_da(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_bwd_dx(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_bwd_dw2(const GemmLaunch &p, cudaStream_t st);
cudaError_t launch_bwd_dw1(const GemmLaunch &p, cudaStream_t st);
cudaError_t setup_bwd_gemm_kernels();

// Per-device one-time kernel attribute set-up (dynamic shared memory limits).
cudaError_t setup_metadata_kernels();
cudaError_t setup_gemm_kernels();

// bf16 tensor [rows, inner] (inner contiguous) with a box_inner x box_rows box,
// zero fill out of bounds; the swizzle span equals the box row (64 or 128 bytes). False if the encoder is missing
// or rejects the arguments.
bool encode_bf16_2d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows);

// bf16 tensor [depth, rows, inner] with a box_inner x box_rows x 1 box, zero
// fill out of bounds, 128- or 64-byte swizzle as for encode_bf16_2d.
bool encode_bf16_3d(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows, uint64_t depth,
                    uint32_t box_inner, uint32_t box_rows);

// bf16 2-D view with an explicit row stride (elements): a column slice of a
// wider row-major tensor.
bool encode_bf16_2d_strided(CUtensorMap *map, const void *base, uint64_t inner, uint64_t rows,
                            uint64_t row_stride, uint32_t box_inner, uint32_t box_rows);

// Statistics: kernels launched by this library.
void note_launches(int n);

// Programmatic dependent launch. Every kernel of this library is launched with
// launch_dep, which lets the stream schedule it while the preceding kernel is
// still finishing (its prologue overlaps that kernel's tail), and every kernel
// calls griddep_wait() before it reads or writes memory another kernel touches:
// the wait returns once the preceding grid has completed and its writes are
// visible (at once when there is no programmatic predecessor).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream be scheduled before this one finishes (it
// still waits in griddep_wait); used by the persistent GEMM, whose CTAs are all
// resident from the start.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_dep(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace moe
