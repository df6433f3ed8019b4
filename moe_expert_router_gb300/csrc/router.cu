// router.cu -- the fused router of the MegaMoE layer (MegaMoE guide, opening
// section: score function + group-limited top-k + aux score; the aux
// load-balance value is computed on the device and returned).
//
//   split kernel  : w_r (fp32) -> w3 = [hi; mid; lo] (bf16) with
//                   w_r = hi + mid + lo exactly; block 0 also clears the aux
//                   accumulators of this call.
//   router GEMM   : partial logits [splits, T, E] = x . w3^T on the tensor
//                   cores (grouped_gemm.cu, router mode). x is bf16, so each
//                   product is exact and the fp32 accumulation matches an
//                   fp32 dot product of x with w_r.
//   top-k kernel  : one warp per token. Logits = fixed-order sum of the split
//                   partials (+ logit_offset). Scores (softmax over the row, or
//                   elementwise sigmoid), selection scores sel = s + sel_bias,
//                   optional group limit (group score = sum of the group_topn
//                   best sel; keep topk_group groups), k rounds of a warp
//                   arg-max over (sel desc, expert index asc), weights s / sum
//                   * scale. Per-block partial sums of s and of the chosen
//                   experts go to global accumulators; the last block to
//                   finish computes aux = E * sum_e (c_e / (T k)) * P_e.
#include <math.h>

#include "internal.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kTopkWarps = 8;
constexpr int kTopkFastSplits = 4;          // split counts the top-k loads all at once
constexpr int kMaxE = 1024;

__global__ void __launch_bounds__(256)
router_split_kernel(const float *__restrict__ w_r, __nv_bfloat16 *__restrict__ w3, int64_t n,
                    int E, float *__restrict__ score_sum, int32_t *__restrict__ counts,
                    int32_t *__restrict__ ticket) {
    griddep_wait();
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            score_sum[e] = 0.0f;
            counts[e] = 0;
        }
        if (threadIdx.x == 0) *ticket = 0;
    }
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float w = w_r[i];
        const __nv_bfloat16 hi = __float2bfloat16_rn(w);
        const float r1 = w - __bfloat162float(hi);          // exact
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(mid);        // exact, <= 8 significant bits
        w3[i] = hi;
        w3[n + i] = mid;
        w3[2 * n + i] = __float2bfloat16_rn(r2);
    }
}

// Router logits for few tokens, on the CUDA cores: logits[t, e] = sum_h x[t, h] w_r[e, h]
// in fp32 (x is bf16: each product is exact but for one fp32 rounding). With few
// tokens the tensor-core path is all latency (a split kernel, a split-K GEMM whose
// units hold a mostly empty 128-row tile, and its partials); here one warp takes one
// expert and a group of kSmallTok tokens, each lane accumulates columns 8 lane +
// 256 j of those tokens, and the warp sums its lanes in a fixed butterfly order.
// Block 0 also clears the aux accumulators of this call, as the split kernel does on
// the tensor-core path.
constexpr int kSmallTok = 2;
constexpr int kSmallMaxT = 256;

__global__ void __launch_bounds__(256)
router_logits_small_kernel(const __nv_bfloat16 *__restrict__ x, const float *__restrict__ w_r, int T, int H, int E,
                           float *__restrict__ logits, float *__restrict__ score_sum, int32_t *__restrict__ counts,
                           int32_t *__restrict__ ticket) {
    griddep_wait();
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            score_sum[e] = 0.0f;
            counts[e] = 0;
        }
        if (threadIdx.x == 0) *ticket = 0;
    }
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int tgroups = (T + kSmallTok - 1) / kSmallTok;
    if (gw >= E * tgroups) return;                  // whole warp
    const int e = gw / tgroups;
    const int t0 = (gw - e * tgroups) * kSmallTok;
    const float *wrow = w_r + static_cast<int64_t>(e) * H;
    float acc[kSmallTok];
#pragma unroll
    for (int j = 0; j < kSmallTok; ++j) acc[j] = 0.0f;
#pragma unroll 8
    for (int h = lane * 8; h < H; h += 256) {
        const float4 w0 = __ldg(reinterpret_cast<const float4 *>(wrow + h));
        const float4 w1 = __ldg(reinterpret_cast<const float4 *>(wrow + h + 4));
#pragma unroll
        for (int j = 0; j < kSmallTok; ++j) {
            if (t0 + j < T) {
                const uint4 xv = __ldg(reinterpret_cast<const uint4 *>(x + static_cast<int64_t>(t0 + j) * H + h));
                float a = acc[j];
                a = fmaf(__uint_as_float(xv.x << 16), w0.x, a);
                a = fmaf(__uint_as_float(xv.x & 0xffff0000u), w0.y, a);
                a = fmaf(__uint_as_float(xv.y << 16), w0.z, a);
                a = fmaf(__uint_as_float(xv.y & 0xffff0000u), w0.w, a);
                a = fmaf(__uint_as_float(xv.z << 16), w1.x, a);
                a = fmaf(__uint_as_float(xv.z & 0xffff0000u), w1.y, a);
                a = fmaf(__uint_as_float(xv.w << 16), w1.z, a);
                a = fmaf(__uint_as_float(xv.w & 0xffff0000u), w1.w, a);
                acc[j] = a;
            }
        }
    }
#pragma unroll
    for (int j = 0; j < kSmallTok; ++j) {
        float v = acc[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
        if (lane == 0 && t0 + j < T) logits[static_cast<int64_t>(t0 + j) * E + e] = v;
    }
}

// Warp-wide arg-max in the order (value desc, index asc); every lane gets the winner.
__device__ __forceinline__ void warp_argmax(float &v, int &i) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, v, off);
        const int oi = __shfl_xor_sync(0xffffffffu, i, off);
        if (ov > v || (ov == v && oi < i)) {
            v = ov;
            i = oi;
        }
    }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
}

struct TopkArgs {
    const float *logits_part;   // [splits, T, E]
    int splits;
    const float *logit_offset;
    const float *sel_bias;
    int T, E, k, score_fn, normalize;
    float scale;
    int n_group, topk_group, group_topn;
    int32_t *topk_idx;
    float *topk_w;
    float *score_sum;
    int32_t *counts;
    int32_t *ticket;
    float *aux;
    float *logits_out;          // [T, E] fp32 logits (offset included) or null
};

// V = experts per lane (lane l holds experts l, l+32, ..., l+32(V-1)).
template <int V>
__global__ void __launch_bounds__(kTopkWarps * 32)
router_topk_kernel(const TopkArgs p) {
    griddep_wait();
    __shared__ float blk_sum[kMaxE];
    __shared__ int blk_cnt[kMaxE];
    __shared__ float sel_sh[kTopkWarps][kMaxE];
    __shared__ int is_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        blk_sum[e] = 0.0f;
        blk_cnt[e] = 0;
    }
    __syncthreads();

    const int t = blockIdx.x * kTopkWarps + warp;
    if (t < p.T) {
        float s[V], sel[V];
        bool elig[V];
        const int64_t split_stride = static_cast<int64_t>(p.T) * p.E;
        const float *lrow = p.logits_part + static_cast<int64_t>(t) * p.E;
        // each logit is the sum of its split partials in split order
        bool loaded = false;
        if constexpr (V <= 8) {
            if (p.splits <= kTopkFastSplits) {
            // every partial of the lane's experts in flight at once
            float part[V][kTopkFastSplits];
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int e = lane + 32 * i;
#pragma unroll
                for (int j = 0; j < kTopkFastSplits; ++j)
                    part[i][j] = (e < p.E && j < p.splits) ? __ldcg(&lrow[j * split_stride + e]) : 0.0f;
            }
#pragma unroll
            for (int i = 0; i < V; ++i) {
                float l = 0.0f;
#pragma unroll
                for (int j = 0; j < kTopkFastSplits; ++j)
                    if (j < p.splits) l += part[i][j];
                s[i] = l;
            }
            loaded = true;
            }
        }
        if (!loaded) {
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int e = lane + 32 * i;
                float l = 0.0f;
                if (e < p.E) {
                    // eight loads in flight at a time
                    for (int sp0 = 0; sp0 < p.splits; sp0 += 8) {
                        float part[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            part[j] = (sp0 + j < p.splits) ? __ldcg(&lrow[(sp0 + j) * split_stride + e]) : 0.0f;
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            if (sp0 + j < p.splits) l += part[j];
                    }
                }
                s[i] = l;
            }
        }
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int e = lane + 32 * i;
            if (e < p.E) {
                if (p.logit_offset) s[i] += p.logit_offset[e];
                if (p.logits_out) p.logits_out[static_cast<int64_t>(t) * p.E + e] = s[i];
            } else {
                s[i] = -INFINITY;
            }
        }
        if (p.score_fn == MOE_SCORE_SOFTMAX) {
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < V; ++i) m = fmaxf(m, s[i]);
            m = warp_max(m);
            float z = 0.0f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int e = lane + 32 * i;
                s[i] = (e < p.E) ? expf(s[i] - m) : 0.0f;
                z += s[i];
            }
            z = warp_sum(z);
            const float inv = 1.0f / z;
#pragma unroll
            for (int i = 0; i < V; ++i) s[i] *= inv;
        } else {
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int e = lane + 32 * i;
                s[i] = (e < p.E) ? 1.0f / (1.0f + expf(-s[i])) : 0.0f;
            }
        }
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int e = lane + 32 * i;
            elig[i] = e < p.E;
            sel[i] = elig[i] ? s[i] + (p.sel_bias ? p.sel_bias[e] : 0.0f) : -INFINITY;
            if (elig[i]) atomicAdd(&blk_sum[e], s[i]);
        }

        if (p.n_group > 1 && p.E == 32 * p.n_group && p.group_topn <= 2) {
            // groups of 32 experts: group g is register g across the warp's lanes, so
            // each group's sum of its best group_topn (1 or 2) sel values is a warp
            // reduction of the top two; lane g keeps group g's sum
            float gscore = -INFINITY;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                if (i < p.n_group) {
                    float a1 = sel[i], a2 = -INFINITY;        // the best two seen (a1 >= a2)
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) {
                        const float b1 = __shfl_xor_sync(0xffffffffu, a1, off);
                        const float b2 = __shfl_xor_sync(0xffffffffu, a2, off);
                        const float hi = fmaxf(a1, b1);
                        a2 = fmaxf(fminf(a1, b1), fmaxf(a2, b2));
                        a1 = hi;
                    }
                    const float sum = p.group_topn == 1 ? a1 : a1 + a2;
                    if (lane == i) gscore = sum;
                }
            }
            unsigned kept = 0;
            float gv = gscore;
            for (int n = 0; n < p.topk_group; ++n) {
                float v = gv;
                int i = (lane < p.n_group) ? lane : 0x7fffffff;
                warp_argmax(v, i);
                kept |= 1u << i;
                if (lane == i) gv = -INFINITY;
            }
#pragma unroll
            for (int i = 0; i < V; ++i)
                if (!((kept >> i) & 1u)) elig[i] = false;
        } else if (p.n_group > 1) {
            const int gs = p.E / p.n_group;
            float *row = sel_sh[warp];
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int e = lane + 32 * i;
                if (e < p.E) row[e] = sel[i];
            }
            __syncwarp();
            // lane g: sum of the group_topn best sel of group g, taken in the
            // order (value desc, index asc) by repeatedly finding the best
            // element ranked after the previous pick
            float gscore = -INFINITY;
            if (lane < p.n_group) {
                float prev_v = INFINITY;
                int prev_i = -1;
                float sum = 0.0f;
                for (int n = 0; n < p.group_topn && n < gs; ++n) {
                    float bv = -INFINITY;
                    int bi = -1;
                    for (int i = 0; i < gs; ++i) {
                        const float v = row[lane * gs + i];
                        const bool after = (v < prev_v) || (v == prev_v && i > prev_i);
                        if (after && (bi < 0 || v > bv)) {
                            bv = v;
                            bi = i;
                        }
                    }
                    sum += bv;
                    prev_v = bv;
                    prev_i = bi;
                }
                gscore = sum;
            }
            unsigned kept = 0;
            float gv = gscore;
            for (int n = 0; n < p.topk_group; ++n) {
                float v = gv;
                int i = (lane < p.n_group) ? lane : 0x7fffffff;
                warp_argmax(v, i);
                kept |= 1u << i;
                if (lane == i) gv = -INFINITY;
            }
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int e = lane + 32 * i;
                if (e < p.E && !((kept >> (e / gs)) & 1u)) elig[i] = false;
            }
        }

        int my_idx = 0;
        float my_s = 0.0f, chosen_sum = 0.0f;
        for (int j = 0; j < p.k; ++j) {
            float v = -INFINITY;
            int idx = 0x7fffffff;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                const int e = lane + 32 * i;
                if (elig[i] && (idx == 0x7fffffff || sel[i] > v)) {
                    v = sel[i];
                    idx = e;
                }
            }
            warp_argmax(v, idx);
            float mine = 0.0f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                if (lane + 32 * i == idx) {
                    elig[i] = false;
                    mine = s[i];
                }
            }
            const float sc = __shfl_sync(0xffffffffu, mine, idx & 31);
            chosen_sum += sc;
            if (lane == j) {
                my_idx = idx;
                my_s = sc;
            }
            if (lane == 0) atomicAdd(&blk_cnt[idx], 1);
        }
        if (lane < p.k) {
            float w = my_s;
            if (p.normalize) w = w / chosen_sum;
            w *= p.scale;
            p.topk_idx[static_cast<int64_t>(t) * p.k + lane] = my_idx;
            p.topk_w[static_cast<int64_t>(t) * p.k + lane] = w;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < p.E; e += blockDim.x) {
        if (blk_sum[e] != 0.0f) atomicAdd(&p.score_sum[e], blk_sum[e]);
        if (blk_cnt[e] != 0) atomicAdd(&p.counts[e], blk_cnt[e]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = (atomicAdd(p.ticket, 1) == static_cast<int>(gridDim.x) - 1);
    __syncthreads();
    if (is_last && p.aux != nullptr) {
        __threadfence();
        float part = 0.0f;
        for (int e = threadIdx.x; e < p.E; e += blockDim.x)
            part += static_cast<float>(__ldcg(&p.counts[e])) * __ldcg(&p.score_sum[e]);
        part = warp_sum(part);
        __shared__ float red[kTopkWarps];
        if (lane == 0) red[warp] = part;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.0f;
            for (int w = 0; w < kTopkWarps; ++w) tot += red[w];
            const float Tf = static_cast<float>(p.T);
            *p.aux = static_cast<float>(p.E) * tot / (Tf * static_cast<float>(p.k) * Tf);
        }
    }
}

template <int V>
cudaError_t launch_topk(const TopkArgs &a, int blocks, cudaStream_t st) {
    return launch_dep(router_topk_kernel<V>, dim3(blocks), dim3(kTopkWarps * 32), 0, st, a);
}

}  // namespace

namespace {

// Selection, weights and aux from fp32 logits: `logits` holds `splits` partial
// logit arrays [splits, T, E] that are summed in order.
cudaError_t launch_selection(const RouterLaunch &p, const float *logits, int splits, cudaStream_t st) {
    const RouterScratch &sc = p.scratch;
    TopkArgs a;
    a.logits_part = logits;
    a.splits = splits;
    a.logit_offset = p.logit_offset;
    a.sel_bias = p.sel_bias;
    a.T = p.T;
    a.E = p.E;
    a.k = p.k;
    a.score_fn = p.score_fn;
    a.normalize = p.normalize;
    a.scale = p.scale;
    a.n_group = p.n_group;
    a.topk_group = p.topk_group;
    a.group_topn = p.group_topn;
    a.topk_idx = p.topk_idx;
    a.topk_w = p.topk_w;
    a.score_sum = sc.score_sum;
    a.counts = sc.counts;
    a.ticket = sc.ticket;
    a.aux = p.aux;
    a.logits_out = p.logits;
    const int blocks = (p.T + kTopkWarps - 1) / kTopkWarps;
    const int v = (p.E + 31) / 32;
    cudaError_t e;
    if (v <= 2) e = launch_topk<2>(a, blocks, st);
    else if (v <= 4) e = launch_topk<4>(a, blocks, st);
    else if (v <= 8) e = launch_topk<8>(a, blocks, st);
    else if (v <= 16) e = launch_topk<16>(a, blocks, st);
    else e = launch_topk<32>(a, blocks, st);
    note_launches(1);
    return e;
}

}  // namespace

cudaError_t launch_router(const RouterLaunch &p, cudaStream_t st) {
    const RouterScratch &sc = p.scratch;
    if (p.T <= kSmallMaxT) {
        // few tokens: fp32 logits on the CUDA cores into the first partial, then the selection
        const int64_t warps = static_cast<int64_t>(p.E) * ((p.T + kSmallTok - 1) / kSmallTok);
        const cudaError_t e = launch_dep(router_logits_small_kernel, dim3(static_cast<int>((warps + 7) / 8)), dim3(256),
                                         0, st, p.x, p.w_r, p.T, p.H, p.E, sc.logits_part, sc.score_sum, sc.counts,
                                         sc.ticket);
        note_launches(1);
        if (e != cudaSuccess) return e;
        return launch_selection(p, sc.logits_part, 1, st);
    }
    const int64_t n = static_cast<int64_t>(p.E) * p.H;
    int64_t sblocks = (n + 255) / 256;
    if (sblocks > 152 * 8) sblocks = 152 * 8;
    cudaError_t err = launch_dep(router_split_kernel, dim3(static_cast<int>(sblocks)), dim3(256), 0, st, p.w_r, sc.w3,
                                 n, p.E, sc.score_sum, sc.counts, sc.ticket);
    note_launches(1);
    if (err != cudaSuccess) return err;

    CUtensorMap tm_x, tm_w3;
    if (!encode_bf16_2d(&tm_x, p.x, p.H, p.T, kBK, kBM) ||
        !encode_bf16_2d(&tm_w3, sc.w3, p.H, 3 * static_cast<uint64_t>(p.E), kBK,
                        static_cast<uint32_t>(router_n_mma(p.E))))
        return cudaErrorInvalidValue;
    RouterGemmLaunch g;
    g.tm_x = &tm_x;
    g.tm_w3 = &tm_w3;
    g.logits_part = sc.logits_part;
    g.err = p.err;
    g.sched = sc.sched;
    g.T = p.T;
    g.H = p.H;
    g.E = p.E;
    g.splits = sc.splits;
    g.num_sms = p.num_sms;
    if ((err = launch_router_gemm(g, st)) != cudaSuccess) return err;
    return launch_selection(p, sc.logits_part, sc.splits, st);
}

cudaError_t launch_route_logits(const RouterLaunch &p, const float *logits, cudaStream_t st) {
    const RouterScratch &sc = p.scratch;
    // one block of the split kernel with nothing to split: it clears the aux accumulators
    cudaError_t err = launch_dep(router_split_kernel, dim3(1), dim3(256), 0, st, static_cast<const float *>(nullptr),
                                 static_cast<__nv_bfloat16 *>(nullptr), static_cast<int64_t>(0), p.E, sc.score_sum,
                                 sc.counts, sc.ticket);
    note_launches(1);
    if (err != cudaSuccess) return err;
    return launch_selection(p, logits, 1, st);
}

}  // namespace moe
