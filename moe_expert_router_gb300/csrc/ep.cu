// ep.cu -- the device halves of an expert-parallel exchange with fixed-size
// buffers (MegaMoE guide, opening section: dispatch_grouped_gemm fuses the
// dispatch all-to-all, grouped_gemm_combine the combine all-to-all; section
// "Example 2" runs the layer under a full CUDA graph, so nothing in a step may
// wait for the host).
//
// With P ranks, rank q owning experts [q E_loc, (q + 1) E_loc), every rank
// sends each peer a block of `capacity` rows (C), whatever its routing: the
// collective then needs no split sizes, so the per-expert counts never reach
// the host. Block q of the send buffer holds the sender's routed rows of rank
// q's experts in routed order (expert-major), from position 0; rows past C are
// dropped and flag MOE_DEVERR_CAPACITY (C = T k never drops). The receiver's
// rows are P blocks of C; its routing metadata follows from the exchanged
// counts alone. After the expert path the receiver returns one output row per
// received row, at the same place, and the sender sums each token's rows.
#include "internal.cuh"

namespace moe {

namespace {

// Expert of routed row r: the largest e with offsets[e] <= r (empty experts
// share their offset with the next one).
__device__ __forceinline__ int expert_of_row(const int32_t *__restrict__ offsets, int E, int r) {
    int lo = 0, hi = E;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(&offsets[mid]) <= r) lo = mid; else hi = mid;
    }
    return lo;
}

// Place of routed row r in the send buffer: q * C + (r - offsets[q E_loc]),
// or -1 past the block's capacity.
__device__ __forceinline__ int64_t send_place(const int32_t *__restrict__ offsets, int E, int E_loc, int64_t C,
                                              int r) {
    const int q = expert_of_row(offsets, E, r) / E_loc;
    const int64_t pos = r - __ldg(&offsets[q * E_loc]);
    return pos < C ? q * C + pos : -1;
}

// Send buffer of the dispatch: one warp per token (its row read once), each of
// its routed rows copied to its place, with the slot's routing weight. Block 0
// also writes the per-(rank, local expert) counts of the rows that fit.
__global__ void __launch_bounds__(256)
ep_pack_kernel(const __nv_bfloat16 *__restrict__ x, const float *__restrict__ topk_w,
               const int32_t *__restrict__ row_of, const int32_t *__restrict__ counts,
               const int32_t *__restrict__ offsets, int T, int k, int64_t H, int E, int E_loc, int64_t C,
               __nv_bfloat16 *__restrict__ send_rows, float *__restrict__ send_w, int32_t *__restrict__ send_counts,
               int32_t *__restrict__ err) {
    griddep_wait();
    if (blockIdx.x == 0) {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int64_t first = offsets[e] - offsets[(e / E_loc) * E_loc];   // position of e's first row
            const int64_t fit = C - first;
            send_counts[e] = static_cast<int32_t>(fit <= 0 ? 0 : (fit < counts[e] ? fit : counts[e]));
        }
    }
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int chunks = static_cast<int>(H / 8);
    for (int64_t t = blockIdx.x * static_cast<int64_t>(blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const int r = lane < k ? __ldg(&row_of[t * k + lane]) : -1;
        const int64_t place = r >= 0 ? send_place(offsets, E, E_loc, C, r) : -1;
        if (r >= 0 && place < 0) atomicOr(err, MOE_DEVERR_CAPACITY);
        if (place >= 0) send_w[place] = topk_w[t * k + lane];
        const uint4 *src = reinterpret_cast<const uint4 *>(x + t * H);
        for (int cb = 0; cb < chunks; cb += 256) {
            const int c0 = cb + lane;
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                v[j] = (c0 + 32 * j < chunks) ? __ldg(src + c0 + 32 * j) : make_uint4(0u, 0u, 0u, 0u);
            for (int j2 = 0; j2 < k; ++j2) {
                const int64_t pl = __shfl_sync(0xffffffffu, place, j2);
                if (pl < 0) continue;
                uint4 *dst = reinterpret_cast<uint4 *>(send_rows + pl * H);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (c0 + 32 * j < chunks) dst[c0 + 32 * j] = v[j];
            }
        }
    }
}

// Receiver, step 1: every received slot empty (row_of = -1) and its combine
// counters at 1 (its k = 1 slot dropped), until step 3 fills the live ones.
__global__ void __launch_bounds__(256)
ep_recv_init_kernel(int64_t slots, int n_tiles, int32_t *__restrict__ row_of, int32_t *__restrict__ ccnt) {
    griddep_wait();
    for (int64_t s = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; s < slots;
         s += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        row_of[s] = -1;
        for (int n = 0; n < n_tiles; ++n) ccnt[s * n_tiles + n] = 1;
    }
}

// Receiver, step 2 (one CTA): per local expert the rows of all sources,
// counts[e] = sum_p recv[p][e], their exclusive prefix and the 256-row tile
// prefix. A source block holding more than C rows flags the error word (its
// rows past C are not there).
__global__ void __launch_bounds__(1024)
ep_recv_counts_kernel(const int32_t *__restrict__ recv, int P, int E_loc, int64_t C, int32_t *__restrict__ counts,
                      int32_t *__restrict__ offsets, int32_t *__restrict__ mt_prefix, int32_t *__restrict__ err) {
    griddep_wait();
    __shared__ int32_t s_cnt[1024], s_mt[1024];
    __shared__ int32_t s_over;
    if (threadIdx.x == 0) s_over = 0;
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        int64_t n = 0;
        for (int e = 0; e < E_loc; ++e) n += recv[static_cast<int64_t>(p) * E_loc + e];
        if (n > C) atomicOr(&s_over, 1);
    }
    const int e = threadIdx.x;
    int c = 0;
    if (e < E_loc)
        for (int p = 0; p < P; ++p) {
            const int v = recv[static_cast<int64_t>(p) * E_loc + e];
            c += v > 0 ? v : 0;
        }
    s_cnt[e] = e < E_loc ? c : 0;
    s_mt[e] = e < E_loc ? (c + kUnitM - 1) / kUnitM : 0;
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0, mrun = 0;
        for (int i = 0; i < E_loc; ++i) {
            counts[i] = s_cnt[i];
            offsets[i] = run;
            mt_prefix[i] = mrun;
            run += s_cnt[i];
            mrun += s_mt[i];
        }
        offsets[E_loc] = run;
        mt_prefix[E_loc] = mrun;
        if (s_over) atomicOr(err, MOE_DEVERR_CAPACITY);
    }
}

// Receiver, step 3: one CTA per (source p, local expert e). Source p's rows of
// expert e sit in its block at [pref, pref + n), pref = sum_{e' < e} recv[p][e'];
// they take the routed rows offsets[e] + base .. + n, base = sum_{p' < p}
// recv[p'][e]: expert-major, then source, then position -- increasing slot
// order p C + i within each expert, the order moe_routing_metadata gives.
__global__ void __launch_bounds__(256)
ep_recv_place_kernel(const int32_t *__restrict__ recv, int P, int E_loc, int64_t C,
                     const int32_t *__restrict__ offsets, int n_tiles, int32_t *__restrict__ perm_slot,
                     int32_t *__restrict__ row_of, int32_t *__restrict__ ccnt) {
    griddep_wait();
    __shared__ int64_t s_pref, s_base;
    const int p = blockIdx.x / E_loc, e = blockIdx.x % E_loc;
    if (threadIdx.x < 32) {
        int64_t pref = 0, base = 0;
        for (int i = threadIdx.x; i < e; i += 32) pref += max(0, recv[static_cast<int64_t>(p) * E_loc + i]);
        for (int i = threadIdx.x; i < p; i += 32) base += max(0, recv[static_cast<int64_t>(i) * E_loc + e]);
#pragma unroll
        for (int d = 16; d > 0; d >>= 1) {
            pref += __shfl_xor_sync(0xffffffffu, pref, d);
            base += __shfl_xor_sync(0xffffffffu, base, d);
        }
        if (threadIdx.x == 0) {
            s_pref = pref;
            s_base = base;
        }
    }
    __syncthreads();
    const int64_t n = max(0, recv[static_cast<int64_t>(p) * E_loc + e]);
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
        if (s_pref + i >= C) break;                        // not in the block (flagged in step 2)
        const int64_t slot = static_cast<int64_t>(p) * C + s_pref + i;
        const int64_t r = offsets[e] + s_base + i;
        perm_slot[r] = static_cast<int32_t>(slot);
        row_of[slot] = static_cast<int32_t>(r);
        for (int t = 0; t < n_tiles; ++t) ccnt[slot * n_tiles + t] = 0;
    }
}

// Sender's combine of the returned rows: y[t] = sum over the token's slots of
// back[place of its routed row] (fp32, slot order, bf16 once); slots dropped by
// the routing or by the capacity add nothing. One warp per token.
__global__ void __launch_bounds__(256)
ep_combine_kernel(const __nv_bfloat16 *__restrict__ back, const int32_t *__restrict__ row_of,
                  const int32_t *__restrict__ offsets, int T, int k, int H, int E, int E_loc, int64_t C,
                  __nv_bfloat16 *__restrict__ y) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int groups = H >> 3;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const int r = lane < k ? __ldg(&row_of[static_cast<int64_t>(t) * k + lane]) : -1;
        const int64_t my_place = r >= 0 ? send_place(offsets, E, E_loc, C, r) : -1;
        for (int g0 = 0; g0 < groups; g0 += 32) {
            const int g = g0 + lane;
            const bool live = g < groups;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j = 0; j < k; ++j) {
                const int64_t pl = __shfl_sync(0xffffffffu, my_place, j);
                const uint4 v = (live && pl >= 0) ? __ldg(reinterpret_cast<const uint4 *>(back + pl * H) + g)
                                                  : make_uint4(0u, 0u, 0u, 0u);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[2 * q] += __uint_as_float(w[q] << 16);
                    acc[2 * q + 1] += __uint_as_float(w[q] & 0xffff0000u);
                }
            }
            if (live) {
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
                    o[q] = *reinterpret_cast<const uint32_t *>(&b);
                }
                reinterpret_cast<uint4 *>(y + static_cast<int64_t>(t) * H)[g] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

int grid_for(int64_t items, int per_block) {
    int64_t g = (items + per_block - 1) / per_block;
    if (g > 152 * 8) g = 152 * 8;
    return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_ep_pack(const EpPackLaunch &p, cudaStream_t st) {
    const cudaError_t e = launch_dep(ep_pack_kernel, dim3(grid_for(p.T, 8)), dim3(256), 0, st, p.x, p.topk_w,
                                     p.row_of, p.counts, p.offsets, p.T, p.k, p.H, p.E, p.E_loc, p.C, p.send_rows,
                                     p.send_w, p.send_counts, p.err);
    note_launches(1);
    return e;
}

cudaError_t launch_ep_receive_metadata(const EpRecvLaunch &p, cudaStream_t st) {
    const int64_t slots = static_cast<int64_t>(p.P) * p.C;
    cudaError_t e = launch_dep(ep_recv_init_kernel, dim3(grid_for(slots, 256)), dim3(256), 0, st, slots, p.n_tiles,
                               p.row_of, p.ccnt);
    if (e == cudaSuccess)
        e = launch_dep(ep_recv_counts_kernel, dim3(1), dim3(1024), 0, st, p.recv, p.P, p.E_loc, p.C, p.counts,
                       p.offsets, p.mt_prefix, p.err);
    if (e == cudaSuccess)
        e = launch_dep(ep_recv_place_kernel, dim3(p.P * p.E_loc), dim3(256), 0, st, p.recv, p.P, p.E_loc, p.C,
                       p.offsets, p.n_tiles, p.perm_slot, p.row_of, p.ccnt);
    note_launches(3);
    return e;
}

cudaError_t launch_ep_combine(const EpCombineLaunch &p, cudaStream_t st) {
    const cudaError_t e = launch_dep(ep_combine_kernel, dim3(grid_for(p.T, 8)), dim3(256), 0, st, p.back, p.row_of,
                                     p.offsets, p.T, p.k, p.H, p.E, p.E_loc, p.C, p.y);
    note_launches(1);
    return e;
}

}  // namespace moe
