// routing.cu -- routing metadata: the single-device stand-in for the dispatch
// all-to-all of dispatch_grouped_gemm (MegaMoE guide, opening section).
//
// From topk_idx [T*k] it builds, entirely on the device (no host sync, so the
// ragged, step-varying counts the guide's "Router force load balancing"
// section talks about never reach the host):
//   counts[e], offsets[e] (exclusive prefix), mt_prefix[e] (prefix of row
//   tiles ceil(counts/256)), perm_slot[r] (flat slot of routed row r, stable:
//   increasing slot order inside each expert) and row_of[s] (inverse, -1 for a
//   dropped slot).
//
// Two kernels over chunks of kChunk consecutive slots (one CTA per chunk; each
// lane loads its slots' expert indices up front, so a warp pays one memory
// latency per kernel):
//   count : per-chunk expert histogram (warp __match_any + shared atomics),
//           stored as block_hist[chunk][e]. The last CTA to finish (ticket)
//           turns the histograms into per-(chunk, expert) starting rows, the
//           counts, offsets and the row-tile prefix.
//   place : each warp of a chunk counts its own contiguous sub-range, the CTA
//           turns those into per-warp starting ranks, and the warp walks its
//           sub-range again in slot order, giving every slot its row.
// Chunks, warps and lanes all walk slots in increasing order, so the
// permutation is stable without a sort.
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kChunk = kMetaChunk;       // slots per CTA
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kWarpSlots = kChunk / kWarps;
constexpr int kPerLane = kWarpSlots / 32;   // slots s = beg + 32 i + lane of a lane
static_assert(kWarpSlots % 32 == 0, "whole warp passes");

// The expert index of each of this lane's slots (-1 past the end).
__device__ __forceinline__ void load_lane_slots(const int32_t *__restrict__ topk_idx, int beg, int end, int lane,
                                                int (&ev)[kPerLane]) {
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int s = beg + 32 * i + lane;
        ev[i] = (s < end) ? __ldg(&topk_idx[s]) : -1;
    }
}

// The count kernel's work for chunk `chunk`, with hist = E ints of shared memory.
__device__ __forceinline__ void metadata_count_body(const int32_t *__restrict__ topk_idx, int R, int E, int n_chunks,
                                                    int chunk, int32_t *__restrict__ block_hist,
                                                    int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                                    int32_t *__restrict__ mt_prefix, int32_t *__restrict__ ticket,
                                                    int32_t *__restrict__ err, int32_t *hist) {
    __shared__ int is_last;
    __shared__ int32_t warp_tot_c[32], warp_tot_m[32];
    for (int e = threadIdx.x; e < E; e += kThreads) hist[e] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int beg = chunk * kChunk + warp * kWarpSlots;
    const int end = min(R, beg + kWarpSlots);
    int bad = 0;
    int ev[kPerLane];
    load_lane_slots(topk_idx, beg, end, lane, ev);
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int s = beg + 32 * i + lane;
        const int e = ev[i];
        const bool valid = (s < end) && e >= 0 && e < E;
        bad |= (s < end) && !valid;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        if (valid && lane == __ffs(peers) - 1) atomicAdd(&hist[e], __popc(peers));
    }
    if (bad) atomicOr(err, MOE_DEVERR_BAD_EXPERT_INDEX);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) block_hist[static_cast<int64_t>(chunk) * E + e] = hist[e];
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) is_last = (atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1);
    __syncthreads();
    if (!is_last) return;
    __threadfence();

    // last CTA: per expert, running total over chunks (chunk order = slot order),
    // eight chunks' histograms loaded before they are replaced by starting rows
    constexpr int kBatch = 8;
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int run = 0;
        for (int b0 = 0; b0 < n_chunks; b0 += kBatch) {
            int c[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                c[j] = (b0 + j < n_chunks) ? __ldcg(&block_hist[static_cast<int64_t>(b0 + j) * E + e]) : 0;
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                if (b0 + j < n_chunks) block_hist[static_cast<int64_t>(b0 + j) * E + e] = run;
                run += c[j];
            }
        }
        hist[e] = run;                    // counts
    }
    __syncthreads();
    // exclusive scans over experts of counts and of 256-row tiles, kThreads per pass
    int carry_c = 0, carry_m = 0;
    for (int e0 = 0; e0 < E; e0 += kThreads) {
        const int e = e0 + threadIdx.x;
        const int c = (e < E) ? hist[e] : 0;
        const int m = (c + kUnitM - 1) / kUnitM;
        int ic = c, im = m;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int yc = __shfl_up_sync(0xffffffffu, ic, off);
            const int ym = __shfl_up_sync(0xffffffffu, im, off);
            if (lane >= off) { ic += yc; im += ym; }
        }
        if (lane == 31) { warp_tot_c[warp] = ic; warp_tot_m[warp] = im; }
        __syncthreads();
        if (warp == 0) {
            int vc = lane < kWarps ? warp_tot_c[lane] : 0, vm = lane < kWarps ? warp_tot_m[lane] : 0;
            const int oc = vc, om = vm;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int yc = __shfl_up_sync(0xffffffffu, vc, off);
                const int ym = __shfl_up_sync(0xffffffffu, vm, off);
                if (lane >= off) { vc += yc; vm += ym; }
            }
            if (lane < kWarps) { warp_tot_c[lane] = vc - oc; warp_tot_m[lane] = vm - om; }
        }
        __syncthreads();
        const int ex_c = carry_c + ic - c + warp_tot_c[warp];
        const int ex_m = carry_m + im - m + warp_tot_m[warp];
        if (e < E) {
            counts[e] = c;
            offsets[e] = ex_c;
            mt_prefix[e] = ex_m;
            if (e == E - 1) {
                offsets[E] = ex_c + c;
                mt_prefix[E] = ex_m + m;
            }
        }
        // carry the pass total to the next pass
        __syncthreads();
        if (threadIdx.x == kThreads - 1) { warp_tot_c[31] = ex_c + c; warp_tot_m[31] = ex_m + m; }
        __syncthreads();
        carry_c = warp_tot_c[31];
        carry_m = warp_tot_m[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) *ticket = 0;   // ready for the next launch
}

__global__ void __launch_bounds__(kThreads)
metadata_count_kernel(const int32_t *__restrict__ topk_idx, int R, int E, int n_chunks,
                      int32_t *__restrict__ block_hist, int32_t *__restrict__ counts,
                      int32_t *__restrict__ offsets, int32_t *__restrict__ mt_prefix,
                      int32_t *__restrict__ ticket, int32_t *__restrict__ err) {
    griddep_wait();
    extern __shared__ int32_t hist[];    // [E]
    metadata_count_body(topk_idx, R, E, n_chunks, blockIdx.x, block_hist, counts, offsets, mt_prefix, ticket, err,
                        hist);
}

// The place kernel's work for chunk `chunk`, with sh = (kWarps + 1) E ints of shared memory.
__device__ __forceinline__ void metadata_place_body(const int32_t *__restrict__ topk_idx, int R, int E, int chunk,
                                                    const int32_t *__restrict__ block_hist,
                                                    const int32_t *__restrict__ offsets,
                                                    int32_t *__restrict__ perm_slot, int32_t *__restrict__ row_of,
                                                    int32_t *sh) {
    int32_t *base = sh;                  // [E]: first row of this chunk in each expert
    int32_t *whist = sh + E;             // [kWarps][E]: per-warp counts, then start ranks
    for (int e = threadIdx.x; e < E; e += kThreads) {
        base[e] = offsets[e] + block_hist[static_cast<int64_t>(chunk) * E + e];
        for (int w = 0; w < kWarps; ++w) whist[w * E + e] = 0;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int beg = chunk * kChunk + warp * kWarpSlots;
    const int end = min(R, beg + kWarpSlots);
    int32_t *mine = whist + warp * E;
    int ev[kPerLane];
    load_lane_slots(topk_idx, beg, end, lane, ev);
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int s = beg + 32 * i + lane;
        const int e = ev[i];
        const bool valid = (s < end) && e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        if (valid && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kThreads) {
        int run = base[e];
        for (int w = 0; w < kWarps; ++w) {
            const int c = whist[w * E + e];
            whist[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const int s = beg + 32 * i + lane;
        const int e = ev[i];
        const bool valid = (s < end) && e >= 0 && e < E;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        if (valid) {
            const int pos = mine[e] + __popc(peers & ((1u << lane) - 1u));
            perm_slot[pos] = s;
            row_of[s] = pos;
        } else if (s < end) {
            row_of[s] = -1;
        }
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
        __syncwarp();
    }
}

// Counters of stage 2's fused k-way sum, one per (token, 256-column output
// tile): each starts at the number of the token's dropped slots, so the token's
// sum over a tile is complete when its counter reaches k (threads first,
// first + stride, ... over the tokens).
__device__ __forceinline__ void init_combine_counters(const int32_t *__restrict__ topk_idx, int E,
                                                      const CombineCounters &c, int first, int stride) {
    if (c.cnt == nullptr) return;
    for (int t = first; t < c.T; t += stride) {
        int dropped = 0;
        for (int j = 0; j < c.k; ++j) {
            const int e = __ldg(&topk_idx[static_cast<int64_t>(t) * c.k + j]);
            dropped += (e < 0 || e >= E) ? 1 : 0;
        }
        for (int n = 0; n < c.n_tiles; ++n) c.cnt[static_cast<int64_t>(t) * c.n_tiles + n] = dropped;
    }
}

__global__ void __launch_bounds__(kThreads)
metadata_place_kernel(const int32_t *__restrict__ topk_idx, int R, int E,
                      const int32_t *__restrict__ block_hist, const int32_t *__restrict__ offsets,
                      int32_t *__restrict__ perm_slot, int32_t *__restrict__ row_of, CombineCounters cc) {
    griddep_wait();
    extern __shared__ int32_t sh[];
    metadata_place_body(topk_idx, R, E, blockIdx.x, block_hist, offsets, perm_slot, row_of, sh);
    init_combine_counters(topk_idx, E, cc, blockIdx.x * kThreads + threadIdx.x, gridDim.x * kThreads);
}

// All slots in one chunk (at most kChunk, e.g. decode): one CTA runs the count and the
// place work back to back, saving a launch. The CTA is its own last CTA, so the count
// part also scans; its global writes are visible to the place part after the barrier.
__global__ void __launch_bounds__(kThreads)
metadata_single_chunk_kernel(const int32_t *__restrict__ topk_idx, int R, int E, int32_t *__restrict__ block_hist,
                             int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                             int32_t *__restrict__ mt_prefix, int32_t *__restrict__ ticket,
                             int32_t *__restrict__ err, int32_t *__restrict__ perm_slot,
                             int32_t *__restrict__ row_of, CombineCounters cc) {
    griddep_wait();
    extern __shared__ int32_t sh[];
    metadata_count_body(topk_idx, R, E, 1, 0, block_hist, counts, offsets, mt_prefix, ticket, err, sh);
    __syncthreads();
    metadata_place_body(topk_idx, R, E, 0, block_hist, offsets, perm_slot, row_of, sh);
    init_combine_counters(topk_idx, E, cc, threadIdx.x, kThreads);
}

size_t place_smem(int E) { return sizeof(int32_t) * static_cast<size_t>(kWarps + 1) * E; }

}  // namespace

cudaError_t setup_metadata_kernels() {
    cudaError_t e = cudaFuncSetAttribute(metadata_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(place_smem(1024)));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(metadata_single_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(place_smem(1024)));
    return e;
}

cudaError_t launch_routing_metadata(const MetadataLaunch &p, cudaStream_t st) {
    const int n_chunks = (p.R + kChunk - 1) / kChunk;
    if (n_chunks == 0) return cudaSuccess;
    if (n_chunks == 1) {
        const cudaError_t e = launch_dep(metadata_single_chunk_kernel, dim3(1), dim3(kThreads), place_smem(p.E), st,
                                         p.topk_idx, p.R, p.E, p.block_hist, p.counts, p.offsets, p.mt_prefix,
                                         p.ticket, p.err, p.perm_slot, p.row_of, p.combine);
        note_launches(1);
        return e;
    }
    cudaError_t e = launch_dep(metadata_count_kernel, dim3(n_chunks), dim3(kThreads), sizeof(int32_t) * p.E, st,
                               p.topk_idx, p.R, p.E, n_chunks, p.block_hist, p.counts, p.offsets, p.mt_prefix, p.ticket,
                               p.err);
    if (e == cudaSuccess)
        e = launch_dep(metadata_place_kernel, dim3(n_chunks), dim3(kThreads), place_smem(p.E), st, p.topk_idx, p.R,
                       p.E, p.block_hist, p.offsets, p.perm_slot, p.row_of, p.combine);
    note_launches(2);
    return e;
}

}  // namespace moe
