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
// One CTA of 32 warps. Warp w owns the contiguous slot range
// [w*chunk, (w+1)*chunk): pass 1 counts per (warp, expert) with __match_any,
// pass 2 turns those counts into per-warp starting ranks and the expert
// offsets, pass 3 re-walks the range and places every slot. Walking the slots
// in order inside each warp and the warps in order makes the permutation
// stable without sorting.
#include "internal.cuh"

namespace moe {

namespace {

constexpr int kMetaThreads = 1024;
constexpr int kMetaWarps = kMetaThreads / 32;

__global__ void __launch_bounds__(kMetaThreads, 1)
routing_metadata_kernel(const int32_t *__restrict__ topk_idx, int R, int E,
                        int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                        int32_t *__restrict__ mt_prefix, int32_t *__restrict__ perm_slot,
                        int32_t *__restrict__ row_of, int32_t *__restrict__ err) {
    extern __shared__ int32_t sh[];
    int32_t *hist = sh;                       // [kMetaWarps][E]: counts, then start ranks
    int32_t *base = sh + kMetaWarps * E;      // [E]: expert offsets
    __shared__ int32_t warp_tot_c[kMetaWarps], warp_tot_m[kMetaWarps];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kMetaWarps * E; i += kMetaThreads) hist[i] = 0;
    __syncthreads();

    const int chunk = (R + kMetaWarps - 1) / kMetaWarps;
    const int beg = warp * chunk;
    const int end = min(R, beg + chunk);
    int bad = 0;

    // pass 1: rows per (warp, expert)
    for (int s0 = beg; s0 < end; s0 += 32) {
        const int s = s0 + lane;
        const int e = (s < end) ? topk_idx[s] : -1;
        const bool valid = (s < end) && e >= 0 && e < E;
        bad |= (s < end) && !valid;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
        if (valid && lane == __ffs(peers) - 1) hist[warp * E + e] += __popc(peers);
    }
    __syncthreads();

    // pass 2a: per expert, running total over warps -> each warp's starting rank
    for (int e = threadIdx.x; e < E; e += kMetaThreads) {
        int run = 0;
        for (int w = 0; w < kMetaWarps; ++w) {
            const int c = hist[w * E + e];
            hist[w * E + e] = run;
            run += c;
        }
        base[e] = run;
    }
    __syncthreads();

    // pass 2b: exclusive scans over experts of counts and of row tiles (E <= 1024)
    const int e = threadIdx.x;
    const int c = (e < E) ? base[e] : 0;
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
        int vc = warp_tot_c[lane], vm = warp_tot_m[lane];
        const int oc = vc, om = vm;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int yc = __shfl_up_sync(0xffffffffu, vc, off);
            const int ym = __shfl_up_sync(0xffffffffu, vm, off);
            if (lane >= off) { vc += yc; vm += ym; }
        }
        warp_tot_c[lane] = vc - oc;   // exclusive prefix of the warp totals
        warp_tot_m[lane] = vm - om;
    }
    __syncthreads();
    const int ex_c = ic - c + warp_tot_c[warp];
    const int ex_m = im - m + warp_tot_m[warp];
    if (e < E) {
        counts[e] = c;
        offsets[e] = ex_c;
        mt_prefix[e] = ex_m;
        base[e] = ex_c;
        if (e == E - 1) {
            offsets[E] = ex_c + c;
            mt_prefix[E] = ex_m + m;
        }
    }
    __syncthreads();

    // pass 3: place every slot
    for (int s0 = beg; s0 < end; s0 += 32) {
        const int s = s0 + lane;
        const int ee = (s < end) ? topk_idx[s] : -1;
        const bool valid = (s < end) && ee >= 0 && ee < E;
        const unsigned peers = __match_any_sync(0xffffffffu, valid ? ee : -1);
        if (valid) {
            const int rank = __popc(peers & ((1u << lane) - 1u));
            const int pos = base[ee] + hist[warp * E + ee] + rank;
            perm_slot[pos] = s;
            row_of[s] = pos;
        } else if (s < end) {
            row_of[s] = -1;
        }
        __syncwarp();
        if (valid && lane == __ffs(peers) - 1) hist[warp * E + ee] += __popc(peers);
        __syncwarp();
    }
    if (bad) atomicOr(err, MOE_DEVERR_BAD_EXPERT_INDEX);
}

size_t metadata_smem(int E) { return sizeof(int32_t) * static_cast<size_t>(kMetaWarps + 1) * E; }

}  // namespace

cudaError_t setup_metadata_kernels() {
    return cudaFuncSetAttribute(routing_metadata_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(metadata_smem(1024)));
}

cudaError_t launch_routing_metadata(const MetadataLaunch &p, cudaStream_t st) {
    routing_metadata_kernel<<<1, kMetaThreads, metadata_smem(p.E), st>>>(
        p.topk_idx, p.R, p.E, p.counts, p.offsets, p.mt_prefix, p.perm_slot, p.row_of, p.err);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace moe
