// grouped_gemm.cu -- forward instantiations of the tcgen05 grouped-GEMM kernel
// (gemm_kernel.cuh): stage 1 (dispatch_grouped_gemm with the fused SwiGLU),
// stage 2 (grouped_gemm_combine's GEMM with the weighted scatter) and the
// router GEMM; plus the final k-way combine of stage 2 (MegaMoE guide, opening
// section and section "Design: two stages").
#include "gemm_kernel.cuh"

namespace moe {

namespace {

// y[t, :] = sum over the token's k slots s of obuf[row_of[s], :] (rows already
// weighted, in routed order); dropped slots (row_of < 0) are skipped. fp32 sum
// in slot order, bf16 result. One warp per token (grid-stride over tokens):
// lane j < k reads the token's row_of[j] once; every lane then sums 8-column
// groups lane, lane + 32, ... with the k row loads of a group issued together
// (all lanes run the same passes, so the shuffles see the whole warp).
__global__ void __launch_bounds__(256)
combine_kernel(const __nv_bfloat16 *__restrict__ obuf, const int32_t *__restrict__ row_of,
               __nv_bfloat16 *__restrict__ y, int T, int H, int k) {
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int groups = H >> 3;
    const int warps = gridDim.x * (blockDim.x >> 5);
    for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps) {
        const int my_row = lane < k ? __ldg(&row_of[static_cast<int64_t>(t) * k + lane]) : -1;
        for (int g0 = 0; g0 < groups; g0 += 32) {
            const int g = g0 + lane;
            const bool live = g < groups;
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            for (int j0 = 0; j0 < k; j0 += 8) {
                uint4 v[8];
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) {
                    const int r = __shfl_sync(0xffffffffu, my_row, (j0 + jj) & 31);
                    v[jj] = (live && j0 + jj < k && r >= 0)
                                ? __ldg(reinterpret_cast<const uint4 *>(obuf + static_cast<int64_t>(r) * H) + g)
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
                reinterpret_cast<uint4 *>(y + static_cast<int64_t>(t) * H)[g] =
                    make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                               pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
        }
    }
}

}  // namespace

cudaError_t setup_gemm_kernels() {
    cudaError_t e = set_gemm_smem<kStage1>();
    if (e == cudaSuccess) e = set_gemm_smem<kStage1SaveH>();
    if (e == cudaSuccess) e = set_gemm_smem<kStage2>();
    if (e == cudaSuccess) e = set_gemm_smem<kRouter>();
    if (e == cudaSuccess) e = setup_bwd_gemm_kernels();
    if (e == cudaSuccess) e = setup_mx_gemm_kernels();
    return e;
}

cudaError_t launch_gemm1_swiglu(const GemmLaunch &p, cudaStream_t st) {
    if (p.save_h) return launch_tc_gemm<kStage1SaveH>(maps_of(p), grouped_args(p), p.num_sms, st);
    return launch_tc_gemm<kStage1>(maps_of(p), grouped_args(p), p.num_sms, st);
}

cudaError_t launch_gemm2_scatter(const GemmLaunch &p, cudaStream_t st) {
    return launch_tc_gemm<kStage2>(maps_of(p), grouped_args(p), p.num_sms, st);
}

cudaError_t launch_router_gemm(const RouterGemmLaunch &p, cudaStream_t st) {
    GemmArgs g{};
    g.err = p.err;
    g.sched = p.sched;
    g.logits_part = p.logits_part;
    g.E = p.E;
    g.K = p.H;
    g.n_out = p.E;
    g.router_seg = router_seg(p.E);
    g.n_mma = g.router_seg ? 3 * g.router_seg : router_n_mma(p.E);
    g.n_tiles = (p.E + BN - 1) / BN;
    g.T = p.T;
    g.kb_total = static_cast<int>(router_kb_total(p.H, p.E));
    g.splits = p.splits;
    g.kb_per_split = (g.kb_total + p.splits - 1) / p.splits;
    g.total_units = ((p.T + UM - 1) / UM) * g.n_tiles * p.splits;
    // every split must own at least one k-block: an empty split would leave its
    // accumulator unwritten
    if (p.splits < 1 || (p.splits - 1) * g.kb_per_split >= g.kb_total) return cudaErrorInvalidValue;
    const int grid = g.total_units < p.num_sms ? g.total_units : p.num_sms;
    GemmMaps m;
    m.a = *p.tm_x;
    m.b = *p.tm_w3;
    m.out = *p.tm_w3;
    m.out2 = *p.tm_w3;
    m.out3 = *p.tm_w3;
    m.sfa = *p.tm_w3;
    m.sfb = *p.tm_w3;
    return launch_tc_gemm<kRouter>(m, g, grid, st);
}

cudaError_t launch_combine(const CombineLaunch &p, cudaStream_t st) {
    if (p.T == 0 || p.H == 0) return cudaSuccess;
    int64_t blocks = (static_cast<int64_t>(p.T) + 7) / 8;     // eight tokens (warps) per block
    if (blocks > 152 * 8) blocks = 152 * 8;
    const cudaError_t e = launch_dep(combine_kernel, dim3(static_cast<int>(blocks)), dim3(256), 0, st, p.obuf,
                                     p.row_of, p.y, p.T, p.H, p.k);
    note_launches(1);
    return e;
}

}  // namespace moe
