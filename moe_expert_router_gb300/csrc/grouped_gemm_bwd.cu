// grouped_gemm_bwd.cu -- backward instantiations of the tcgen05 grouped-GEMM
// kernel (gemm_kernel.cuh). The guide's stage order (MegaMoE guide, section
// "Design: two stages": stage 2's backward yields dW2, then stage 1's yields
// dW1) maps onto four launches:
//   dA  (stage 2 backward, data):    dA_u = dY . w2[e], SwiGLU backward epilogue
//   dW2 (stage 2 backward, weights): dW2[e] = dY_e^T (w a)_e
//   dX  (stage 1 backward, data):    dXr = dH . w1[e]
//   dW1 (stage 1 backward, weights): dW1[e] = dH_e^T x_e
#include "gemm_kernel.cuh"

namespace moe {

cudaError_t setup_bwd_gemm_kernels() {
    cudaError_t e = set_gemm_smem<kBwdDA>();
    if (e == cudaSuccess) e = set_gemm_smem<kBwdDX>();
    if (e == cudaSuccess) e = set_gemm_smem<kBwdDW2>();
    if (e == cudaSuccess) e = set_gemm_smem<kBwdDW1>();
    return e;
}

cudaError_t launch_bwd_da(const GemmLaunch &p, cudaStream_t st) {
    return launch_tc_gemm<kBwdDA>(maps_of(p), grouped_args(p), p.num_sms, st);
}

cudaError_t launch_bwd_dx(const GemmLaunch &p, cudaStream_t st) {
    return launch_tc_gemm<kBwdDX>(maps_of(p), grouped_args(p), p.num_sms, st);
}

cudaError_t launch_bwd_dw2(const GemmLaunch &p, cudaStream_t st) {
    GemmArgs g = grouped_args(p);
    g.total_units = g.E * g.m_tiles * g.n_tiles;
    const int grid = g.total_units < p.num_sms ? g.total_units : p.num_sms;
    if (grid <= 0) return cudaSuccess;
    return launch_tc_gemm<kBwdDW2>(maps_of(p), g, grid, st);
}

cudaError_t launch_bwd_dw1(const GemmLaunch &p, cudaStream_t st) {
    GemmArgs g = grouped_args(p);
    g.total_units = g.E * g.m_tiles * g.n_tiles;
    const int grid = g.total_units < p.num_sms ? g.total_units : p.num_sms;
    if (grid <= 0) return cudaSuccess;
    return launch_tc_gemm<kBwdDW1>(maps_of(p), g, grid, st);
}

}  // namespace moe
