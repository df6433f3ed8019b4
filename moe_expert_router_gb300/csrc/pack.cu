// pack.cu -- the tile-packed weight layout of the forward expert GEMMs.
//
// The grouped GEMMs read a weight slab per pipeline stage: 256 rows x 64
// K-elements (bf16) of one expert, in the 128-byte-swizzled K-major image the
// tensor core reads from shared memory. From the row-major tensors each slab
// is 256 strided 128-byte pieces; packed, it is one contiguous 32 KB block that
// a single bulk copy moves into shared memory, which keeps DRAM pages open
// while the weights stream (the weights are read once per step, so their
// streaming rate bounds the weight-heavy configurations).
//
//   w1p: tiles (e, n, kb), n < ceil(I / 128), kb < ceil(H / 64): row r < 128 is
//        w1[e][n*128 + r] (gate), row 128 + r is w1[e][I + n*128 + r] (up);
//   w2p: tiles (e, n, kb), n < ceil(H / 256), kb < ceil(I / 64): row r is
//        w2[e][n*256 + r].
// Rows past the projection (gate/up index >= I, or output row >= H) and
// columns past K are zero. Inside a tile, 16-byte chunk c of row r sits at
// byte r * 128 + ((c ^ (r % 8)) * 16). Tiles are ordered (e, n, kb), so a
// unit's stages are consecutive blocks.
#include "internal.cuh"

namespace moe {

namespace {

// mode 1: w1 (gate / up halves), mode 2: w2. One thread per 16-byte chunk of the
// packed output, grid-stride.
__global__ void __launch_bounds__(256)
pack_weights_kernel(const __nv_bfloat16 *__restrict__ w, int mode, int64_t E, int64_t half, int64_t K,
                    int64_t n_tiles, int64_t kb_tiles, uint4 *__restrict__ out) {
    griddep_wait();
    const int64_t total = E * n_tiles * kb_tiles * 256 * 8;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int slot = static_cast<int>(i & 7);
        const int r = static_cast<int>((i >> 3) & 255);
        const int64_t tile = i >> 11;
        const int64_t kb = tile % kb_tiles;
        const int64_t en = tile / kb_tiles;
        const int64_t n = en % n_tiles;
        const int64_t e = en / n_tiles;
        const int c = slot ^ (r & 7);                       // the source chunk stored in this slot
        const int64_t col = kb * 64 + c * 8;
        int64_t row;                                       // row inside the expert's matrix
        bool ok;
        if (mode == 1) {
            const int64_t j = n * 128 + (r & 127);          // gate / up index
            ok = j < half;
            row = (r < 128 ? 0 : half) + j;
        } else {
            row = n * 256 + r;
            ok = row < half;                                // half = H, the expert's rows
        }
        ok = ok && col < K;
        const int64_t rows_per_e = (mode == 1) ? 2 * half : half;
        out[i] = ok ? __ldg(reinterpret_cast<const uint4 *>(w + (e * rows_per_e + row) * K + col))
                    : make_uint4(0u, 0u, 0u, 0u);
    }
}

}  // namespace

int64_t packed_w1_tiles(int64_t E, int64_t H, int64_t I) { return E * ((I + 127) / 128) * ((H + 63) / 64); }
int64_t packed_w2_tiles(int64_t E, int64_t H, int64_t I) { return E * ((H + 255) / 256) * ((I + 63) / 64); }

cudaError_t launch_pack_w1(const __nv_bfloat16 *w1, int64_t E, int64_t H, int64_t I, void *w1p, cudaStream_t st) {
    const int64_t chunks = packed_w1_tiles(E, H, I) * 256 * 8;
    if (chunks == 0) return cudaSuccess;
    int64_t grid = (chunks + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    const cudaError_t e = launch_dep(pack_weights_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, w1, 1, E, I,
                                     H, (I + 127) / 128, (H + 63) / 64, static_cast<uint4 *>(w1p));
    note_launches(1);
    return e;
}

cudaError_t launch_pack_w2(const __nv_bfloat16 *w2, int64_t E, int64_t H, int64_t I, void *w2p, cudaStream_t st) {
    const int64_t chunks = packed_w2_tiles(E, H, I) * 256 * 8;
    if (chunks == 0) return cudaSuccess;
    int64_t grid = (chunks + 255) / 256;
    if (grid > 152 * 16) grid = 152 * 16;
    const cudaError_t e = launch_dep(pack_weights_kernel, dim3(static_cast<int>(grid)), dim3(256), 0, st, w2, 2, E, H,
                                     I, (H + 255) / 256, (I + 63) / 64, static_cast<uint4 *>(w2p));
    note_launches(1);
    return e;
}

}  // namespace moe
