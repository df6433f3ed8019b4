// mx.cuh -- MXFP8 element and scale conversion on the device (the guide's
// mxfp8 expert precision, section "Expert precision"; the format is the Open
// Compute Project Microscaling format, OCP MX v1.0): blocks of 32 elements
// share a power-of-two scale 2^(floor(log2 max|v|) - 8) stored as E8M0 (bias
// 127, clamped to [2^-127, 2^127]); elements are E4M3, converted with
// round-to-nearest-even and saturation to +-448. A zero block gets scale code 0.
#pragma once

#include <stdint.h>

namespace moe {

// floor(log2 |a|) of a finite, non-zero float, exactly (normal or subnormal).
__device__ __forceinline__ int floor_log2(float a) {
    const uint32_t bits = __float_as_uint(a) & 0x7fffffffu;
    const int e = static_cast<int>(bits >> 23);
    if (e != 0) return e - 127;
    return (31 - __clz(static_cast<int>(bits))) - 149;       // subnormal: highest set mantissa bit
}

// E8M0 code of a block whose largest magnitude is amax.
__device__ __forceinline__ uint32_t mx_scale_code(float amax) {
    if (amax == 0.0f) return 0u;
    int e = floor_log2(amax) - 8;
    e = max(-127, min(127, e));
    return static_cast<uint32_t>(e + 127);
}

// 2^(127 - code): the factor that maps a block onto its E4M3 range (exact).
__device__ __forceinline__ float mx_inv_scale(uint32_t code) {
    const int e = 127 - static_cast<int>(code);               // in [-127, 127]
    return (e >= -126) ? __uint_as_float(static_cast<uint32_t>(e + 127) << 23)
                       : __uint_as_float(0x00400000u);        // 2^-127, subnormal
}

// Two floats to two E4M3 codes (round to nearest even, saturating); lo goes to
// the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Quantize 32 values of one block: 8 words of 4 codes (element 4w + b in byte
// b of word w) and the block's E8M0 scale code.
__device__ __forceinline__ uint32_t mx_quantize32(const float (&v)[32], uint32_t (&q)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const uint32_t code = mx_scale_code(amax);
    const float inv = mx_inv_scale(code);
#pragma unroll
    for (int w = 0; w < 8; ++w)
        q[w] = e4m3x2(v[4 * w] * inv, v[4 * w + 1] * inv) |
               (e4m3x2(v[4 * w + 2] * inv, v[4 * w + 3] * inv) << 16);
    return code;
}

}  // namespace moe
