/*
 * c_abi_forward.c -- a plain C caller of libmoe (no Python, no PyTorch): device
 * buffers from cudaMalloc, the workspace sized and initialised through the C ABI,
 * one moe_forward, and y compared with the fp64 CPU oracle (oracle/liboracle.so,
 * test infrastructure only). Built and run by tests/test_gpu_c_abi.py.
 *
 * Exit status 0 when every call returns MOE_OK, the device error word is 0 and y
 * is within the output bound (relative Frobenius error <= 1e-2); 1 otherwise.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "moe.h"

/* oracle/moe_oracle.c */
int oracle_expert_forward(int64_t T, int64_t H, int64_t I, int64_t E, int32_t k, const uint16_t *x,
                          const int32_t *topk_idx, const double *topk_w, const uint16_t *w1,
                          const uint16_t *w2, double *y, double *a_slot, double *o_slot);

static uint32_t g_state = 12345u;

/* uniform in [0, 1): a 32-bit linear congruential generator, top 24 bits */
static float uniform01(void) {
    g_state = g_state * 1664525u + 1013904223u;
    return (float)(g_state >> 8) / 16777216.0f;
}

/* round-to-nearest-even fp32 -> bf16 bits (finite values only) */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static double from_bf16(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

#define CHECK_MOE(call)                                                                   \
    do {                                                                                  \
        const moe_status_t st_ = (call);                                                  \
        if (st_ != MOE_OK) {                                                              \
            fprintf(stderr, "%s failed: %s\n", #call, moe_status_string(st_));           \
            return 1;                                                                     \
        }                                                                                 \
    } while (0)

#define CHECK_CUDA(call)                                                                  \
    do {                                                                                  \
        const cudaError_t e_ = (call);                                                    \
        if (e_ != cudaSuccess) {                                                          \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));            \
            return 1;                                                                     \
        }                                                                                 \
    } while (0)

int main(void) {
    /* a partial 256-row tile per expert, an H tail past 64 and an I tail past 128 */
    const int64_t T = 300, H = 200, I = 136, E = 5;
    const int32_t k = 2;
    const int64_t nx = T * H, nw1 = E * 2 * I * H, nw2 = E * H * I, ny = T * H;

    uint16_t *x = malloc(sizeof(uint16_t) * nx), *w1 = malloc(sizeof(uint16_t) * nw1),
             *w2 = malloc(sizeof(uint16_t) * nw2), *y = malloc(sizeof(uint16_t) * ny);
    int32_t *idx = malloc(sizeof(int32_t) * T * k);
    float *tw = malloc(sizeof(float) * T * k);
    double *tw64 = malloc(sizeof(double) * T * k), *y_ref = malloc(sizeof(double) * ny);
    if (!x || !w1 || !w2 || !y || !idx || !tw || !tw64 || !y_ref) return 1;
    for (int64_t i = 0; i < nx; ++i) x[i] = to_bf16(2.0f * uniform01() - 1.0f);
    for (int64_t i = 0; i < nw1; ++i) w1[i] = to_bf16((2.0f * uniform01() - 1.0f) / sqrtf((float)H));
    for (int64_t i = 0; i < nw2; ++i) w2[i] = to_bf16((2.0f * uniform01() - 1.0f) / sqrtf((float)I));
    for (int64_t t = 0; t < T; ++t) {      /* two distinct experts per token */
        const int32_t e0 = (int32_t)(uniform01() * E);
        const int32_t e1 = (int32_t)((e0 + 1 + (int32_t)(uniform01() * (E - 1))) % E);
        idx[t * k] = e0;
        idx[t * k + 1] = e1;
        for (int j = 0; j < k; ++j) {
            tw[t * k + j] = 0.1f + 0.9f * uniform01();
            tw64[t * k + j] = tw[t * k + j];
        }
    }

    moe_shape_t s;
    memset(&s, 0, sizeof(s));
    s.T = T;
    s.H = H;
    s.I = I;
    s.E = E;
    s.k = k;
    size_t ws_bytes = 0;
    CHECK_MOE(moe_workspace_size(&s, &ws_bytes));

    void *dx, *dw1, *dw2, *dy, *dws, *didx, *dtw;
    CHECK_CUDA(cudaMalloc(&dx, sizeof(uint16_t) * nx));
    CHECK_CUDA(cudaMalloc(&dw1, sizeof(uint16_t) * nw1));
    CHECK_CUDA(cudaMalloc(&dw2, sizeof(uint16_t) * nw2));
    CHECK_CUDA(cudaMalloc(&dy, sizeof(uint16_t) * ny));
    CHECK_CUDA(cudaMalloc(&didx, sizeof(int32_t) * T * k));
    CHECK_CUDA(cudaMalloc(&dtw, sizeof(float) * T * k));
    CHECK_CUDA(cudaMalloc(&dws, ws_bytes));
    CHECK_CUDA(cudaMemcpy(dx, x, sizeof(uint16_t) * nx, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dw1, w1, sizeof(uint16_t) * nw1, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dw2, w2, sizeof(uint16_t) * nw2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(didx, idx, sizeof(int32_t) * T * k, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dtw, tw, sizeof(float) * T * k, cudaMemcpyHostToDevice));

    CHECK_MOE(moe_workspace_init(dws, ws_bytes, NULL));
    CHECK_MOE(moe_forward(dx, (const int32_t *)didx, (const float *)dtw, dw1, dw2, &s, dy, dws, ws_bytes, NULL));
    int32_t code = -1;
    CHECK_MOE(moe_get_device_error(dws, &code, NULL));
    if (code != 0) {
        fprintf(stderr, "device error word %d\n", code);
        return 1;
    }
    CHECK_CUDA(cudaMemcpy(y, dy, sizeof(uint16_t) * ny, cudaMemcpyDeviceToHost));

    if (oracle_expert_forward(T, H, I, E, k, x, idx, tw64, w1, w2, y_ref, NULL, NULL) != 0) {
        fprintf(stderr, "oracle failed\n");
        return 1;
    }
    double err = 0.0, ref = 0.0;
    for (int64_t i = 0; i < ny; ++i) {
        const double d = from_bf16(y[i]) - y_ref[i];
        if (!isfinite(from_bf16(y[i]))) {
            fprintf(stderr, "non-finite y at %lld\n", (long long)i);
            return 1;
        }
        err += d * d;
        ref += y_ref[i] * y_ref[i];
    }
    const double rel = sqrt(err / ref);
    printf("c_abi_forward: T=%lld H=%lld I=%lld E=%lld k=%d, y relative Frobenius error %.3e\n",
           (long long)T, (long long)H, (long long)I, (long long)E, k, rel);

    cudaFree(dx);
    cudaFree(dw1);
    cudaFree(dw2);
    cudaFree(dy);
    cudaFree(didx);
    cudaFree(dtw);
    cudaFree(dws);
    free(x);
    free(w1);
    free(w2);
    free(y);
    free(idx);
    free(tw);
    free(tw64);
    free(y_ref);
    return rel <= 1e-2 ? 0 : 1;
}
