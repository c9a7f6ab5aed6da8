/* A plain C host program on the C ABI of libfkl.so (no Python, no torch): it builds
 * a small synthetic problem from a counter hash, runs fkl_forward, fkl_backward and
 * fkl_forward_noalloc, and writes loss, lse, dh and dW to a binary file.  The GPU
 * test that compiles it rebuilds the same inputs from the same hash and compares the
 * file with the fp64 oracle.
 *
 *   fkl_c_demo <out-file>          exit status 0 on success
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "fkl.h"

enum { N = 300, D = 128, V = 2048, K = 16, CHUNK = 128 };
static const float T = 1.5f;

/* 32-bit integer hash (xorshift-multiply), the same formula as the test's. */
static uint32_t mix32(uint32_t x) {
    x ^= x >> 16;
    x *= 0x7feb352dU;
    x ^= x >> 15;
    x *= 0x846ca68bU;
    x ^= x >> 16;
    return x;
}

/* Uniform in [0, 1) from counter i and stream s: the top 24 bits of the hash. */
static float unif(uint32_t i, uint32_t s) { return (float)(mix32(i * 2654435761U ^ (s * 0x9e3779b9U)) >> 8) / 16777216.0f; }

/* fp32 -> bf16 bits, round to nearest even (finite inputs). */
static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7fffU + ((u >> 16) & 1U);
    return (uint16_t)(u >> 16);
}

#define CHECK_CUDA(x)                                                             \
    do {                                                                          \
        cudaError_t e_ = (x);                                                     \
        if (e_ != cudaSuccess) {                                                  \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));              \
            return 2;                                                             \
        }                                                                         \
    } while (0)
#define CHECK_FKL(x)                                                              \
    do {                                                                          \
        fkl_status s_ = (x);                                                      \
        if (s_ != FKL_OK) {                                                       \
            fprintf(stderr, "%s: %s (%s)\n", #x, fkl_status_string(s_), fkl_last_error()); \
            return 3;                                                             \
        }                                                                         \
    } while (0)

int main(int argc, char** argv) {
    if (argc != 2) {
        fprintf(stderr, "usage: %s <out-file>\n", argv[0]);
        return 1;
    }
    static uint16_t h[N * D], W[V * D], dh[N * D];
    static int32_t idx[N * K];
    static float t[N * K], lse[N], dW[V * D];
    static uint8_t mask[N];
    for (uint32_t i = 0; i < N * D; ++i) h[i] = to_bf16(2.0f * unif(i, 1) - 1.0f);
    for (uint32_t i = 0; i < V * D; ++i) W[i] = to_bf16(0.2f * unif(i, 2) - 0.1f);
    for (uint32_t r = 0; r < N; ++r) {
        mask[r] = (uint8_t)(r % 17 != 0);
        for (uint32_t k = 0; k < K; ++k) {
            idx[r * K + k] = (int32_t)((r * 131U + k * 997U) % V); /* distinct: gcd(997, 2048) = 1 */
            t[r * K + k] = 4.0f * unif(r * K + k, 3) - 2.0f;
        }
    }

    void *dh_d, *dh_w, *didx, *dt, *dmask, *dloss, *dlse, *ddh, *ddW, *dws, *dstat;
    const size_t ws_bytes = fkl_workspace_size(N, D, V, K, CHUNK);
    if (ws_bytes == 0) return 4;
    CHECK_CUDA(cudaMalloc(&dh_d, sizeof h));
    CHECK_CUDA(cudaMalloc(&dh_w, sizeof W));
    CHECK_CUDA(cudaMalloc(&didx, sizeof idx));
    CHECK_CUDA(cudaMalloc(&dt, sizeof t));
    CHECK_CUDA(cudaMalloc(&dmask, sizeof mask));
    CHECK_CUDA(cudaMalloc(&dloss, 2 * sizeof(float)));
    CHECK_CUDA(cudaMalloc(&dlse, sizeof lse));
    CHECK_CUDA(cudaMalloc(&ddh, sizeof dh));
    CHECK_CUDA(cudaMalloc(&ddW, sizeof dW));
    CHECK_CUDA(cudaMalloc(&dws, ws_bytes));
    CHECK_CUDA(cudaMalloc(&dstat, sizeof(int)));
    CHECK_CUDA(cudaMemcpy(dh_d, h, sizeof h, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dh_w, W, sizeof W, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(didx, idx, sizeof idx, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dt, t, sizeof t, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dmask, mask, sizeof mask, cudaMemcpyHostToDevice));

    cudaStream_t st;
    CHECK_CUDA(cudaStreamCreate(&st));
    CHECK_FKL(fkl_forward(dh_d, dh_w, (const int32_t*)didx, (const float*)dt, (const uint8_t*)dmask, N, D, V, K,
                          T, CHUNK, (float*)dloss, (float*)dlse, dws, ws_bytes, st));
    CHECK_FKL(fkl_backward(dh_d, dh_w, (const int32_t*)didx, (const float*)dt, (const uint8_t*)dmask, N, D, V, K,
                           T, CHUNK, (const float*)dlse, NULL, ddh, (float*)ddW, dws, ws_bytes, st));
    CHECK_FKL(fkl_get_status(dws, st));
    /* the same forward on the library's own scratch: no workspace from this program */
    CHECK_FKL(fkl_forward_noalloc(dh_d, dh_w, (const int32_t*)didx, (const float*)dt, (const uint8_t*)dmask, N, D,
                                  V, K, T, CHUNK, (float*)dloss + 1, (float*)dlse, (int*)dstat, st));
    CHECK_CUDA(cudaStreamSynchronize(st));

    float loss[2];
    int dev_status = -1;
    CHECK_CUDA(cudaMemcpy(loss, dloss, sizeof loss, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(&dev_status, dstat, sizeof(int), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(lse, dlse, sizeof lse, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(dh, ddh, sizeof dh, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(dW, ddW, sizeof dW, cudaMemcpyDeviceToHost));
    if (dev_status != 0) return 5;

    FILE* f = fopen(argv[1], "wb");
    if (!f) return 6;
    fwrite(loss, sizeof(float), 2, f);
    fwrite(lse, sizeof(float), N, f);
    fwrite(dh, sizeof(uint16_t), N * D, f);
    fwrite(dW, sizeof(float), V * D, f);
    fclose(f);
    printf("loss %.9g (no-alloc forward %.9g), %lld launches\n", loss[0], loss[1], (long long)fkl_launch_count());
    return 0;
}
