/*
 * gemm_client.c -- a plain C user of libgemm07.so: device buffers from the
 * CUDA runtime, one call of each arithmetic entry point through the header
 * gemm07.h, and a check against a double-precision triple loop on integer
 * operands (every sum is an integer below 2^24, so the result is exact).
 *
 * Build (see tests/test_c_client.py):
 *   gcc -std=c99 -O2 -I include -I <cuda>/include gemm_client.c \
 *       -L <lib dir> -lgemm07 -L <cuda>/lib64 -lcudart -o gemm_client
 * Exit status 0 when both products are exact.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "gemm07.h"

static int check(const char *what, const float *c, const double *ref, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        if ((double)c[i] != ref[i]) {
            fprintf(stderr, "%s: element %lld is %g, expected %g\n", what,
                    (long long)i, (double)c[i], ref[i]);
            return 1;
        }
    printf("%s: %lld elements exact\n", what, (long long)n);
    return 0;
}

/* BF16 bits of a small integer (exact: it needs at most 8 significant bits). */
static uint16_t bf16_of(float x) {
    uint32_t w;
    memcpy(&w, &x, sizeof w);
    return (uint16_t)(w >> 16);
}

int main(void) {
    const int64_t M = 300, N = 260, K = 530;
    float *ha = malloc(sizeof(float) * M * K), *hb = malloc(sizeof(float) * K * N);
    uint16_t *ha16 = malloc(2 * M * K), *hb16 = malloc(2 * K * N);
    float *hc = malloc(sizeof(float) * M * N);
    double *ref = calloc((size_t)(M * N), sizeof(double));
    if (!ha || !hb || !ha16 || !hb16 || !hc || !ref) return 2;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) {
            ha[i * K + k] = (float)((i + 3 * k) % 7 - 3);
            ha16[i * K + k] = bf16_of(ha[i * K + k]);
        }
    for (int64_t k = 0; k < K; ++k)
        for (int64_t j = 0; j < N; ++j) {
            hb[k * N + j] = (float)((2 * k + j) % 5 - 2);
            hb16[k * N + j] = bf16_of(hb[k * N + j]);
        }
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k)
            for (int64_t j = 0; j < N; ++j)
                ref[i * N + j] += (double)ha[i * K + k] * (double)hb[k * N + j];

    float *da, *db, *dc;
    uint16_t *da16, *db16;
    if (cudaMalloc((void **)&da, sizeof(float) * M * K) != cudaSuccess ||
        cudaMalloc((void **)&db, sizeof(float) * K * N) != cudaSuccess ||
        cudaMalloc((void **)&dc, sizeof(float) * M * N) != cudaSuccess ||
        cudaMalloc((void **)&da16, 2 * M * K) != cudaSuccess ||
        cudaMalloc((void **)&db16, 2 * K * N) != cudaSuccess) {
        fprintf(stderr, "cudaMalloc failed\n");
        return 2;
    }
    cudaMemcpy(da, ha, sizeof(float) * M * K, cudaMemcpyHostToDevice);
    cudaMemcpy(db, hb, sizeof(float) * K * N, cudaMemcpyHostToDevice);
    cudaMemcpy(da16, ha16, 2 * M * K, cudaMemcpyHostToDevice);
    cudaMemcpy(db16, hb16, 2 * K * N, cudaMemcpyHostToDevice);

    int bad = 0;
    gemm_status_t s = gemm_f32(M, N, K, da, K, db, N, dc, N, NULL);
    if (s != GEMM_OK || gemm_get_device_status(NULL) != GEMM_OK) {
        fprintf(stderr, "gemm_f32: %s\n", gemm_status_string(s));
        return 3;
    }
    cudaMemcpy(hc, dc, sizeof(float) * M * N, cudaMemcpyDeviceToHost);
    bad |= check("gemm_f32", hc, ref, M * N);

    s = gemm_bf16_f32acc(M, N, K, da16, K, db16, N, dc, N, NULL);
    if (s != GEMM_OK || gemm_get_device_status(NULL) != GEMM_OK) {
        fprintf(stderr, "gemm_bf16_f32acc: %s\n", gemm_status_string(s));
        return 3;
    }
    cudaMemcpy(hc, dc, sizeof(float) * M * N, cudaMemcpyDeviceToHost);
    bad |= check("gemm_bf16_f32acc", hc, ref, M * N);

    /* an argument error is reported before anything is enqueued */
    if (gemm_f32(M, N, K, da, K - 1, db, N, dc, N, NULL) != GEMM_ERR_INVALID_ARG) {
        fprintf(stderr, "short lda was not rejected\n");
        bad = 1;
    }
    gemm_shutdown();
    cudaFree(da); cudaFree(db); cudaFree(dc); cudaFree(da16); cudaFree(db16);
    free(ha); free(hb); free(ha16); free(hb16); free(hc); free(ref);
    printf(bad ? "FAILED\n" : "OK\n");
    return bad;
}
