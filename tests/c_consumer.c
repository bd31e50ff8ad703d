/*
 * A plain C11 consumer of the library's C ABI (include/mxfp8.h): no Python, no
 * C++.  It quantizes a seeded BF16 matrix on the current GPU through
 * mxfp8_quantize (both directions, E5M2, fused dbias with a caller-owned
 * workspace), copies the outputs back and compares them with the CPU oracle
 * (test infrastructure, linked from oracle/), then checks a few host-side
 * rejections.  Exit status 0 and "c consumer ok" on success.
 *
 * Build (from the repository root, after the library and the oracle are built):
 *   gcc -std=c11 -O2 -Wall -Werror -I include -I /usr/local/cuda/include tests/c_consumer.c \
 *       mxfp8_block_scaled_04_gb300/_build/libmxfp8.so oracle/_build/liboracle.so \
 *       -L /usr/local/cuda/lib64 -lcudart -lm -o c_consumer
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "mxfp8.h"

/* the oracle's entry point (oracle/mxfp8_oracle.c) */
int mxo_quantize(const uint16_t *x, int64_t M, int64_t N, int fmt, uint8_t *out_row, uint8_t *scale_row,
                 uint8_t *out_col, uint8_t *scale_col, float *dbias);

#define CHECK_CUDA(call)                                                                          \
    do {                                                                                          \
        cudaError_t e_ = (call);                                                                  \
        if (e_ != cudaSuccess) {                                                                  \
            fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, cudaGetErrorString(e_));           \
            return 1;                                                                             \
        }                                                                                         \
    } while (0)

/* splitmix64: a seeded stream of 64-bit values */
static uint64_t next_u64(uint64_t *s)
{
    uint64_t z = (*s += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* a finite BF16 value with a spread of exponents (sign, exponent 100..150, mantissa) */
static uint16_t seeded_bf16(uint64_t *s)
{
    const uint64_t r = next_u64(s);
    const uint16_t sign = (uint16_t)((r >> 63) << 15);
    const uint16_t expo = (uint16_t)(100 + (r >> 8) % 51);
    const uint16_t mant = (uint16_t)(r & 0x7F);
    return (uint16_t)(sign | (expo << 7) | mant);
}

static double bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int main(void)
{
    const int64_t M = 300, N = 264; /* ragged: M % 32 = 12, N % 32 = 8 */
    const int64_t Cr = (N + 31) / 32, Rc = (M + 31) / 32;
    const size_t nx = (size_t)(M * N);
    uint64_t seed = 12345;

    uint16_t *x = malloc(nx * sizeof *x);
    uint8_t *o_row = malloc(nx), *o_col = malloc(nx), *s_row = malloc((size_t)(M * Cr)), *s_col = malloc((size_t)(Rc * N));
    uint8_t *r_row = malloc(nx), *r_col = malloc(nx), *rs_row = malloc((size_t)(M * Cr)), *rs_col = malloc((size_t)(Rc * N));
    float *dbias = malloc((size_t)N * sizeof(float)), *r_dbias = malloc((size_t)N * sizeof(float));
    if (!x || !o_row || !o_col || !s_row || !s_col || !r_row || !r_col || !rs_row || !rs_col || !dbias || !r_dbias)
        return 1;
    for (size_t i = 0; i < nx; i++)
        x[i] = seeded_bf16(&seed);

    void *dx, *d_orow, *d_srow, *d_ocol, *d_scol, *d_ws;
    float *d_dbias;
    const size_t ws_bytes = mxfp8_quantize_workspace_bytes(M, N, 1);
    if (ws_bytes != (size_t)((M + 127) / 128) * (size_t)N * sizeof(float)) {
        fprintf(stderr, "workspace bytes %zu\n", ws_bytes);
        return 1;
    }
    CHECK_CUDA(cudaMalloc(&dx, nx * 2));
    CHECK_CUDA(cudaMalloc(&d_orow, nx));
    CHECK_CUDA(cudaMalloc(&d_ocol, nx));
    CHECK_CUDA(cudaMalloc(&d_srow, (size_t)(M * Cr)));
    CHECK_CUDA(cudaMalloc(&d_scol, (size_t)(Rc * N)));
    CHECK_CUDA(cudaMalloc((void **)&d_dbias, (size_t)N * sizeof(float)));
    CHECK_CUDA(cudaMalloc(&d_ws, ws_bytes));
    CHECK_CUDA(cudaMemcpy(dx, x, nx * 2, cudaMemcpyHostToDevice));

    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));
    mxfp8_status_t st = mxfp8_quantize(dx, M, N, MXFP8_E5M2, d_orow, d_srow, d_ocol, d_scol, d_dbias, d_ws, NULL,
                                       (void *)stream);
    if (st != MXFP8_OK) {
        fprintf(stderr, "mxfp8_quantize: %s\n", mxfp8_status_string(st));
        return 1;
    }
    CHECK_CUDA(cudaStreamSynchronize(stream));
    CHECK_CUDA(cudaMemcpy(o_row, d_orow, nx, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(o_col, d_ocol, nx, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(s_row, d_srow, (size_t)(M * Cr), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(s_col, d_scol, (size_t)(Rc * N), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(dbias, d_dbias, (size_t)N * sizeof(float), cudaMemcpyDeviceToHost));

    if (mxo_quantize(x, M, N, MXFP8_E5M2, r_row, rs_row, r_col, rs_col, r_dbias) != 0)
        return 1;
    if (memcmp(o_row, r_row, nx) || memcmp(o_col, r_col, nx) || memcmp(s_row, rs_row, (size_t)(M * Cr)) ||
        memcmp(s_col, rs_col, (size_t)(Rc * N))) {
        fprintf(stderr, "FP8 or scale bytes differ from the oracle\n");
        return 1;
    }
    for (int64_t j = 0; j < N; j++) {
        double abs_sum = 0.0;
        for (int64_t i = 0; i < M; i++)
            abs_sum += fabs(bf16_value(x[i * N + j]));
        if (fabs((double)dbias[j] - (double)r_dbias[j]) > 1e-5 * abs_sum) {
            fprintf(stderr, "dbias[%lld] %g vs %g\n", (long long)j, (double)dbias[j], (double)r_dbias[j]);
            return 1;
        }
    }

    /* host-side rejections, decided before any device work */
    if (mxfp8_quantize(dx, M, 36, MXFP8_E4M3, d_orow, d_srow, d_ocol, d_scol, NULL, NULL, NULL, NULL) !=
            MXFP8_ERR_SHAPE ||
        mxfp8_quantize(dx, M, N, 7, d_orow, d_srow, d_ocol, d_scol, NULL, NULL, NULL, NULL) != MXFP8_ERR_FORMAT ||
        mxfp8_quantize(dx, M, N, MXFP8_E4M3, d_orow, NULL, d_ocol, d_scol, NULL, NULL, NULL, NULL) != MXFP8_ERR_NULL ||
        mxfp8_quantize(dx, M, N, MXFP8_E4M3, d_orow, d_srow, d_ocol, d_scol, d_dbias, NULL, NULL, NULL) !=
            MXFP8_ERR_WORKSPACE) {
        fprintf(stderr, "a rejection returned the wrong status\n");
        return 1;
    }
    if (strlen(mxfp8_status_string(MXFP8_ERR_SHAPE)) == 0)
        return 1;

    cudaStreamDestroy(stream);
    cudaFree(dx);
    cudaFree(d_orow);
    cudaFree(d_ocol);
    cudaFree(d_srow);
    cudaFree(d_scol);
    cudaFree(d_dbias);
    cudaFree(d_ws);
    free(x);
    free(o_row);
    free(o_col);
    free(s_row);
    free(s_col);
    free(r_row);
    free(r_col);
    free(rs_row);
    free(rs_col);
    free(dbias);
    free(r_dbias);
    printf("c consumer ok\n");
    return 0;
}
