/* The C ABI used from plain C, with no Python in the process: a caller packs
 * a seeded 4-bit layer on the device with w4a16_pack, runs w4a16_linear at
 * M = 4 and reads y back.  The packed words must equal the oracle's pack bit
 * for bit, and y must be within |y - y_ref| <= 1e-3 * max|y_ref| + 1e-3 of the
 * oracle's binary64 linear.  Test infrastructure: it links the oracle.
 * Exit status 0 on success. */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "w4a16.h"

/* the oracle (oracle/w4a16_oracle.c) */
void w4o_pack(const uint8_t *q, const uint8_t *z, int N, int K, int group, uint32_t *qweight,
              uint32_t *zeros);
void w4o_linear_dt(const uint16_t *x, const uint32_t *qweight, const uint16_t *scales,
                   const uint32_t *zeros, int M, int N, int K, int group, int dtype, double *y,
                   int nthreads);
uint16_t w4o_double_to_half(double v);
double w4o_half_to_double(uint16_t h);

static uint64_t g_state = 0x9e3779b97f4a7c15ull;
static uint32_t next_u32(void) { /* 64-bit LCG, high word */
    g_state = g_state * 6364136223846793005ull + 1442695040888963407ull;
    return (uint32_t)(g_state >> 32);
}
static double next_unit(void) { return (next_u32() >> 8) * (1.0 / 16777216.0); }

#define CHECK_CUDA(call)                                                            \
    do {                                                                            \
        cudaError_t e_ = (call);                                                    \
        if (e_ != cudaSuccess) {                                                    \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));             \
            return 2;                                                               \
        }                                                                           \
    } while (0)
#define CHECK_W4(call)                                                              \
    do {                                                                            \
        int s_ = (call);                                                            \
        if (s_ != W4A16_OK) {                                                       \
            fprintf(stderr, "%s: %s\n", #call, w4a16_status_string(s_));            \
            return 3;                                                               \
        }                                                                           \
    } while (0)

int main(void) {
    const int M = 4, N = 1000, K = 2048, group = 128, G = K / group, ZW = (G + 7) / 8;
    uint8_t *q = malloc((size_t)N * K), *z = malloc((size_t)N * G);
    uint16_t *s = malloc((size_t)N * G * 2), *x = malloc((size_t)M * K * 2);
    uint16_t *y = malloc((size_t)M * N * 2);
    uint32_t *qw = malloc((size_t)N * K / 2), *zw = malloc((size_t)N * ZW * 4);
    uint32_t *qw_dev_copy = malloc((size_t)N * K / 2), *zw_dev_copy = malloc((size_t)N * ZW * 4);
    double *y_ref = malloc((size_t)M * N * sizeof(double));
    for (long i = 0; i < (long)N * K; ++i) q[i] = (uint8_t)(next_u32() & 15u);
    for (long i = 0; i < (long)N * G; ++i) z[i] = (uint8_t)(next_u32() & 15u);
    for (long i = 0; i < (long)N * G; ++i) s[i] = w4o_double_to_half(0.002 + 0.018 * next_unit());
    for (long i = 0; i < (long)M * K; ++i) x[i] = w4o_double_to_half(2.0 * next_unit() - 1.0);

    uint8_t *d_q, *d_z;
    uint16_t *d_s, *d_x, *d_y;
    uint32_t *d_qw, *d_zw;
    CHECK_CUDA(cudaMalloc((void **)&d_q, (size_t)N * K));
    CHECK_CUDA(cudaMalloc((void **)&d_z, (size_t)N * G));
    CHECK_CUDA(cudaMalloc((void **)&d_s, (size_t)N * G * 2));
    CHECK_CUDA(cudaMalloc((void **)&d_x, (size_t)M * K * 2));
    CHECK_CUDA(cudaMalloc((void **)&d_y, (size_t)M * N * 2));
    CHECK_CUDA(cudaMalloc((void **)&d_qw, (size_t)N * K / 2));
    CHECK_CUDA(cudaMalloc((void **)&d_zw, (size_t)N * ZW * 4));
    CHECK_CUDA(cudaMemcpy(d_q, q, (size_t)N * K, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_z, z, (size_t)N * G, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_s, s, (size_t)N * G * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(d_x, x, (size_t)M * K * 2, cudaMemcpyHostToDevice));

    CHECK_W4(w4a16_init(0, (size_t)64 << 20));
    CHECK_W4(w4a16_pack(d_q, d_z, N, K, group, d_qw, d_zw, NULL));
    CHECK_W4(w4a16_linear(d_x, d_qw, d_s, d_zw, M, N, K, group, d_y, NULL));
    CHECK_CUDA(cudaDeviceSynchronize());
    int code = 0;
    CHECK_W4(w4a16_device_status(NULL, &code));
    CHECK_CUDA(cudaMemcpy(y, d_y, (size_t)M * N * 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(qw_dev_copy, d_qw, (size_t)N * K / 2, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(zw_dev_copy, d_zw, (size_t)N * ZW * 4, cudaMemcpyDeviceToHost));

    w4o_pack(q, z, N, K, group, qw, zw);
    if (memcmp(qw, qw_dev_copy, (size_t)N * K / 2) != 0 || memcmp(zw, zw_dev_copy, (size_t)N * ZW * 4) != 0) {
        fprintf(stderr, "packed words differ from the oracle's pack\n");
        return 4;
    }
    w4o_linear_dt(x, qw, s, zw, M, N, K, group, 0, y_ref, 1);
    double ymax = 0.0, err = 0.0;
    for (long i = 0; i < (long)M * N; ++i) ymax = fmax(ymax, fabs(y_ref[i]));
    const double tol = 1e-3 * ymax + 1e-3;
    long bad = 0;
    for (long i = 0; i < (long)M * N; ++i) {
        const double d = fabs(w4o_half_to_double(y[i]) - y_ref[i]);
        if (!(d <= tol)) ++bad;
        if (d > err) err = d;
    }
    CHECK_W4(w4a16_shutdown());
    printf("c abi %s: rung %s, max |err| %.3e, tol %.3e, %ld outside\n", bad ? "FAILED" : "ok",
           w4a16_rung_name(w4a16_select_rung(M, N, K, group)), err, tol, bad);
    return bad ? 5 : 0;
}
