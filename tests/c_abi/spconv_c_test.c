/*
 * Plain-C test of the libspconv C ABI (no Python, no PyTorch): packs a small
 * seeded layer, checks the host-side introspection and error statuses, and --
 * unless run with --host-only -- runs spconv_forward on the GPU and compares
 * every output with the CPU oracle (oracle_csr, fp64, linked from
 * oracle/liboracle.so) under |gpu - oracle| <= 1e-5 * sum|w*x| + 1e-7.
 * Exit status 0 = pass.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "spconv.h"

int oracle_csr(int N, int C, int H, int W, int M, int R, int S, int stride, int pad,
               const int32_t *rowptr, const int32_t *colidx, const double *value,
               const double *x, double *y, double *abs_sum, int nthreads);

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;
static double urand(void) { /* xorshift64*, uniform in [0, 1) */
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    return (double)((rng_state * 2685821657736338717ull) >> 11) / 9007199254740992.0;
}

#define CHECK(cond, msg)                                                     \
    do {                                                                     \
        if (!(cond)) {                                                       \
            fprintf(stderr, "FAIL %s:%d: %s\n", __FILE__, __LINE__, (msg)); \
            return 1;                                                        \
        }                                                                    \
    } while (0)

int main(int argc, char **argv) {
    const int host_only = argc > 1 && strcmp(argv[1], "--host-only") == 0;
    const int N = 2, C = 24, H = 19, W = 21, M = 40, R = 3, S = 3, stride = 1, pad = 1;
    const int CRS = C * R * S;
    const int E = (H + 2 * pad - R) / stride + 1, F = (W + 2 * pad - S) / stride + 1;
    int32_t *rowptr = malloc(sizeof(int32_t) * (M + 1));
    int32_t *colidx = malloc(sizeof(int32_t) * M * CRS);
    float *value = malloc(sizeof(float) * M * CRS);
    int32_t nnz = 0;
    rowptr[0] = 0;
    for (int m = 0; m < M; ++m) {
        for (int k = 0; k < CRS; ++k)
            if (urand() < 0.1) {
                colidx[nnz] = k;
                value[nnz] = (float)(urand() - 0.5);
                ++nnz;
            }
        rowptr[m + 1] = nnz;
    }

    /* host-only packing, introspection, statuses */
    spconv_packed *hp = NULL;
    CHECK(spconv_pack_host(C, H, W, M, R, S, stride, pad, rowptr, colidx, value, &hp) == SPCONV_OK,
          "pack_host");
    spconv_packed_info info;
    CHECK(spconv_packed_info_get(hp, &info) == SPCONV_OK, "info");
    CHECK(info.nnz == nnz && info.E == E && info.F == F && info.on_device == 0, "info fields");
    CHECK(spconv_forward(N, C, H, W, M, R, S, stride, pad, NULL, hp, NULL, NULL) ==
              SPCONV_ERR_MISMATCH, "host-only handle rejected by forward");
    CHECK(spconv_forward_host(N, C, H, W, M, R, S, stride, pad, NULL, hp, NULL, SPCONV_ACT_NONE,
                              NULL, NULL, NULL, NULL) == SPCONV_ERR_MISMATCH,
          "host-only handle rejected by forward_host");
    spconv_packed_free(hp);
    spconv_packed_free(NULL);
    CHECK(spconv_pack_host(0, H, W, M, R, S, stride, pad, rowptr, colidx, value, &hp) ==
              SPCONV_ERR_INVALID_ARG, "C = 0 rejected");
    CHECK(strlen(spconv_status_string(SPCONV_ERR_BAD_CSR)) > 0, "status string");
    if (host_only) {
        printf("host-only ok (nnz %d)\n", nnz);
        return 0;
    }

    /* device: pack, forward, compare with the oracle */
    spconv_packed *dp = NULL;
    CHECK(spconv_pack(C, H, W, M, R, S, stride, pad, rowptr, colidx, value, NULL, &dp) ==
              SPCONV_OK, "pack");
    const size_t nx = (size_t)N * C * H * W, ny = (size_t)N * M * E * F;
    float *hx = malloc(nx * sizeof(float)), *hy = malloc(ny * sizeof(float));
    for (size_t i = 0; i < nx; ++i) hx[i] = (float)fmax(0.0, urand() * 2.0 - 0.6);
    float *dx = NULL, *dy = NULL;
    CHECK(cudaMalloc((void **)&dx, nx * sizeof(float)) == cudaSuccess, "cudaMalloc x");
    CHECK(cudaMalloc((void **)&dy, ny * sizeof(float)) == cudaSuccess, "cudaMalloc y");
    CHECK(cudaMemcpy(dx, hx, nx * sizeof(float), cudaMemcpyHostToDevice) == cudaSuccess, "H2D");
    CHECK(spconv_forward(N, C, H, W, M, R, S, stride, pad, dx, dp, dy, NULL) == SPCONV_OK,
          "forward");
    CHECK(cudaMemcpy(hy, dy, ny * sizeof(float), cudaMemcpyDeviceToHost) == cudaSuccess, "D2H");
    int32_t flags = -1;
    CHECK(spconv_device_status(dp, NULL, &flags) == SPCONV_OK && flags == 0, "device status");

    double *xv = malloc(nx * sizeof(double)), *vv = malloc((size_t)nnz * sizeof(double));
    double *ref = malloc(ny * sizeof(double)), *mag = malloc(ny * sizeof(double));
    for (size_t i = 0; i < nx; ++i) xv[i] = hx[i];
    for (int j = 0; j < nnz; ++j) vv[j] = value[j];
    CHECK(oracle_csr(N, C, H, W, M, R, S, stride, pad, rowptr, colidx, vv, xv, ref, mag, 0) >= 1,
          "oracle");
    size_t bad = 0;
    for (size_t i = 0; i < ny; ++i)
        if (!(fabs((double)hy[i] - ref[i]) <= 1e-5 * mag[i] + 1e-7)) ++bad;
    printf("forward checked %zu outputs, %zu out of tolerance\n", ny, bad);
    CHECK(bad == 0, "parity");

    /* host buffers: page-locked (device-mapped path) and pageable (copy path);
     * the same kernel on the same data gives the same bits */
    float *px = NULL, *py = NULL;
    CHECK(cudaHostAlloc((void **)&px, nx * sizeof(float), cudaHostAllocDefault) == cudaSuccess,
          "cudaHostAlloc x");
    CHECK(cudaHostAlloc((void **)&py, ny * sizeof(float), cudaHostAllocDefault) == cudaSuccess,
          "cudaHostAlloc y");
    memcpy(px, hx, nx * sizeof(float));
    float *gy = malloc(ny * sizeof(float));
    for (int pass = 0; pass < 2; ++pass) {
        float *in = pass == 0 ? px : hx, *out = pass == 0 ? py : gy;
        for (size_t i = 0; i < ny; ++i) out[i] = -1.0f;
        CHECK(spconv_forward_host(N, C, H, W, M, R, S, stride, pad, in, dp, NULL,
                                  SPCONV_ACT_NONE, out, dx, dy, NULL) == SPCONV_OK,
              "forward_host");
        CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
        CHECK(memcmp(out, hy, ny * sizeof(float)) == 0, "forward_host equals forward");
    }
    printf("forward_host matched forward (page-locked and pageable buffers)\n");
    cudaFreeHost(px);
    cudaFreeHost(py);
    free(gy);
    spconv_packed_free(dp);
    cudaFree(dx);
    cudaFree(dy);
    return 0;
}
