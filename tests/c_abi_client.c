/* A plain C client of the library: device buffers from the CUDA runtime, the GEMM through
 * the C ABI, the result checked against the CPU oracle's C entry point.  Built and run by
 * tests/test_c_client.py (test infrastructure: it links the oracle). */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "clcgemm.h"

void oracle_gemm(int64_t M, int64_t N, int64_t K, const uint16_t *A, const uint16_t *B, double *C);

/* small integers are exact in bf16: the high half of the binary32 pattern */
static uint16_t bf16_of_int(int v) {
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

#define CHECK(x) do { int rc_ = (x); if (rc_ != GEMM_OK) { \
    fprintf(stderr, "%s -> %d (%s)\n", #x, rc_, gemm_strerror(rc_)); return 1; } } while (0)
#define CUDA(x) do { if ((x) != cudaSuccess) { fprintf(stderr, "%s failed\n", #x); return 1; } } while (0)

static int compare(const float *c, const double *ref, int64_t n) {
    for (int64_t i = 0; i < n; ++i)
        if ((double)c[i] != ref[i]) {
            fprintf(stderr, "element %lld: %f != %f\n", (long long)i, c[i], ref[i]);
            return 1;
        }
    return 0;
}

int main(void) {
    const int64_t M = 1000, N = 776, K = 520;
    uint16_t *A = malloc(sizeof(uint16_t) * M * K), *B = malloc(sizeof(uint16_t) * K * N);
    float *C = malloc(sizeof(float) * M * N);
    double *ref = malloc(sizeof(double) * M * N);
    int32_t *owner, *claims, *first;
    for (int64_t i = 0; i < M * K; ++i) A[i] = bf16_of_int((int)((i * 7 + 3) % 9) - 4);
    for (int64_t i = 0; i < K * N; ++i) B[i] = bf16_of_int((int)((i * 5 + 1) % 9) - 4);
    oracle_gemm(M, N, K, A, B, ref);

    void *dA, *dB, *dC;
    CUDA(cudaMalloc(&dA, sizeof(uint16_t) * M * K));
    CUDA(cudaMalloc(&dB, sizeof(uint16_t) * K * N));
    CUDA(cudaMalloc(&dC, sizeof(float) * M * N));
    CUDA(cudaMemcpy(dA, A, sizeof(uint16_t) * M * K, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(dB, B, sizeof(uint16_t) * K * N, cudaMemcpyHostToDevice));

    gemm_handle_t h = NULL;
    gemm_opts_t opts;
    gemm_opts_default(&opts);
    CHECK(gemm_create(0, &opts, &h));
    const gemm_tile_t tile = {128, 256, 64};
    const gemm_cluster_t one = {1, 1, 1};
    const gemm_sched_t scheds[3] = {GEMM_SCHED_CLC, GEMM_SCHED_STATIC, GEMM_SCHED_NONPERSISTENT};
    for (int s = 0; s < 3; ++s) {
        CUDA(cudaMemset(dC, 0xFF, sizeof(float) * M * N));   /* NaN pattern */
        CHECK(gemm_run(h, M, N, K, dA, dB, (float *)dC, tile, one, scheds[s], 0, NULL));
        CHECK(gemm_sync(h, NULL));
        CUDA(cudaMemcpy(C, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost));
        if (compare(C, ref, M * N)) return 1;
        gemm_launch_info_t info;
        CHECK(gemm_last_launch(h, &info));
        owner = malloc(sizeof(int32_t) * info.n_tiles);
        claims = malloc(sizeof(int32_t) * info.n_tiles);
        first = malloc(sizeof(int32_t) * info.n_workers);
        CHECK(gemm_get_log(h, owner, claims, first, info.n_tiles, info.n_workers));
        for (int64_t t = 0; t < info.n_tiles; ++t)
            if (claims[t] != 1) { fprintf(stderr, "tile %lld claimed %d times\n", (long long)t, claims[t]); return 1; }
        free(owner); free(claims); free(first);
    }
    /* host buffers, copies inside the call */
    memset(C, 0, sizeof(float) * M * N);
    CHECK(gemm_run_host(h, M, N, K, A, B, C, tile, one, GEMM_SCHED_CLC, 0, NULL));
    CHECK(gemm_sync(h, NULL));
    if (compare(C, ref, M * N)) return 1;
    /* no handle, no allocation */
    CUDA(cudaMemset(dC, 0xFF, sizeof(float) * M * N));
    CHECK(gemm_run_noalloc(M, N, K, dA, dB, (float *)dC, tile, one, GEMM_SCHED_CLC, 0, NULL));
    CUDA(cudaDeviceSynchronize());
    CUDA(cudaMemcpy(C, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost));
    if (compare(C, ref, M * N)) return 1;
    /* argument errors come back as codes */
    if (gemm_run(h, M, N, 60, dA, dB, (float *)dC, tile, one, GEMM_SCHED_CLC, 0, NULL) != GEMM_ERR_ALIGNMENT) return 1;
    gemm_destroy(h);
    cudaFree(dA); cudaFree(dB); cudaFree(dC);
    printf("C client ok\n");
    return 0;
}
