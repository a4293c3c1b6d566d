/*
 * CPU oracle for the dense GEMM C = A * B  (bf16 inputs, accumulation in binary64).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or includes
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline do.  It shares no source with the CUDA path.
 *
 * What it computes (the plain definition of the GEMM the pages schedule):
 *   "CUTLASS CLC dynamic persistent kernel", section "From one tile per block to one
 *   worker working continuously": each task is one complete output tile of the GEMM
 *   output matrix, with no split-K or Stream-K.  Scheduling decides only who computes
 *   a tile, never what it holds, so every output element is
 *
 *       C[i][j] = sum_{k = 0 .. K-1} A[i][k] * B[k][j]
 *
 *   with A row-major M x K and B row-major K x N (element (k, j) of B at k*N + j),
 *   both stored as IEEE bfloat16 bit patterns (the upper 16 bits of a binary32).
 *
 * Arithmetic: each bf16 value is widened exactly to double; a product of two bf16
 * values (8-bit significands) is exact in double; the sum is taken in double in
 * ascending k.  There is no blocking, no reordering of the k sum and no fused
 * multiply-add contraction (the file is compiled with -ffp-contract=off).
 * OpenMP only splits output rows across threads; each element's sum is computed by
 * one thread in the same order whatever the thread count.
 */
#include <stdint.h>
#include <string.h>

/* bfloat16 -> double: the 16 stored bits are the high half of a binary32 value. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Decode an array of bf16 bit patterns (used by the pins on the decoder itself). */
void oracle_bf16_decode(int64_t n, const uint16_t *src, double *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = bf16_bits_to_double(src[i]);
}

/*
 * One block of the output: rows [r0, r1) and columns [c0, c1) of C = A * B, written
 * row-major into out, which holds (r1 - r0) * (c1 - c0) doubles.  A is M x K and B is
 * K x N, both row-major bf16 bit patterns.  The full product is the block
 * [0, M) x [0, N); a single element is a 1 x 1 block.
 */
void oracle_gemm_block(int64_t M, int64_t N, int64_t K,
                       const uint16_t *A, const uint16_t *B,
                       int64_t r0, int64_t r1, int64_t c0, int64_t c1,
                       double *out)
{
    const int64_t w = c1 - c0;
    (void)M;
#pragma omp parallel for schedule(static)
    for (int64_t i = r0; i < r1; ++i) {
        double *c = out + (i - r0) * w;
        for (int64_t j = 0; j < w; ++j)
            c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = bf16_bits_to_double(A[i * K + k]);
            const uint16_t *brow = B + k * N;
            for (int64_t j = c0; j < c1; ++j)
                c[j - c0] += a * bf16_bits_to_double(brow[j]);
        }
    }
}

/* The whole product: C (M x N doubles, row-major). */
void oracle_gemm(int64_t M, int64_t N, int64_t K,
                 const uint16_t *A, const uint16_t *B, double *C)
{
    oracle_gemm_block(M, N, K, A, B, 0, M, 0, N, C);
}

/*
 * Scattered single elements: out[e] = C[rows[e]][cols[e]] for e < n.  Each element is
 * the same ascending-k double sum as above.
 */
void oracle_gemm_entries(int64_t M, int64_t N, int64_t K,
                         const uint16_t *A, const uint16_t *B,
                         int64_t n, const int64_t *rows, const int64_t *cols,
                         double *out)
{
    (void)M;
#pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < n; ++e) {
        const int64_t i = rows[e], j = cols[e];
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += bf16_bits_to_double(A[i * K + k]) * bf16_bits_to_double(B[k * N + j]);
        out[e] = s;
    }
}

/* Number of threads OpenMP will use for the loops above (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
#else
int oracle_num_threads(void) { return 1; }
#endif
