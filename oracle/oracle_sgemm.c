/*
 * oracle_sgemm.c -- the CPU oracle for single-precision GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg call this code.  The library's GPU path shares
 * no code, header, table or helper with it, and never calls it.
 *
 * What it computes (the plain definition, no blocking, fusion or reordering):
 *
 *   C_ref[q,i,j] = alpha * S[q,i,j] + beta * C0[q,i,j]
 *   S[q,i,j]     = sum over k < K of opA[q,i,k] * opB[q,k,j]
 *
 * following "From 1% to 94% of cuBLAS, one kernel at a time"
 * (arpit2412.github.io/blog/cuda-sgemm.html): the SGEMM definition
 * "C = alpha * A @ B + beta * C" with A M x K, B K x N, C M x N, and the
 * first kernel's per-element rule (one dot product of a row of A with a
 * column of B, of length K, then alpha*acc + beta*C); row-major storage,
 * element (r, c) at r * ld + c, from the same page's storage paragraph.
 * Transposed operands follow "Triton Optimization Reference (cuTile ->
 * Triton)", section 2 (transpose by pointer strides), and the batch index q
 * with a per-batch stride follows its sections 2-3.
 *
 * Readings taken where the pages are silent:
 *  - transA: A is stored K x M row-major, element (i,k) at A[k*lda + i];
 *    transB: B is stored N x K row-major, element (k,j) at B[j*ldb + k].
 *  - beta == 0: C0 is not read (BLAS convention), so NaN/Inf in C0 do not
 *    reach the result.
 *  - alpha == 0 or K == 0: C_ref = beta * C0 (0 when beta == 0); A and B are
 *    not read.
 *  - batch strides count elements; a stride of 0 broadcasts that operand.
 *
 * Precision: every fp32 input is promoted exactly to fp64; each product of two
 * fp32 values is exact in fp64; the K-long sum is accumulated in fp64 in
 * increasing k.  C_ref is returned in fp64, not rounded to fp32.
 *
 * It also returns, for the accuracy metric,
 *   D[q,i,j] = |alpha| * sum_k |opA[q,i,k] * opB[q,k,j]| + |beta * C0[q,i,j]|
 * (the second term only when beta != 0), the magnitude against which the
 * error of a floating-point result is measured.
 *
 * Form: a triple loop in i-k-j order, one fp64 accumulator row per output
 * row, output rows spread over OpenMP threads when OpenMP is available.
 * Compiled with -O2 -ffp-contract=off (no fused multiply-add, no fast-math),
 * so the result is the same on x86-64 and aarch64.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef long long i64;

static double opA(const float *A, int transA, i64 lda, i64 i, i64 k)
{
    return transA ? (double)A[k * lda + i] : (double)A[i * lda + k];
}

static double opB(const float *B, int transB, i64 ldb, i64 k, i64 j)
{
    return transB ? (double)B[j * ldb + k] : (double)B[k * ldb + j];
}

/* One output row (q, i): writes N values of C_ref and D. */
static void one_row(int transA, int transB, i64 N, i64 K, double alpha,
                    const float *Aq, i64 lda, const float *Bq, i64 ldb,
                    double beta, const float *C0row, i64 i,
                    double *acc, double *mag, double *Cref_row, double *D_row)
{
    i64 j, k;
    for (j = 0; j < N; ++j) { acc[j] = 0.0; mag[j] = 0.0; }
    if (alpha != 0.0) {
        for (k = 0; k < K; ++k) {
            double a = opA(Aq, transA, lda, i, k);
            for (j = 0; j < N; ++j) {
                double p = a * opB(Bq, transB, ldb, k, j);
                acc[j] += p;
                mag[j] += fabs(p);
            }
        }
    }
    for (j = 0; j < N; ++j) {
        double c = 0.0, cm = 0.0;
        if (beta != 0.0) {
            c = beta * (double)C0row[j];
            cm = fabs(c);
        }
        if (alpha != 0.0) {
            Cref_row[j] = alpha * acc[j] + c;
            D_row[j] = fabs(alpha) * mag[j] + cm;
        } else {
            Cref_row[j] = c;
            D_row[j] = cm;
        }
    }
}

/*
 * oracle_sgemm: see the file header for the definition.
 *
 * A, B, C0 are host arrays; operand q starts at q*strideX.  C0 may be NULL
 * when beta == 0.  If rows == NULL, every (q, i) is computed and
 * Cref/D are Q*M*N packed, index (q*M + i)*N + j.  Otherwise rows holds nrows
 * (q, i) pairs (rows[2r], rows[2r+1]) and output row r is at r*N.
 * Returns 0, or -1 on an invalid argument or allocation failure.
 */
int oracle_sgemm(int transA, int transB, i64 M, i64 N, i64 K, float alpha,
                 const float *A, i64 lda, i64 strideA,
                 const float *B, i64 ldb, i64 strideB,
                 float beta, const float *C0, i64 ldc, i64 strideC, i64 Q,
                 const i64 *rows, i64 nrows, double *Cref, double *D)
{
    i64 total, r;
    int bad = 0;
    double a64 = (double)alpha, b64 = (double)beta;
    if (M < 0 || N < 0 || K < 0 || Q < 0) return -1;
    if (beta != 0.0f && C0 == NULL) return -1;
    if (K == 0) a64 = 0.0; /* C = beta * C0 */
    total = rows ? nrows : Q * M;
    if (N == 0 || total == 0) return 0;

#ifdef _OPENMP
#pragma omp parallel reduction(|:bad)
#endif
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)N);
        double *mag = (double *)malloc(sizeof(double) * (size_t)N);
        if (!acc || !mag) {
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (r = 0; r < total; ++r) {
                i64 q = rows ? rows[2 * r] : r / M;
                i64 i = rows ? rows[2 * r + 1] : r % M;
                const float *C0row = C0 ? C0 + q * strideC + i * ldc : NULL;
                one_row(transA, transB, N, K, a64, A + q * strideA, lda,
                        B + q * strideB, ldb, b64, C0row, i, acc, mag,
                        Cref + r * N, D + r * N);
            }
        }
        free(acc);
        free(mag);
    }
    return bad ? -1 : 0;
}

/* Number of threads the oracle's parallel loop uses. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
