/*
 * Oracle for single-precision GEMM, C = alpha * A * B + beta * C.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plainly correct CPU
 * definition that the CUDA library is checked against.  Only the tests, the
 * package's smoke check and the CPU-baseline leg of the benchmark may load it;
 * the library itself never calls it and shares no code with it.
 *
 * What it computes (the definition on the page "Deep dive into the sgemmNN
 * algorithm" (lazypool blog, cuda-sgemmnn), section "Why SGEMM matters": A is
 * m x k, B is k x n, C is m x n, alpha and beta are scalars):
 *
 *     C[i][j] <- alpha * sum_{p=0}^{K-1} A[i][p] * B[p][j] + beta * C[i][j]
 *
 * Storage is row-major with leading dimensions, as in the row-major indexing
 * A[row*K + k], B[k*N + col] of the naive kernel on page m.lqnn.cn/news/94381
 * section 1.1:
 *     A[i*lda + p], B[p*ldb + j], C[i*ldc + j].
 *
 * Arithmetic: every product of two floats is formed in double (exact: 24+24
 * significand bits fit in 53), the K products of one output are summed in
 * double in ascending p, alpha and beta are applied in double, and the result
 * is rounded once to float (round to nearest even).  Cells outside the M x K,
 * K x N and M x N windows (leading-dimension padding) are never read or
 * written.
 *
 * BLAS conventions where the pages are silent: when alpha == 0 or K == 0 the
 * product term is absent and A, B are not read; when beta == 0 the C term is
 * absent and C is not read (so NaN in an output-only C does not propagate).
 *
 * Loop order is i -> p -> j with one double accumulator per output of the
 * current row: for every (i, j) the additions still happen in ascending p, so
 * the result equals the textbook i -> j -> p triple loop bit for bit.  Rows are
 * independent and are spread over OpenMP threads; the result does not depend
 * on the thread count.
 *
 * Build: gcc -O3 -fopenmp -ffp-contract=off (no -ffast-math: the summation
 * order and the two separate roundings of alpha*s and beta*c are part of the
 * definition written above).
 */
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One output row in double: acc[j] = alpha * sum_p A[i][p] B[p][j] + beta * c0[j].
 * `c0` may be NULL when beta == 0. */
static void row_f64(int N, int K, double alpha, const float *Arow,
                    const float *B, int64_t ldb, double beta, const float *c0,
                    double *acc)
{
    for (int j = 0; j < N; ++j)
        acc[j] = 0.0;
    if (alpha != 0.0 && K > 0) {
        for (int p = 0; p < K; ++p) {
            const double a = (double)Arow[p];
            const float *Bp = B + (int64_t)p * ldb;
            for (int j = 0; j < N; ++j)
                acc[j] += a * (double)Bp[j];
        }
        for (int j = 0; j < N; ++j)
            acc[j] = alpha * acc[j];
    }
    if (beta != 0.0) {
        for (int j = 0; j < N; ++j)
            acc[j] = acc[j] + beta * (double)c0[j];
    }
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure. */
static int check(int M, int N, int K, int64_t lda, int64_t ldb, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0)
        return -1;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
        return -1;
    return 0;
}

/* In-place float result: C <- (float)(alpha*A*B + beta*C). */
int oracle_sgemm(int M, int N, int K, float alpha, const float *A, int64_t lda,
                 const float *B, int64_t ldb, float beta, float *C, int64_t ldc)
{
    if (check(M, N, K, lda, ldb, ldc))
        return -1;
    if (M == 0 || N == 0)
        return 0;
    int status = 0;
#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            status = -2;
        }
#pragma omp for schedule(dynamic, 1)
        for (int i = 0; i < M; ++i) {
            if (!acc)
                continue;
            float *Ci = C + (int64_t)i * ldc;
            row_f64(N, K, (double)alpha, A + (int64_t)i * lda, B, ldb,
                    (double)beta, Ci, acc);
            for (int j = 0; j < N; ++j)
                Ci[j] = (float)acc[j];
        }
        free(acc);
    }
    return status;
}

/* Unrounded double result into a separate array: D = alpha*A*B + beta*C0. */
int oracle_sgemm_f64(int M, int N, int K, float alpha, const float *A,
                     int64_t lda, const float *B, int64_t ldb, float beta,
                     const float *C0, int64_t ldc0, double *D, int64_t ldd)
{
    if (check(M, N, K, lda, ldb, ldc0) || ldd < (N > 1 ? N : 1))
        return -1;
    if (beta != 0.0f && C0 == NULL)
        return -1;
    if (M == 0 || N == 0)
        return 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < M; ++i)
        row_f64(N, K, (double)alpha, A + (int64_t)i * lda, B, ldb, (double)beta,
                C0 ? C0 + (int64_t)i * ldc0 : NULL, D + (int64_t)i * ldd);
    return 0;
}

/* Threads an OpenMP parallel region of this library uses by default. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}
