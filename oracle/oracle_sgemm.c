/*
 * oracle_sgemm.c -- CPU oracle for the single-precision GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls
 * this file; only the tests, the package's smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes (plain definition, no blocking, fusion or reordering):
 *
 *   C[i][j] = fl32( alpha * S[i][j] + beta * C0[i][j] ),
 *   S[i][j] = sum_{k=0}^{K-1} A[i*lda + k] * B[k*ldb + j]
 *
 * - "Micro_gemm_4x4 - cuBLAS micro GEMM skeleton", section 2 (kernel
 *   signature: C = alpha*A*B + beta*C on (M,K), (K,N), (M,N) operands) and
 *   section 9 (final C write: beta == 0 means the old C is not read).
 * - velog @levelstage "AutoMinepp4", section "현재 알고리즘" (each C entry is
 *   the inner product of a row of A and a column of B).
 * - "GPU Target" (MLIR tutorial), section "타일링된 행렬 곱셈": operands carry
 *   dynamic strides, realised here as the leading dimensions lda/ldb/ldc.
 *
 * Arithmetic: S is accumulated in IEEE double in ascending k.  A product of two
 * floats is exact in double (24+24 significant bits <= 53), so the only
 * roundings before the final one are the K-1 double additions.  alpha*S and
 * beta*C0 are formed in double and the sum is rounded once to float
 * (round-to-nearest-even).  When alpha == 0 or K == 0 the product term is 0 and
 * A and B are not read; when beta == 0 the C0 term is dropped and C0 is not
 * read (BLAS convention; the pages are silent on alpha == 0 and K == 0).
 *
 * Loop order: i over rows (OpenMP-parallel), then k, then j, with a double row
 * accumulator, so every S[i][j] still sums in ascending k.
 *
 * Compile with -ffp-contract=off and without -ffast-math so the double
 * arithmetic is plain IEEE on every host.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static void oracle_row(int64_t i, int64_t N, int64_t K, float alpha,
                       const float *A, int64_t lda, const float *B, int64_t ldb,
                       float beta, const float *C0, int64_t ldc0,
                       double *acc, float *out)
{
    for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
    if (alpha != 0.0f) {
        for (int64_t k = 0; k < K; ++k) {
            const double a = (double)A[i * lda + k];
            const float *brow = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) acc[j] += a * (double)brow[j];
        }
    }
    for (int64_t j = 0; j < N; ++j) {
        double v = (alpha != 0.0f) ? (double)alpha * acc[j] : 0.0;
        if (beta != 0.0f) v += (double)beta * (double)C0[i * ldc0 + j];
        out[j] = (float)v;
    }
}

/* Number of OpenMP threads a parallel oracle call uses (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Selected rows: out[r*N + j] = C[rows[r]][j].  nthreads <= 0 means all. */
int oracle_sgemm_rows(int64_t M, int64_t N, int64_t K, float alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      float beta, const float *C0, int64_t ldc0,
                      const int64_t *rows, int64_t nrows, float *out,
                      int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return 1;
    if (N == 0 || nrows == 0) return 0;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
#endif
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (!acc) {
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t r = 0; r < nrows; ++r) {
                const int64_t i = rows[r];
                if (i < 0 || i >= M) { bad = 1; continue; }
                oracle_row(i, N, K, alpha, A, lda, B, ldb, beta, C0, ldc0, acc,
                           out + r * N);
            }
            free(acc);
        }
    }
    return bad;
}

/* Full product: C[i*ldc + j] for 0<=i<M, 0<=j<N; C's padding columns are not
 * touched. */
int oracle_sgemm(int64_t M, int64_t N, int64_t K, float alpha,
                 const float *A, int64_t lda, const float *B, int64_t ldb,
                 float beta, const float *C0, int64_t ldc0,
                 float *C, int64_t ldc, int nthreads)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (M == 0 || N == 0) return 0;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
#endif
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (!acc) {
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (int64_t i = 0; i < M; ++i)
                oracle_row(i, N, K, alpha, A, lda, B, ldb, beta, C0, ldc0, acc,
                           C + i * ldc);
            free(acc);
        }
    }
    return bad;
}

/* Selected entries, each as one inner product (ascending k, double):
 * out[t] = C[ii[t]][jj[t]]. */
int oracle_sgemm_entries(int64_t M, int64_t N, int64_t K, float alpha,
                         const float *A, int64_t lda, const float *B, int64_t ldb,
                         float beta, const float *C0, int64_t ldc0,
                         const int64_t *ii, const int64_t *jj, int64_t n,
                         float *out)
{
    int bad = 0;
    for (int64_t t = 0; t < n; ++t) {
        const int64_t i = ii[t], j = jj[t];
        if (i < 0 || i >= M || j < 0 || j >= N) { bad = 1; out[t] = 0.0f; continue; }
        double s = 0.0;
        if (alpha != 0.0f)
            for (int64_t k = 0; k < K; ++k)
                s += (double)A[i * lda + k] * (double)B[k * ldb + j];
        double v = (alpha != 0.0f) ? (double)alpha * s : 0.0;
        if (beta != 0.0f) v += (double)beta * (double)C0[i * ldc0 + j];
        out[t] = (float)v;
    }
    return bad;
}

/*
 * The general form, for b in [0, batch):
 *
 *   C_b[i][j] = fl32( act( alpha * S_b[i][j] + beta * C0_b[i][j] + bias[j] ) )
 *   S_b[i][j] = sum_k opA_b[i][k] * opB_b[k][j]
 *   opA_b[i][k] = A[b*sa + i*lda + k]  (op_a = 0)   or  A[b*sa + k*lda + i]  (op_a = 1)
 *   opB_b[k][j] = B[b*sb + k*ldb + j]  (op_b = 0)   or  B[b*sb + j*ldb + k]  (op_b = 1)
 *
 * - "GPU Target" (MLIR tutorial), section "타일링된 행렬 곱셈": the batched
 *   variant indexes a third dimension by batch (per attention head), and
 *   operands are strided views (a transposed matrix is a view with swapped
 *   strides).
 * - "GPU Target", GPT-2 sublayers: a projection is x @ W + b; the MLP applies
 *   GELU in its tanh form, 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
 *   act = 0: none, act = 1: that GELU.  bias == NULL: no bias.
 * Everything in double, one final rounding to float; S in ascending k.  The
 * same special cases as oracle_sgemm (alpha == 0 or K == 0: A and B not
 * read; beta == 0: C0 not read).  Output: C[b*M*N + i*N + j] (dense).
 */
static double oracle_gelu_tanh(double x)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

int oracle_sgemm_ex(int op_a, int op_b, int64_t M, int64_t N, int64_t K, float alpha,
                    const float *A, int64_t lda, int64_t sa, const float *B, int64_t ldb,
                    int64_t sb, float beta, const float *C0, int64_t ldc0, int64_t sc,
                    int64_t batch, const float *bias, int act, float *C, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || batch < 0) return 1;
    if (M == 0 || N == 0 || batch == 0) return 0;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads) reduction(| : bad)
#endif
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (!acc) {
            bad = 1;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1) collapse(2)
#endif
            for (int64_t b = 0; b < batch; ++b) {
                for (int64_t i = 0; i < M; ++i) {
                    const float *Ab = A + b * sa;
                    const float *Bb = B + b * sb;
                    for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
                    if (alpha != 0.0f) {
                        for (int64_t k = 0; k < K; ++k) {
                            const double a = (double)(op_a ? Ab[k * lda + i] : Ab[i * lda + k]);
                            for (int64_t j = 0; j < N; ++j) {
                                const double bv =
                                    (double)(op_b ? Bb[j * ldb + k] : Bb[k * ldb + j]);
                                acc[j] += a * bv;
                            }
                        }
                    }
                    for (int64_t j = 0; j < N; ++j) {
                        double v = (alpha != 0.0f) ? (double)alpha * acc[j] : 0.0;
                        if (beta != 0.0f) v += (double)beta * (double)C0[b * sc + i * ldc0 + j];
                        if (bias) v += (double)bias[j];
                        if (act == 1) v = oracle_gelu_tanh(v);
                        C[(b * M + i) * N + j] = (float)v;
                    }
                }
            }
            free(acc);
        }
    }
    return bad;
}
