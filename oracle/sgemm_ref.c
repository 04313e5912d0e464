/*
 * Oracle for single-precision GEMM, C = alpha * (A . B) + beta * C, row-major.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the bench's CPU
 * baseline call this file. It shares no code, header or table with the CUDA library and
 * includes nothing from it.
 *
 * What it computes (the plain definition, written out):
 *   every cell of C is one row of A dotted with one column of B, summed over k
 *   ("a CUDA matmul", section 00 for the alpha/beta form and section 02 for the loop;
 *    "GEMM scrapbook", the GEMM definition and the 2D block-tiling chapter, where
 *    C = sum over k of (column k of A) outer (row k of B);
 *    "The 1% kernel", section 1 for the cell formula, written there for square matrices).
 *
 *   out[i][j] = fl32( alpha * S_ij + beta * C[i][j] ),  S_ij = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *
 * Readings where the pages are silent (BLAS conventions):
 *   - the sum runs in ascending k in fp64; each product of two fp32 values is exact in fp64,
 *     so the only rounding inside S_ij is that of the fp64 additions;
 *   - beta == 0: C is not read at all (a NaN or Inf there does not reach the result);
 *   - alpha == 0: A and B are not read, out = fl32(beta * C) (0 when beta == 0 too);
 *   - K == 0: S_ij = 0, so out = fl32(beta * C) (0 when beta == 0);
 *   - the single rounding to fp32 is round-to-nearest-even, done by the C cast.
 *
 * Storage: element (r, c) of a row-major matrix with leading dimension ld sits at r * ld + c
 * ("The 1% kernel", section 4).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARGS 1
#define ORACLE_NO_MEMORY 2

static int check_args(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                      int64_t ldo) {
    if (M < 0 || N < 0 || K < 0) return 0;
    if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldo < (N > 1 ? N : 1)) return 0;
    if (ldc < (N > 1 ? N : 1)) return 0;
    return 1;
}

/*
 * Rows rows[0..nrows-1] of the result (all M rows, in order, when rows == NULL; then
 * nrows is ignored). out is nrows x N with leading dimension ldo; out row r holds result
 * row rows[r]. A is M x K (lda), B is K x N (ldb), C is M x N (ldc) and is read only when
 * beta != 0. Returns 0 on success.
 */
int sgemm_ref_rows(int64_t M, int64_t N, int64_t K, double alpha,
                   const float *A, int64_t lda, const float *B, int64_t ldb,
                   double beta, const float *C, int64_t ldc,
                   const int64_t *rows, int64_t nrows, float *out, int64_t ldo) {
    if (!check_args(M, N, K, lda, ldb, ldc, ldo)) return ORACLE_BAD_ARGS;
    const int64_t R = rows ? nrows : M;
    if (R < 0) return ORACLE_BAD_ARGS;
    for (int64_t r = 0; rows && r < R; ++r)
        if (rows[r] < 0 || rows[r] >= M) return ORACLE_BAD_ARGS;
    if (R == 0 || N == 0) return ORACLE_OK;
    int failed = 0;

#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < R; ++r) {
            if (!acc) continue;
            const int64_t i = rows ? rows[r] : r;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            if (alpha != 0.0) {
                /* i-k-j order: for every j, the sum over k still runs in ascending k. */
                for (int64_t k = 0; k < K; ++k) {
                    const double a = (double)A[i * lda + k];
                    const float *brow = B + k * ldb;
                    for (int64_t j = 0; j < N; ++j) acc[j] += a * (double)brow[j];
                }
            }
            float *orow = out + r * ldo;
            for (int64_t j = 0; j < N; ++j) {
                double v = (alpha != 0.0) ? alpha * acc[j] : 0.0;
                if (beta != 0.0) v += beta * (double)C[i * ldc + j];
                orow[j] = (float)v;
            }
        }
        free(acc);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/*
 * Denominator of the normalised error used to judge a GPU result:
 * den[r][j] = sum_k |A[i][k]| * |B[k][j]| in fp64 (ascending k), for i = rows[r]
 * (all rows when rows == NULL). Same argument conventions as sgemm_ref_rows; the result
 * stays in fp64 so that the tolerance check itself adds no fp32 rounding.
 */
int sgemm_ref_absdot_rows(int64_t M, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          const int64_t *rows, int64_t nrows, double *den, int64_t ldd) {
    if (!check_args(M, N, K, lda, ldb, N > 1 ? N : 1, ldd)) return ORACLE_BAD_ARGS;
    const int64_t R = rows ? nrows : M;
    if (R < 0) return ORACLE_BAD_ARGS;
    for (int64_t r = 0; rows && r < R; ++r)
        if (rows[r] < 0 || rows[r] >= M) return ORACLE_BAD_ARGS;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *drow = den + r * ldd;
        for (int64_t j = 0; j < N; ++j) drow[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = fabs((double)A[i * lda + k]);
            const float *brow = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) drow[j] += a * fabs((double)brow[j]);
        }
    }
    return ORACLE_OK;
}

/*
 * The same product with transposed operands (BLAS transa / transb, row-major storage):
 *   op(A)[i][k] = transa ? A[k * lda + i] : A[i * lda + k]   (A stored K x M when transposed)
 *   op(B)[k][j] = transb ? B[j * ldb + k] : B[k * ldb + j]   (B stored N x K when transposed)
 *   out[i][j]   = fl32( alpha * sum_k op(A)[i][k] * op(B)[k][j] + beta * C[i][j] )
 * with the same readings as sgemm_ref_rows (fp64 sum in ascending k, beta == 0 leaves C unread,
 * alpha == 0 leaves A and B unread). Leading dimensions: lda >= max(1, transa ? M : K),
 * ldb >= max(1, transb ? K : N), ldc, ldo >= max(1, N).
 */
int sgemm_ref_ex_rows(int transa, int transb, int64_t M, int64_t N, int64_t K, double alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      double beta, const float *C, int64_t ldc,
                      const int64_t *rows, int64_t nrows, float *out, int64_t ldo) {
    if (M < 0 || N < 0 || K < 0) return ORACLE_BAD_ARGS;
    const int64_t a_cols = transa ? M : K, b_cols = transb ? K : N;
    if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1)) return ORACLE_BAD_ARGS;
    if (ldc < (N > 1 ? N : 1) || ldo < (N > 1 ? N : 1)) return ORACLE_BAD_ARGS;
    const int64_t R = rows ? nrows : M;
    if (R < 0) return ORACLE_BAD_ARGS;
    for (int64_t r = 0; rows && r < R; ++r)
        if (rows[r] < 0 || rows[r] >= M) return ORACLE_BAD_ARGS;
    if (R == 0 || N == 0) return ORACLE_OK;
    int failed = 0;

#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < R; ++r) {
            if (!acc) continue;
            const int64_t i = rows ? rows[r] : r;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            if (alpha != 0.0) {
                for (int64_t k = 0; k < K; ++k) {
                    const double a = (double)(transa ? A[k * lda + i] : A[i * lda + k]);
                    for (int64_t j = 0; j < N; ++j)
                        acc[j] += a * (double)(transb ? B[j * ldb + k] : B[k * ldb + j]);
                }
            }
            float *orow = out + r * ldo;
            for (int64_t j = 0; j < N; ++j) {
                double v = (alpha != 0.0) ? alpha * acc[j] : 0.0;
                if (beta != 0.0) v += beta * (double)C[i * ldc + j];
                orow[j] = (float)v;
            }
        }
        free(acc);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* sum_k |op(A)[i][k]| * |op(B)[k][j]| in fp64 for the listed rows (transposes as above). */
int sgemm_ref_absdot_ex_rows(int transa, int transb, int64_t M, int64_t N, int64_t K,
                             const float *A, int64_t lda, const float *B, int64_t ldb,
                             const int64_t *rows, int64_t nrows, double *den, int64_t ldd) {
    if (M < 0 || N < 0 || K < 0) return ORACLE_BAD_ARGS;
    const int64_t a_cols = transa ? M : K, b_cols = transb ? K : N;
    if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1)) return ORACLE_BAD_ARGS;
    if (ldd < (N > 1 ? N : 1)) return ORACLE_BAD_ARGS;
    const int64_t R = rows ? nrows : M;
    if (R < 0) return ORACLE_BAD_ARGS;
    for (int64_t r = 0; rows && r < R; ++r)
        if (rows[r] < 0 || rows[r] >= M) return ORACLE_BAD_ARGS;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *drow = den + r * ldd;
        for (int64_t j = 0; j < N; ++j) drow[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = fabs((double)(transa ? A[k * lda + i] : A[i * lda + k]));
            for (int64_t j = 0; j < N; ++j)
                drow[j] += a * fabs((double)(transb ? B[j * ldb + k] : B[k * ldb + j]));
        }
    }
    return ORACLE_OK;
}

/*
 * Activation functions of the fused epilogue, in fp64, from their published definitions:
 *   0 identity;  1 ReLU, max(x, 0) (NaN stays NaN);
 *   2 GELU, x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2))   (Hendrycks & Gimpel, 2016);
 *   3 GELU, tanh form 0.5 x (1 + tanh(sqrt(2 / pi) (x + 0.044715 x^3)))  (same paper);
 *   4 SiLU, x * sigmoid(x) = x / (1 + exp(-x))   (Elfwing, Uchibe & Doya, 2018).
 */
static double activation(double x, int act) {
    switch (act) {
        case 1: return x > 0.0 ? x : (x != x ? x : 0.0);
        case 2: return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
        case 3: {
            const double c = sqrt(2.0 / 3.14159265358979323846);
            return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
        }
        case 4: return x / (1.0 + exp(-x));
        default: return x;
    }
}

/*
 * Fused epilogue: out[i][j] = fl32( act(alpha * S_ij + bias[j]) + beta * C[i][j] ), with S_ij
 * the transposed-operand sum of sgemm_ref_ex_rows (fp64, ascending k), bias a length-N vector
 * (NULL: no bias), act as above, and C read only when beta != 0. act codes outside 0..4 are
 * rejected.
 */
int sgemm_ref_epilogue_rows(int transa, int transb, int64_t M, int64_t N, int64_t K,
                            double alpha, const float *A, int64_t lda, const float *B,
                            int64_t ldb, double beta, const float *C, int64_t ldc,
                            const float *bias, int act, const int64_t *rows, int64_t nrows,
                            float *out, int64_t ldo) {
    if (act < 0 || act > 4) return ORACLE_BAD_ARGS;
    if (M < 0 || N < 0 || K < 0) return ORACLE_BAD_ARGS;
    const int64_t a_cols = transa ? M : K, b_cols = transb ? K : N;
    if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1)) return ORACLE_BAD_ARGS;
    if (ldc < (N > 1 ? N : 1) || ldo < (N > 1 ? N : 1)) return ORACLE_BAD_ARGS;
    const int64_t R = rows ? nrows : M;
    if (R < 0) return ORACLE_BAD_ARGS;
    for (int64_t r = 0; rows && r < R; ++r)
        if (rows[r] < 0 || rows[r] >= M) return ORACLE_BAD_ARGS;
    if (R == 0 || N == 0) return ORACLE_OK;
    int failed = 0;

#pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)N * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < R; ++r) {
            if (!acc) continue;
            const int64_t i = rows ? rows[r] : r;
            for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
            if (alpha != 0.0) {
                for (int64_t k = 0; k < K; ++k) {
                    const double a = (double)(transa ? A[k * lda + i] : A[i * lda + k]);
                    for (int64_t j = 0; j < N; ++j)
                        acc[j] += a * (double)(transb ? B[j * ldb + k] : B[k * ldb + j]);
                }
            }
            float *orow = out + r * ldo;
            for (int64_t j = 0; j < N; ++j) {
                double v = (alpha != 0.0) ? alpha * acc[j] : 0.0;
                if (bias) v += (double)bias[j];
                v = activation(v, act);
                if (beta != 0.0) v += beta * (double)C[i * ldc + j];
                orow[j] = (float)v;
            }
        }
        free(acc);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Threads the loops above use (OpenMP over result rows). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
