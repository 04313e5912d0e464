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

/* Element strides of op(A) and op(B) in the stored operands (BLAS transa / transb, row-major
 * storage): op(A)[i][k] = A[i * ai + k * ak] and op(B)[k][j] = B[k * bk + j * bj]. A is stored
 * M x K (lda >= K), or K x M when transposed (lda >= M); B is stored K x N (ldb >= N), or N x K
 * when transposed (ldb >= K). */
typedef struct {
    int64_t ai, ak, bk, bj;
} op_strides;

static op_strides strides_of(int transa, int transb, int64_t lda, int64_t ldb) {
    op_strides s;
    s.ai = transa ? 1 : lda;
    s.ak = transa ? lda : 1;
    s.bk = transb ? 1 : ldb;
    s.bj = transb ? ldb : 1;
    return s;
}

/* Checks the sizes, leading dimensions and row list shared by every entry point below.
 * ldc and ldo are the leading dimensions of C and of the output (both >= max(1, N)). */
static int check_args(int transa, int transb, int64_t M, int64_t N, int64_t K, int64_t lda,
                      int64_t ldb, int64_t ldc, int64_t ldo, const int64_t *rows, int64_t nrows) {
    if (M < 0 || N < 0 || K < 0) return 0;
    const int64_t a_cols = transa ? M : K, b_cols = transb ? K : N;
    const int64_t n1 = N > 1 ? N : 1;
    if (lda < (a_cols > 1 ? a_cols : 1) || ldb < (b_cols > 1 ? b_cols : 1)) return 0;
    if (ldc < n1 || ldo < n1) return 0;
    if (rows && nrows < 0) return 0;
    for (int64_t r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return 0;
    return 1;
}

/*
 * The one product loop every result entry point uses. For each listed result row i (all M
 * rows when rows == NULL) and every column j:
 *   S_ij      = sum_{k=0}^{K-1} op(A)[i][k] * op(B)[k][j]     (fp64, ascending k)
 *   out[r][j] = fl32( act(alpha * S_ij + bias[j]) + beta * C[i][j] )
 * with the bias term only when bias != NULL, act as above (0: identity), the C term only when
 * beta != 0 (C is then not read at all), and S_ij neither formed nor A and B read when
 * alpha == 0. With act = 0 and no bias this is the plain alpha * S + beta * C.
 * Each product of two fp32 values is exact in fp64, so the only roundings are those of the
 * fp64 additions and the single final rounding to fp32 (round-to-nearest-even, the C cast).
 * The loop runs i-k-j (a row of op(B) at a time); for every j the sum still runs in ascending k.
 */
static int product_rows(int transa, int transb, int64_t M, int64_t N, int64_t K, double alpha,
                        const float *A, int64_t lda, const float *B, int64_t ldb, double beta,
                        const float *C, int64_t ldc, const float *bias, int act,
                        const int64_t *rows, int64_t nrows, float *out, int64_t ldo) {
    if (act < 0 || act > 4) return ORACLE_BAD_ARGS;
    if (!check_args(transa, transb, M, N, K, lda, ldb, ldc, ldo, rows, nrows))
        return ORACLE_BAD_ARGS;
    const int64_t R = rows ? nrows : M;
    if (R == 0 || N == 0) return ORACLE_OK;
    const op_strides st = strides_of(transa, transb, lda, ldb);
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
                    const double a = (double)A[i * st.ai + k * st.ak];
                    const float *brow = B + k * st.bk;   /* row k of op(B) */
                    for (int64_t j = 0; j < N; ++j) acc[j] += a * (double)brow[j * st.bj];
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

/*
 * Rows rows[0..nrows-1] of C = alpha * (A . B) + beta * C (all M rows, in order, when
 * rows == NULL; then nrows is ignored). out is nrows x N with leading dimension ldo; out row r
 * holds result row rows[r]. A is M x K (lda), B is K x N (ldb), C is M x N (ldc) and is read
 * only when beta != 0. Returns 0 on success.
 */
int sgemm_ref_rows(int64_t M, int64_t N, int64_t K, double alpha,
                   const float *A, int64_t lda, const float *B, int64_t ldb,
                   double beta, const float *C, int64_t ldc,
                   const int64_t *rows, int64_t nrows, float *out, int64_t ldo) {
    return product_rows(0, 0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, NULL, 0, rows,
                        nrows, out, ldo);
}

/*
 * The same product with transposed operands (BLAS transa / transb, row-major storage):
 *   out[i][j] = fl32( alpha * sum_k op(A)[i][k] * op(B)[k][j] + beta * C[i][j] )
 * with the strides above and the same readings as sgemm_ref_rows. Leading dimensions:
 * lda >= max(1, transa ? M : K), ldb >= max(1, transb ? K : N), ldc, ldo >= max(1, N).
 */
int sgemm_ref_ex_rows(int transa, int transb, int64_t M, int64_t N, int64_t K, double alpha,
                      const float *A, int64_t lda, const float *B, int64_t ldb,
                      double beta, const float *C, int64_t ldc,
                      const int64_t *rows, int64_t nrows, float *out, int64_t ldo) {
    return product_rows(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, NULL, 0,
                        rows, nrows, out, ldo);
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
    return product_rows(transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias, act,
                        rows, nrows, out, ldo);
}

/*
 * Denominator of the normalised error used to judge a GPU result:
 * den[r][j] = sum_k |op(A)[i][k]| * |op(B)[k][j]| in fp64 (ascending k), for i = rows[r]
 * (all rows when rows == NULL), transposes as in sgemm_ref_ex_rows. The result stays in fp64
 * so that the tolerance check itself adds no fp32 rounding.
 */
int sgemm_ref_absdot_ex_rows(int transa, int transb, int64_t M, int64_t N, int64_t K,
                             const float *A, int64_t lda, const float *B, int64_t ldb,
                             const int64_t *rows, int64_t nrows, double *den, int64_t ldd) {
    if (!check_args(transa, transb, M, N, K, lda, ldb, N > 1 ? N : 1, ldd, rows, nrows))
        return ORACLE_BAD_ARGS;
    const int64_t R = rows ? nrows : M;
    const op_strides st = strides_of(transa, transb, lda, ldb);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *drow = den + r * ldd;
        for (int64_t j = 0; j < N; ++j) drow[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double a = fabs((double)A[i * st.ai + k * st.ak]);
            const float *brow = B + k * st.bk;
            for (int64_t j = 0; j < N; ++j) drow[j] += a * fabs((double)brow[j * st.bj]);
        }
    }
    return ORACLE_OK;
}

/* sum_k |A[i][k]| * |B[k][j]| for the plain (non-transposed) operands. */
int sgemm_ref_absdot_rows(int64_t M, int64_t N, int64_t K,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          const int64_t *rows, int64_t nrows, double *den, int64_t ldd) {
    return sgemm_ref_absdot_ex_rows(0, 0, M, N, K, A, lda, B, ldb, rows, nrows, den, ldd);
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
