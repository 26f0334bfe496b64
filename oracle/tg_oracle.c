/*
 * CPU oracle for the row-major FP32 matrix product C = A x B.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load, call or
 * link this file; it is used by tests/, by __graft_entry__.smoke() and by the
 * CPU-baseline and reference legs of bench.py.  It shares no code, header,
 * table or helper with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *
 *     C[i][j] = sum_{k=0}^{K-1} A[i][k] * B[k][j]
 *
 * - "03 CUDA Shared Memory: Tiling, Bank Conflicts, and Reduction",
 *   section "Shared Memory와 Tiling": one output element is the dot product of
 *   one row of A with one column of B, two FLOP (a multiply and an add) per k.
 * - "PMPP 단권화", ch. 3 card on matrix multiplication: the same product with
 *   row-major linear indexing r*W + c.
 * - PMPP ch. 5 notes ("메모리 계층과 데이터 지역성"), §5.5: out-of-range
 *   (ghost) elements are zeros that do not change the sum, so the oracle needs
 *   no padding at all.
 *
 * Readings taken where the pages are silent:
 * - shapes: A is M x K, B is K x N, C is M x N, each row-major with leading
 *   dimensions lda >= K, ldb >= N, ldc >= N (the pages show only square
 *   matrices with the width as stride);
 * - accumulation: in double, k ascending from +0.0, then one round-to-nearest-
 *   even conversion to float.  Every product of two floats is exact in double
 *   (24 + 24 significant bits <= 53), so the only double-precision error is
 *   from the additions;
 * - C is overwritten (no alpha/beta); K == 0 gives +0.0 everywhere;
 * - columns j >= N of a padded C row (ldc > N) are never written.
 *
 * Loop order: i (rows, split across OpenMP threads), then k ascending, then j.
 * Each C element still receives its terms one at a time in ascending k into
 * its own double accumulator, i.e. exactly the sum order of the definition;
 * the k-outer order only makes B's rows stream contiguously.
 *
 * Parity status: every entry point here is pinned by tests/test_oracle.py
 * (hand-worked products, identities, permutations, the transpose law, exact
 * rational brute force, closed forms, zero-padding invariance and integer
 * exactness; for the general form also alpha/beta closed forms, stored
 * transposes and exact rational brute force).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One output row: C_row[0..N) = A_row[0..K) . B.  acc is caller scratch of N
 * doubles. */
static void oracle_row(int64_t N, int64_t K, const float* A_row,
                       const float* B, int64_t ldb, double* acc,
                       float* C_row) {
    for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double a = (double)A_row[k];
        const float* B_row = B + k * ldb;
        for (int64_t j = 0; j < N; ++j) acc[j] += a * (double)B_row[j];
    }
    for (int64_t j = 0; j < N; ++j) C_row[j] = (float)acc[j];
}

static int bad_shape(int64_t M, int64_t N, int64_t K, int64_t lda,
                     int64_t ldb, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return 1;
    if (lda < (K > 1 ? K : 1)) return 1;
    if (ldb < (N > 1 ? N : 1)) return 1;
    if (ldc < (N > 1 ? N : 1)) return 1;
    return 0;
}

/* Full product.  Returns 0 on success, 1 on a bad shape, 2 on allocation
 * failure. */
int tg_oracle_sgemm(int64_t M, int64_t N, int64_t K, const float* A,
                    int64_t lda, const float* B, int64_t ldb, float* C,
                    int64_t ldc) {
    if (bad_shape(M, N, K, lda, ldb, ldc)) return 1;
    if (M == 0 || N == 0) return 0;
    int failed = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc((size_t)N * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < M; ++i) {
            if (acc) oracle_row(N, K, A + i * lda, B, ldb, acc, C + i * ldc);
        }
        free(acc);
    }
    return failed ? 2 : 0;
}

/* Selected rows only: C_rows[r*ldc_rows + j] = (A x B)[rows[r]][j].  Used
 * where the full product is too slow to check (rows sampled by the caller). */
int tg_oracle_sgemm_rows(int64_t nrows, const int64_t* rows, int64_t M,
                         int64_t N, int64_t K, const float* A, int64_t lda,
                         const float* B, int64_t ldb, float* C_rows,
                         int64_t ldc_rows) {
    if (nrows < 0 || bad_shape(M, N, K, lda, ldb, ldc_rows)) return 1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return 1;
    if (nrows == 0 || N == 0) return 0;
    int failed = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc((size_t)N * sizeof(double));
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (acc)
                oracle_row(N, K, A + rows[r] * lda, B, ldb, acc,
                           C_rows + r * ldc_rows);
        }
        free(acc);
    }
    return failed ? 2 : 0;
}

/*
 * General form: C = alpha * op(A) * op(B) + beta * C.
 *
 * op(A) is M x K: A is stored M x K (lda >= K) when op_a == 0 and K x M
 * (lda >= M) when op_a == 1 (transposed); op(B) is K x N: B is stored K x N
 * (ldb >= N) when op_b == 0 and N x K (ldb >= K) when op_b == 1.  These are
 * the shapes of the backward products of a fully connected layer
 * ("PMPP 단권화", deep-learning chapter: FC layer = GEMM; dW = X^T dY and
 * dX = dY W^T).  Per element, in double: s = sum_k op(A)[i][k] op(B)[k][j]
 * (k ascending, from +0.0), r = alpha * s + beta * C[i][j], rounded once to
 * float.  When beta == 0, C is not read (it may hold NaN), as in BLAS.
 * K == 0 gives r = beta * C[i][j] (the empty sum).
 */
static int bad_general(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                       int64_t lda, int64_t ldb, int64_t ldc) {
    if (op_a < 0 || op_a > 1 || op_b < 0 || op_b > 1) return 1;
    if (M < 0 || N < 0 || K < 0) return 1;
    const int64_t a_row = op_a ? M : K, b_row = op_b ? K : N;
    if (lda < (a_row > 1 ? a_row : 1)) return 1;
    if (ldb < (b_row > 1 ? b_row : 1)) return 1;
    if (ldc < (N > 1 ? N : 1)) return 1;
    return 0;
}

int tg_oracle_sgemm_general(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                            float alpha, const float* A, int64_t lda,
                            const float* B, int64_t ldb, float beta, float* C,
                            int64_t ldc) {
    if (bad_general(op_a, op_b, M, N, K, lda, ldb, ldc)) return 1;
    if (M == 0 || N == 0) return 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                const double a = op_a ? (double)A[k * lda + i] : (double)A[i * lda + k];
                const double b = op_b ? (double)B[j * ldb + k] : (double)B[k * ldb + j];
                s += a * b;
            }
            double r = (double)alpha * s;
            if (beta != 0.0f) r += (double)beta * (double)C[i * ldc + j];
            C[i * ldc + j] = (float)r;
        }
    }
    return 0;
}

/*
 * Matrix transpose: out[c][r] = in[r][c] for 0 <= r < rows, 0 <= c < cols
 * (in is rows x cols with row stride ld_in >= cols; out is cols x rows with
 * ld_out >= rows).  The workload of "03 CUDA Shared Memory: Tiling, Bank
 * Conflicts, and Reduction", section "Bank Conflict": a tile is read along
 * rows and written along columns.  Pure index permutation, so any correct
 * implementation matches bit for bit.  Returns 0, or 1 on a bad shape.
 */
int tg_oracle_transpose(int64_t rows, int64_t cols, const float* in, int64_t ld_in,
                        float* out, int64_t ld_out) {
    if (rows < 0 || cols < 0) return 1;
    if (ld_in < (cols > 1 ? cols : 1) || ld_out < (rows > 1 ? rows : 1)) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) out[c * ld_out + r] = in[r * ld_in + c];
    return 0;
}

/*
 * Sum reduction: the sum of x[0..n) accumulated in double in ascending index
 * order from +0.0, rounded once to float ("03 CUDA Shared Memory: Tiling,
 * Bank Conflicts, and Reduction", section "Reduction": N values folded into
 * one).  Any summation order agrees with it to within the rounding of its own
 * fp32 partial sums.  Returns 0, or 1 on n < 0.
 */
int tg_oracle_sum(int64_t n, const float* x, float* result) {
    if (n < 0) return 1;
    double s = 0.0;
    for (int64_t i = 0; i < n; ++i) s += (double)x[i];
    *result = (float)s;
    return 0;
}

/* Set the number of threads later calls use (n >= 1); returns the new count.
 * Only the timing of the oracle changes: every output is still one thread's
 * ascending-k sum. */
int tg_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Number of threads the two entry points above use. */
int tg_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
