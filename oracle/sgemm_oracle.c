/*
 * CPU oracle for the row-major FP32 matrix product C[M x N] = A[M x K] . B[K x N].
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or constant with the CUDA library.
 *
 * What it computes is the plain definition of the product, written out:
 *
 *     C[i,j] = sum_{k=0}^{K-1} A[i,k] * B[k,j]          0 <= i < M, 0 <= j < N
 *
 * ("Micro Kernel 입문하기", §3 "K 루프": the GEMM formula the register
 *  accumulators c_ij hold; "누산 개념을 Grid-Block-Warp-Thread 계층에 끼워넣기",
 *  §2 (4): every thread's acc[i][j] is stored to C[(row)*ldc + col]).
 *
 * Two accumulation modes:
 *
 *   oracle_gemm_f64*      each fp32 input is widened to double; a product of two
 *                         fp32 values is exact in double; the K products are
 *                         summed in double with k ascending.  This is the parity
 *                         reference for every GPU result.
 *
 *   oracle_gemm_f32_fma_seq
 *                         acc = fmaf(A[i,k], B[k,j], acc) in fp32 with k
 *                         ascending, which is what the single-thread 4x4 example
 *                         of "Micro Kernel 입문하기" §2 does once nvcc contracts
 *                         `c += a*b` into one fused multiply-add (its default).
 *                         Used only to reproduce that page's printed output.
 *
 * Storage is row-major with leading dimensions (elements between rows): A[i,k]
 * is A[i*lda + k], B[k,j] is B[k*ldb + j], C[i,j] is C[i*ldc + j].  Elements in
 * the padding of a row (column index >= the logical width) are never read or
 * written.
 *
 * The loops run i -> k -> j with a row of double accumulators, so every C[i,j]
 * still receives its K terms one at a time in ascending k; rows are independent
 * and are spread over OpenMP threads, which does not change any result.
 *
 * Return value: 0 on success, -1 on invalid arguments (negative sizes, a leading
 * dimension below the logical width, a null pointer with a non-empty extent).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static int bad_args(int M, int N, int K, const float* A, int64_t lda,
                    const float* B, int64_t ldb, const void* C, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    if (lda < (K > 0 ? K : 1) || ldb < (N > 0 ? N : 1) || ldc < (N > 0 ? N : 1)) return 1;
    if (M > 0 && K > 0 && A == NULL) return 1;
    if (K > 0 && N > 0 && B == NULL) return 1;
    if (M > 0 && N > 0 && C == NULL) return 1;
    return 0;
}

static void one_row_f64(int N, int K, const float* Arow, const float* B, int64_t ldb,
                        double* crow)
{
    for (int j = 0; j < N; ++j) crow[j] = 0.0;
    for (int k = 0; k < K; ++k) {
        const double a = (double)Arow[k];
        const float* brow = B + (int64_t)k * ldb;
        for (int j = 0; j < N; ++j) crow[j] += a * (double)brow[j];
    }
}

/* Full product in double.  C is M x N doubles with leading dimension ldc. */
int oracle_gemm_f64(int M, int N, int K, const float* A, int64_t lda, const float* B,
                    int64_t ldb, double* C, int64_t ldc, int nthreads)
{
    if (bad_args(M, N, K, A, lda, B, ldb, C, ldc)) return -1;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int i = 0; i < M; ++i)
        one_row_f64(N, K, A + (int64_t)i * lda, B, ldb, C + (int64_t)i * ldc);
    return 0;
}

/* Selected rows only: out[r*N + j] = C[rows[r], j].  For full-size checks where
 * the whole product would take too long on the host. */
int oracle_gemm_f64_rows(int M, int N, int K, const float* A, int64_t lda, const float* B,
                         int64_t ldb, const int32_t* rows, int nrows, double* out,
                         int nthreads)
{
    if (bad_args(M, N, K, A, lda, B, ldb, out, N > 0 ? N : 1)) return -1;
    if (nrows < 0 || (nrows > 0 && rows == NULL)) return -1;
    for (int r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= M) return -1;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int r = 0; r < nrows; ++r)
        one_row_f64(N, K, A + (int64_t)rows[r] * lda, B, ldb, out + (int64_t)r * N);
    return 0;
}

/* Selected elements only: out[e] = C[ii[e], jj[e]]. */
int oracle_gemm_f64_elems(int M, int N, int K, const float* A, int64_t lda, const float* B,
                          int64_t ldb, const int32_t* ii, const int32_t* jj, int n,
                          double* out)
{
    if (bad_args(M, N, K, A, lda, B, ldb, out, N > 0 ? N : 1)) return -1;
    if (n < 0 || (n > 0 && (ii == NULL || jj == NULL))) return -1;
    for (int e = 0; e < n; ++e) {
        if (ii[e] < 0 || ii[e] >= M || jj[e] < 0 || jj[e] >= N) return -1;
        double acc = 0.0;
        for (int k = 0; k < K; ++k)
            acc += (double)A[(int64_t)ii[e] * lda + k] * (double)B[(int64_t)k * ldb + jj[e]];
        out[e] = acc;
    }
    return 0;
}

/* fp32 accumulation, one fused multiply-add per term, k ascending. */
int oracle_gemm_f32_fma_seq(int M, int N, int K, const float* A, int64_t lda,
                            const float* B, int64_t ldb, float* C, int64_t ldc)
{
    if (bad_args(M, N, K, A, lda, B, ldb, C, ldc)) return -1;
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k)
                acc = fmaf(A[(int64_t)i * lda + k], B[(int64_t)k * ldb + j], acc);
            C[(int64_t)i * ldc + j] = acc;
        }
    return 0;
}

/* Scaled form, in double:  out[r][j] = alpha * C[i][j] + beta * C0[i][j]  with
 * C[i][j] the product above and i = rows[r] (rows == NULL: i = r for all M rows).
 * BLAS conventions: beta == 0 -> C0 is not read; alpha == 0 -> A and B are not
 * read.  ("기존 작성한 GE_v2 의 regemm 타일드 커널의 1:1 매핑, gemm_tiled_test 작성"
 * names the GE_v2 epilogue that its test kernel strips; this is the usual
 * alpha/beta reading of it.)  out is nrows x N with leading dimension N. */
int oracle_gemm_f64_ex(int M, int N, int K, double alpha, const float* A, int64_t lda,
                       const float* B, int64_t ldb, double beta, const float* C0,
                       int64_t ldc0, const int32_t* rows, int nrows, double* out,
                       int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (rows == NULL && nrows != M) return -1;
    if (lda < (K > 0 ? K : 1) || ldb < (N > 0 ? N : 1) || ldc0 < (N > 0 ? N : 1)) return -1;
    if (nrows > 0 && N > 0 && out == NULL) return -1;
    if (alpha != 0.0 && K > 0 && nrows > 0 && N > 0 && (A == NULL || B == NULL)) return -1;
    if (beta != 0.0 && nrows > 0 && N > 0 && C0 == NULL) return -1;
    for (int r = 0; r < nrows; ++r)
        if (rows != NULL && (rows[r] < 0 || rows[r] >= M)) return -1;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int r = 0; r < nrows; ++r) {
        const int i = rows != NULL ? rows[r] : r;
        double* o = out + (int64_t)r * N;
        if (alpha != 0.0) {
            one_row_f64(N, K, A + (int64_t)i * lda, B, ldb, o);
            for (int j = 0; j < N; ++j) o[j] *= alpha;
        } else {
            for (int j = 0; j < N; ++j) o[j] = 0.0;
        }
        if (beta != 0.0)
            for (int j = 0; j < N; ++j) o[j] += beta * (double)C0[(int64_t)i * ldc0 + j];
    }
    return 0;
}

/* Transposed operands, BLAS style, in double:
 *   out[i][j] = alpha * sum_k opA[i][k] * opB[k][j] + beta * C0[i][j]
 * with opA[i][k] = A[i*lda + k] (transa == 0, A stored M x K) or A[k*lda + i]
 * (transa == 1, A stored K x M), and opB[k][j] = B[k*ldb + j] (transb == 0, B
 * stored K x N) or B[j*ldb + k] (transb == 1, B stored N x K).  The product of
 * the pages ("Register/Shared Memory Tiling", 관련 개념) taken on op(A), op(B);
 * the same i -> k -> j loops and k order as above, only the reads change.
 * beta == 0 does not read C0; alpha == 0 does not read A or B.  out is M x N
 * with leading dimension N. */
int oracle_gemm_f64_op(int transa, int transb, int M, int N, int K, double alpha,
                       const float* A, int64_t lda, const float* B, int64_t ldb, double beta,
                       const float* C0, int64_t ldc0, double* out, int nthreads)
{
    if ((transa != 0 && transa != 1) || (transb != 0 && transb != 1)) return -1;
    if (M < 0 || N < 0 || K < 0) return -1;
    const int wa = transa ? M : K, wb = transb ? K : N;   /* stored row widths */
    if (lda < (wa > 0 ? wa : 1) || ldb < (wb > 0 ? wb : 1) || ldc0 < (N > 0 ? N : 1)) return -1;
    if (M > 0 && N > 0 && out == NULL) return -1;
    if (alpha != 0.0 && K > 0 && M > 0 && N > 0 && (A == NULL || B == NULL)) return -1;
    if (beta != 0.0 && M > 0 && N > 0 && C0 == NULL) return -1;
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int i = 0; i < M; ++i) {
        double* o = out + (int64_t)i * N;
        for (int j = 0; j < N; ++j) o[j] = 0.0;
        if (alpha != 0.0) {
            for (int k = 0; k < K; ++k) {
                const double a = transa ? (double)A[(int64_t)k * lda + i]
                                        : (double)A[(int64_t)i * lda + k];
                for (int j = 0; j < N; ++j) {
                    const double b = transb ? (double)B[(int64_t)j * ldb + k]
                                            : (double)B[(int64_t)k * ldb + j];
                    o[j] += a * b;
                }
            }
            for (int j = 0; j < N; ++j) o[j] *= alpha;
        }
        if (beta != 0.0)
            for (int j = 0; j < N; ++j) o[j] += beta * (double)C0[(int64_t)i * ldc0 + j];
    }
    return 0;
}

/* Threads an OpenMP region would use here (for reporting the CPU baseline). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
