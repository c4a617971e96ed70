/*
 * ref_sgemm.c -- CPU oracle for single-precision GEMM.  TEST INFRASTRUCTURE.
 *
 * This file is test infrastructure, not part of the product.  Only the tests,
 * the package's smoke entry (__graft_entry__.smoke) and the CPU-baseline leg of
 * bench.py may load it.  It shares no code, header or constant with the CUDA
 * path and includes nothing from it.
 *
 * What it computes (the plain definition, nothing more):
 *   "Beyond Kernel 7: Closing the Gap to cuBLAS on an H100 FP32 GEMM",
 *   section "The operation: GEMM and the precision of the comparison":
 *   for A (M x K) and B (K x N), C[m, n] = sum over k of A[m, k] * B[k, n];
 *   the experiments compute only A*B (alpha = 1, beta = 0).
 *   Layout: row-major ("the arrays are row-major", same page, "Kernel 1"),
 *   with an explicit row stride (ld) in elements.
 *
 * Precision: every FP32 input is widened to double.  A product of two FP32
 * values has at most 48 significant bits and is therefore exact in double
 * (53 bits); only the additions round, in the order k = 0, 1, ..., K-1.
 *
 * Besides C it returns E[m, n] = sum over k of |A[m, k] * B[k, n]|, the
 * magnitude that the acceptance bound |C_gpu - C| <= 4 K 2^-24 E scales with.
 *
 * The loops are the definition's m, n, k loops; rows of C are shared out to
 * OpenMP threads, which leaves every element's summation order unchanged.
 * Build: gcc -O2 -fno-fast-math -ffp-contract=off -fopenmp -shared -fPIC.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes: 0 = ok, 1 = invalid argument. */
#define REF_OK 0
#define REF_INVALID 1

static int ref_check(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                     const float *B, int64_t ldb) {
  if (M < 0 || N < 0 || K < 0) return REF_INVALID;
  if (M > 0 && K > 0 && (A == NULL || lda < K)) return REF_INVALID;
  if (N > 0 && K > 0 && (B == NULL || ldb < N)) return REF_INVALID;
  return REF_OK;
}

/* One element of the definition: C[m, n] and E[m, n] in double. */
static void ref_element(int64_t m, int64_t n, int64_t K, const float *A, int64_t lda,
                        const float *B, int64_t ldb, double *c, double *e) {
  double s = 0.0, a = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    double p = (double)A[m * lda + k] * (double)B[k * ldb + n];
    s += p;
    a += fabs(p);
  }
  *c = s;
  *e = a;
}

/*
 * Full product.  C (M x N, row stride ldc) receives the double result;
 * E (row stride lde) receives sum |a*b| and may be NULL.
 */
int ref_sgemm_f64(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                  const float *B, int64_t ldb, double *C, int64_t ldc, double *E,
                  int64_t lde) {
  int st = ref_check(M, N, K, A, lda, B, ldb);
  if (st != REF_OK) return st;
  if (M == 0 || N == 0) return REF_OK;
  if (C == NULL || ldc < N) return REF_INVALID;
  if (E != NULL && lde < N) return REF_INVALID;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double c, e;
      ref_element(m, n, K, A, lda, B, ldb, &c, &e);
      C[m * ldc + n] = c;
      if (E != NULL) E[m * lde + n] = e;
    }
  }
  return REF_OK;
}

/*
 * Selected elements only: for i < count, out_c[i] = C[rows[i], cols[i]] and
 * out_e[i] = E[rows[i], cols[i]] (out_e may be NULL).  Used to check sampled
 * outputs of products too large to compute in full on the host.
 */
int ref_sgemm_entries_f64(int64_t M, int64_t N, int64_t K, const float *A, int64_t lda,
                          const float *B, int64_t ldb, int64_t count, const int64_t *rows,
                          const int64_t *cols, double *out_c, double *out_e) {
  int st = ref_check(M, N, K, A, lda, B, ldb);
  if (st != REF_OK) return st;
  if (count < 0) return REF_INVALID;
  if (count > 0 && (rows == NULL || cols == NULL || out_c == NULL)) return REF_INVALID;
  for (int64_t i = 0; i < count; ++i)
    if (rows[i] < 0 || rows[i] >= M || cols[i] < 0 || cols[i] >= N) return REF_INVALID;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < count; ++i) {
    double c, e;
    ref_element(rows[i], cols[i], K, A, lda, B, ldb, &c, &e);
    out_c[i] = c;
    if (out_e != NULL) out_e[i] = e;
  }
  return REF_OK;
}

/*
 * The general form with scaling and either storage order.  The epilogue of
 * "Vectorized Memory Access: Pushing CUDA SGEMM to 29 TFLOPS on H100", section
 * 5, and "2D Block Tiling: Scaling Matrix Multiplication on NVIDIA H100",
 * section 5, writes C[m, n] = alpha * (sum_k A[m, k] B[k, n]) + beta * C[m, n].
 * Here C0 holds the old C (it may be NULL when beta == 0, which never reads
 * it, so a NaN there does not propagate) and the result goes to Cout, all in
 * double.  col_major != 0 means element (r, c) of a matrix with leading
 * dimension ld sits at base[r + c * ld] instead of base[r * ld + c].
 */
int ref_sgemm_ex_f64(int col_major, int64_t M, int64_t N, int64_t K, double alpha,
                     const float *A, int64_t lda, const float *B, int64_t ldb, double beta,
                     const float *C0, int64_t ldc, double *Cout, int64_t ldo) {
  if (M < 0 || N < 0 || K < 0) return REF_INVALID;
  if (M == 0 || N == 0) return REF_OK;
  if (Cout == NULL || ldo < N) return REF_INVALID;
  if (beta != 0.0 && C0 == NULL) return REF_INVALID;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const float a = col_major ? A[m + k * lda] : A[m * lda + k];
        const float b = col_major ? B[k + n * ldb] : B[k * ldb + n];
        s += (double)a * (double)b;
      }
      double r = alpha * s;
      if (beta != 0.0) r += beta * (double)(col_major ? C0[m + n * ldc] : C0[m * ldc + n]);
      Cout[m * ldo + n] = r;  /* the double result is always row-major */
    }
  }
  return REF_OK;
}

/* Element (r, c) of a matrix stored with leading dimension ld. */
static float ref_at(const float *X, int64_t ld, int col_major, int64_t r, int64_t c) {
  return col_major ? X[r + c * ld] : X[r * ld + c];
}

/*
 * The general form with a transposition flag per operand, the BLAS-style
 * op() the same epilogue is usually paired with:
 *   C[m, n] = alpha * (sum_k op(A)[m, k] op(B)[k, n]) + beta * C0[m, n],
 * op(A) = A (stored M x K) when trans_a == 0 and A^T (A stored K x M, so
 * op(A)[m, k] is the stored element (k, m)) otherwise; likewise op(B) = B
 * (stored K x N) or B^T (stored N x K).  Storage order (row- or column-major)
 * is `col_major`, as in ref_sgemm_ex_f64, and applies to A, B and C0; Cout is
 * row-major double.  The sum runs over k = 0, 1, ..., K-1 in double, every
 * product exact.  beta == 0 never reads C0.
 */
int ref_sgemm_op_f64(int col_major, int trans_a, int trans_b, int64_t M, int64_t N, int64_t K,
                     double alpha, const float *A, int64_t lda, const float *B, int64_t ldb,
                     double beta, const float *C0, int64_t ldc, double *Cout, int64_t ldo) {
  if (M < 0 || N < 0 || K < 0) return REF_INVALID;
  if (M == 0 || N == 0) return REF_OK;
  if (Cout == NULL || ldo < N) return REF_INVALID;
  if (beta != 0.0 && C0 == NULL) return REF_INVALID;
  if (K > 0 && (A == NULL || B == NULL)) return REF_INVALID;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const float a = trans_a ? ref_at(A, lda, col_major, k, m) : ref_at(A, lda, col_major, m, k);
        const float b = trans_b ? ref_at(B, ldb, col_major, n, k) : ref_at(B, ldb, col_major, k, n);
        s += (double)a * (double)b;
      }
      double r = alpha * s;
      if (beta != 0.0) r += beta * (double)ref_at(C0, ldc, col_major, m, n);
      Cout[m * ldo + n] = r;
    }
  }
  return REF_OK;
}

/* Thread control for timing: 0 or less leaves the OpenMP default. */
void ref_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int ref_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
