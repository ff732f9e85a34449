/*
 * CPU oracle for the preshuffle GEMM  C[M,N] = A[M,K] . B[N,K]^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header or table with the CUDA path.
 *
 * These are the plain definitions, written as triple loops without blocking
 * or reordering.  Parallelism covers only independent output elements.
 *
 * - "gemm-optimization" guide, section 1.1 (three-level tiling): states the
 *   product C = A . B^T.  Section 12.1 fixes B as [N, K] row-major.
 * - Section 7.1 (direct-store epilogue): the scaled epilogue multiplies the
 *   accumulator by scale_a * scale_b.  The Python side applies that rule to
 *   the sums these functions return.
 * - Section 8.2 (MXFP4 bytes): the block-scaled form, one scale per 32
 *   K-elements for each operand.
 *
 * Precision: int64 for integer operands and fp64 for everything else.
 */
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* C[m*N+n] = sum_k A[m*K+k] * B[n*K+k], exact in int64. */
void oracle_gemm_i8_i64(const int8_t* A, const int8_t* B, int64_t M, int64_t N,
                        int64_t K, int64_t* C) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      const int8_t* a = A + m * K;
      const int8_t* b = B + n * K;
      int64_t acc = 0;
      for (int64_t k = 0; k < K; ++k) acc += (int64_t)a[k] * (int64_t)b[k];
      C[m * N + n] = acc;
    }
  }
}

/* C[m*N+n] = sum_k A[m*K+k] * B[n*K+k] in fp64 (operands already decoded). */
void oracle_gemm_f64(const double* A, const double* B, int64_t M, int64_t N,
                     int64_t K, double* C) {
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      const double* a = A + m * K;
      const double* b = B + n * K;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += a[k] * b[k];
      C[m * N + n] = acc;
    }
  }
}

/*
 * Block-scaled product in fp64:
 *   C[m,n] = sum_{j < K/blk} SA[m,j] * SB[n,j] * sum_{k in block j} A[m,k]*B[n,k]
 * A, B hold decoded element values and SA [M, K/blk], SB [N, K/blk] hold
 * decoded block scales.
 */
void oracle_gemm_block_f64(const double* A, const double* B, const double* SA,
                           const double* SB, int64_t M, int64_t N, int64_t K,
                           int64_t blk, double* C) {
  const int64_t nb = K / blk;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = 0; m < M; ++m) {
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t j = 0; j < nb; ++j) {
        const double* a = A + m * K + j * blk;
        const double* b = B + n * K + j * blk;
        double part = 0.0;
        for (int64_t k = 0; k < blk; ++k) part += a[k] * b[k];
        acc += SA[m * nb + j] * SB[n * nb + j] * part;
      }
      C[m * N + n] = acc;
    }
  }
}

/* Number of OpenMP threads the loops above use (for the CPU baseline). */
int oracle_num_threads(void) {
  int t = 1;
#pragma omp parallel
  {
#pragma omp single
    {
#ifdef _OPENMP
      t = omp_get_num_threads();
#endif
    }
  }
  return t;
}
