/*
 * CPU oracle for half-precision GEMM -- TEST INFRASTRUCTURE ONLY.
 *
 * Only tests, the smoke check and the CPU-baseline leg of the benchmark may
 * load this library.  The GPU library never links, includes or calls it, and
 * it shares no code with the GPU path.
 *
 * What it computes (FalconGEMM talk write-up, section "从 Strassen 出发"):
 * every Strassen-family algorithm equals the ordinary matrix product in exact
 * arithmetic, so the oracle for all three algorithms is the plain definition
 *
 *     C64[i,j] = sum_k double(A[i,k]) * double(B[k,j])
 *
 * as a sequential triple loop in FP64 (OpenMP over output rows only; the k sum
 * of one output element is always taken in ascending k order).  Products of
 * two FP16 or two BF16 values are exact in FP64 (at most 22 significant bits).
 *
 * Layouts are those of the library boundary: A is row-major M x K with
 * leading dimension lda; B is the K x N operand stored column-major, i.e. as
 * N rows of K contiguous elements with leading dimension ldb; the result is
 * written row-major (nrows x N, leading dimension N) in FP64.
 *
 * Input elements are raw 16-bit patterns decoded by oracle_decode_f16/bf16
 * from the IEEE 754 binary16 and the bfloat16 definitions.  Those decoders are
 * pinned exhaustively (all 65536 patterns) against numpy in the CPU tests.
 */
#include <stdint.h>
#include <stdlib.h>
#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
  } else if (e == 31) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_decode_bf16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 7) & 0xff;
  int f = h & 0x7f;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133); /* subnormal: f * 2^-7 * 2^-126 */
  } else if (e == 255) {
    v = (f == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) * 2^(e-127) */
  }
  return sign ? -v : v;
}

static void build_table(int dtype, double* tbl) {
  for (uint32_t x = 0; x < 65536u; ++x)
    tbl[x] = (dtype == ORACLE_BF16) ? oracle_decode_bf16((uint16_t)x) : oracle_decode_f16((uint16_t)x);
}

/*
 * C[r, j] = sum_k A[rows[r], k] * B[k, j] for r < nrows, j < N (FP64).
 * rows == NULL means rows 0..nrows-1.  Returns 0, or -1 on bad arguments.
 */
int oracle_gemm(int dtype, int64_t M, int64_t N, int64_t K,
                const uint16_t* A, int64_t lda, const uint16_t* B, int64_t ldb,
                const int64_t* rows, int64_t nrows, double* C) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
  if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
  if (nrows > 0 && N > 0 && K > 0 && (!A || !B || lda < K || ldb < K)) return -1;
  if (nrows > 0 && N > 0 && !C) return -1;
  double* tbl = (double*)malloc(sizeof(double) * 65536);
  if (!tbl) return -1;
  build_table(dtype, tbl);
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t i = rows ? rows[r] : r;
    if (i < 0 || i >= M) { bad = 1; continue; }
    double* arow = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    if (!arow) { bad = 1; continue; }
    for (int64_t k = 0; k < K; ++k) arow[k] = tbl[A[i * lda + k]];
    for (int64_t j = 0; j < N; ++j) {
      const uint16_t* bcol = B + j * ldb;
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += arow[k] * tbl[bcol[k]];
      C[r * N + j] = s;
    }
    free(arow);
  }
  free(tbl);
  return bad ? -1 : 0;
}

/* Number of threads the OpenMP loop in oracle_gemm uses. */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
