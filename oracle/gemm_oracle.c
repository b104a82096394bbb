/*
 * gemm_oracle.c -- CPU ground truth for the blocked matrix multiply.
 *
 * TEST INFRASTRUCTURE ONLY. The test-suite, the package's smoke check and the
 * benchmark's CPU-baseline leg are the only callers. The GPU library shares no
 * source, header, table or helper with this file, and this file includes
 * nothing of it.
 *
 * What is computed (the plain definition, written out):
 *
 *     C[i,j] = sum_{k=0}^{K-1} A[i,k] * B[k,j]     over the logical extents only,
 *
 * "Chapter 13: The Blocked Matmul Kernel", section 13.1 (one output tile depends
 * on all of A's rows and B's columns across the whole shared dimension K) and
 * section 13.2 (out-of-range M, N and K elements never contribute). Inputs are
 * decoded exactly into fp64 from their stored format by the bit-level decoders
 * below, so the ground truth is built from the identical rounded inputs the GPU
 * sees (section 13.3, Worked Example 13.3.1: "an fp64 ground truth computed from
 * the identical fp16-rounded inputs"). Sums run in fp64, k in ascending order.
 * Products of two fp16/bf16/fp32 values are exact in fp64.
 *
 * Besides C the oracle returns D[i,j] = sum_k |A[i,k] * B[k,j]|, the scale of
 * the relative error metric max |C_gpu - C| / D.
 *
 * Three further routines follow the pages' own algorithms step by step, for the
 * pins only:
 *   oracle_gemm_blocked  -- the 2D grid of BM x BN tiles with a K-loop and an
 *                           accumulator initialised once (section 13.1, Worked
 *                           Example 13.1.1), with the optional omission of the
 *                           K mask of section 13.2, Worked Example 13.2.2;
 *   oracle_gemm_f16acc   -- the fp16 accumulator of section 13.3, Worked
 *                           Example 13.3.1 (each K-chunk's dot rounded to fp16,
 *                           then added into an fp16 running total);
 *   oracle_round         -- round-to-nearest-even into fp16 / bf16 / fp32.
 *
 * And the second workload the pages point to, the row softmax of "Triton from
 * zero, Lesson 4: Block Pointers", homework 4 (the masked columns of a tile are
 * set to -inf before the max, so they add exp(-inf) = 0 to the sum):
 *   oracle_softmax_rows  -- y[i,j] = exp(x[i,j] - m_i) / sum_k exp(x[i,k] - m_i),
 *                           m_i = max_k x[i,k], in fp64 over the row's N values.
 *
 * Build: gcc -O3 -fopenmp -ffp-contract=off -shared -fPIC (oracle/build.py).
 * -ffp-contract=off keeps a*b+c as two roundings on every host, so x86_64 and
 * aarch64 builds give bit-identical results.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Storage formats understood by the oracle (its own numbering). */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_F64 = 3 };
/* Operand layouts: ROW = [rows][cols] with leading dimension ld;
 * COL = the transposed storage [cols][rows]. */
enum { OR_ROW = 0, OR_COL = 1 };

enum {
  OR_OK = 0,
  OR_EINVAL = -1,  /* bad dims, leading dimension, dtype or layout */
  OR_EBOUNDS = -2, /* an unmasked read would leave the caller's allocation */
  OR_ENOMEM = -3
};

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double dec_f16(uint16_t h) {
  int sign = h >> 15;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^(1-15-10) */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25); /* 1.m * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 word. */
static double dec_bf16(uint16_t h) {
  uint32_t w = (uint32_t)h << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double dec_elem(const void *base, int dtype, int64_t idx) {
  switch (dtype) {
  case OR_F32: return (double)((const float *)base)[idx];
  case OR_F16: return dec_f16(((const uint16_t *)base)[idx]);
  case OR_BF16: return dec_bf16(((const uint16_t *)base)[idx]);
  case OR_F64: return ((const double *)base)[idx];
  }
  return NAN;
}

/* Element (r, c) of a logical rows x cols operand stored with the given layout. */
static int64_t elem_index(int layout, int64_t ld, int64_t r, int64_t c) {
  return layout == OR_ROW ? r * ld + c : c * ld + r;
}

static int check_operand(int64_t rows, int64_t cols, int64_t ld, int dtype, int layout) {
  if (rows < 0 || cols < 0) return OR_EINVAL;
  if (dtype < OR_F32 || dtype > OR_F64) return OR_EINVAL;
  if (layout != OR_ROW && layout != OR_COL) return OR_EINVAL;
  int64_t inner = layout == OR_ROW ? cols : rows;
  if (ld < (inner > 0 ? inner : 1)) return OR_EINVAL;
  return OR_OK;
}

/* Decode one whole element, exposed so tests can check the decoders exhaustively. */
double oracle_decode(int dtype, uint64_t bits) {
  switch (dtype) {
  case OR_F16: return dec_f16((uint16_t)bits);
  case OR_BF16: return dec_bf16((uint16_t)bits);
  case OR_F32: {
    uint32_t w = (uint32_t)bits;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
  }
  case OR_F64: {
    double d;
    memcpy(&d, &bits, sizeof d);
    return d;
  }
  }
  return NAN;
}

/* ----------------------------------------------------------------- rounding */

/* Round x to the nearest value of a binary format with p significand bits
 * (implicit bit included), minimum normal exponent emin and maximum exponent
 * emax; ties go to the even significand; overflow gives infinity. Written from
 * the IEEE 754 definition of roundTiesToEven. */
static double round_format(double x, int p, int emin, int emax) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double a = fabs(x);
  int e;
  (void)frexp(a, &e);  /* a in [2^(e-1), 2^e) */
  int E = e - 1;
  if (E < emin) E = emin; /* subnormal range: fixed quantum */
  double quantum = ldexp(1.0, E - (p - 1));
  double q = a / quantum; /* exact: scaling by a power of two */
  double r = floor(q);
  double frac = q - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  double v = r * quantum;
  double max_finite = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
  if (v > max_finite) v = INFINITY;
  return copysign(v, x);
}

static double round_to(int dtype, double x) {
  switch (dtype) {
  case OR_F16: return round_format(x, 11, -14, 15);
  case OR_BF16: return round_format(x, 8, -126, 127);
  case OR_F32: return round_format(x, 24, -126, 127);
  case OR_F64: return x;
  }
  return NAN;
}

/* Round n doubles in place to the values of the given format. */
int oracle_round(double *x, int64_t n, int dtype) {
  if (dtype < OR_F32 || dtype > OR_F64 || n < 0) return OR_EINVAL;
  for (int64_t i = 0; i < n; ++i) x[i] = round_to(dtype, x[i]);
  return OR_OK;
}

/* ----------------------------------------------------------- plain product */

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * C and D for the listed rows of the product (all rows when rows == NULL).
 * Output row r (0 <= r < n_rows) holds logical row rows[r]: C[r*N + j], D[r*N + j].
 * A is M x K, B is K x N, each with its layout and leading dimension in elements.
 * n_threads <= 0 uses every OpenMP thread. Returns OR_OK or an OR_E* code;
 * nothing is read or written on error.
 */
int oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                    const void *A, int64_t lda, int a_dtype, int a_layout,
                    const void *B, int64_t ldb, int b_dtype, int b_layout,
                    const int64_t *rows, int64_t n_rows,
                    double *C, double *D, int n_threads) {
  if (M < 0 || N < 0 || K < 0) return OR_EINVAL;
  if (check_operand(M, K, lda, a_dtype, a_layout) ||
      check_operand(K, N, ldb, b_dtype, b_layout))
    return OR_EINVAL;
  if (rows == NULL) n_rows = M;
  if (n_rows < 0) return OR_EINVAL;
  for (int64_t r = 0; rows != NULL && r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= M) return OR_EINVAL;
  if (n_rows == 0 || N == 0) return OR_OK;
  if ((M > 0 && K > 0 && A == NULL) || (K > 0 && B == NULL) || C == NULL) return OR_EINVAL;

  /* B decoded once into a dense K x N fp64 matrix. */
  double *Bd = NULL;
  if (K > 0) {
    Bd = (double *)malloc((size_t)K * (size_t)N * sizeof(double));
    if (!Bd) return OR_ENOMEM;
    for (int64_t k = 0; k < K; ++k)
      for (int64_t j = 0; j < N; ++j)
        Bd[k * N + j] = dec_elem(B, b_dtype, elem_index(b_layout, ldb, k, j));
  }

  int status = OR_OK;
#ifdef _OPENMP
  int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
  {
    double *arow = (double *)malloc((size_t)(K > 0 ? K : 1) * sizeof(double));
    double *acc = (double *)malloc((size_t)N * sizeof(double));
    double *mag = (double *)malloc((size_t)N * sizeof(double));
    const int have_buffers = arow && acc && mag;
    if (!have_buffers) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = OR_ENOMEM;
    }
    /* Every thread reaches the work-sharing loop; one without buffers skips its rows. */
    {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int64_t r = 0; r < n_rows; ++r) {
        if (!have_buffers) continue;
        int64_t i = rows ? rows[r] : r;
        for (int64_t k = 0; k < K; ++k)
          arow[k] = dec_elem(A, a_dtype, elem_index(a_layout, lda, i, k));
        for (int64_t j = 0; j < N; ++j) acc[j] = 0.0, mag[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
          const double a = arow[k];
          const double *b = Bd + k * N;
          for (int64_t j = 0; j < N; ++j) {
            const double p = a * b[j];
            acc[j] += p;
            mag[j] += fabs(p);
          }
        }
        memcpy(C + r * N, acc, (size_t)N * sizeof(double));
        if (D) memcpy(D + r * N, mag, (size_t)N * sizeof(double));
      }
    }
    free(arow);
    free(acc);
    free(mag);
  }
  free(Bd);
  return status;
}

/* ---------------------------------------------------- the pages' algorithm */

/*
 * The blocked algorithm of "Chapter 13: The Blocked Matmul Kernel", section
 * 13.1, Worked Example 13.1.1: the output is a grid of ceil(M/BM) x ceil(N/BN)
 * tiles; each tile sets its accumulator to zero once, then walks ceil(K/BK)
 * K-chunks, adding the chunk's partial product (the tile-level dot) into the
 * accumulator; the store is masked by rows < M and cols < N.
 *
 * Loads are masked by rows < M and cols < N always and by k < K when mask_k is
 * non-zero (section 13.2's three-way masking). mask_k == 0 reproduces section
 * 13.2, Worked Example 13.2.2: chunk elements past K are read from the
 * underlying buffer. a_k_alloc / b_k_alloc give how many k positions the
 * caller's buffers really hold (>= K); an unmasked read past them is refused
 * with OR_EBOUNDS before anything is read.
 *
 * tile_order (a permutation of the tile indices, tile = pid_m * tiles_n +
 * pid_n) and kblock_order (a permutation of the K-chunk indices) set the
 * visiting order; NULL means ascending. The result is C[i*ldc + j] in fp64.
 */
int oracle_gemm_blocked(int64_t M, int64_t N, int64_t K,
                        const void *A, int64_t lda, int a_dtype, int a_layout, int64_t a_k_alloc,
                        const void *B, int64_t ldb, int b_dtype, int b_layout, int64_t b_k_alloc,
                        int64_t BM, int64_t BN, int64_t BK, int mask_k,
                        const int64_t *tile_order, const int64_t *kblock_order,
                        double *C, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0 || BM <= 0 || BN <= 0 || BK <= 0) return OR_EINVAL;
  if (check_operand(M, K, lda, a_dtype, a_layout) ||
      check_operand(K, N, ldb, b_dtype, b_layout))
    return OR_EINVAL;
  if (ldc < (N > 0 ? N : 1)) return OR_EINVAL;
  const int64_t tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
  const int64_t kblocks = (K + BK - 1) / BK;
  if (!mask_k) {
    /* Every k the unmasked chunks touch must lie inside the caller's buffers. */
    const int64_t k_end = kblocks * BK;
    if (a_k_alloc < k_end || b_k_alloc < k_end) return OR_EBOUNDS;
    if (check_operand(M, k_end, lda, a_dtype, a_layout) ||
        check_operand(k_end, N, ldb, b_dtype, b_layout))
      return OR_EBOUNDS;
  }
  double *acc = (double *)malloc((size_t)BM * (size_t)BN * sizeof(double));
  if (!acc) return OR_ENOMEM;
  for (int64_t t = 0; t < tiles_m * tiles_n; ++t) {
    const int64_t tile = tile_order ? tile_order[t] : t;
    if (tile < 0 || tile >= tiles_m * tiles_n) { free(acc); return OR_EINVAL; }
    const int64_t pid_m = tile / tiles_n, pid_n = tile % tiles_n;
    for (int64_t x = 0; x < BM * BN; ++x) acc[x] = 0.0; /* initialised once, before the K-loop */
    for (int64_t s = 0; s < kblocks; ++s) {
      const int64_t kb = kblock_order ? kblock_order[s] : s;
      if (kb < 0 || kb >= kblocks) { free(acc); return OR_EINVAL; }
      for (int64_t r = 0; r < BM; ++r) {
        const int64_t i = pid_m * BM + r;
        for (int64_t c = 0; c < BN; ++c) {
          const int64_t j = pid_n * BN + c;
          double partial = 0.0; /* this chunk's contribution to acc[r][c] */
          for (int64_t kk = 0; kk < BK; ++kk) {
            const int64_t k = kb * BK + kk;
            const int k_ok = mask_k ? (k < K) : 1;
            const double a = (i < M && k_ok) ? dec_elem(A, a_dtype, elem_index(a_layout, lda, i, k)) : 0.0;
            const double b = (j < N && k_ok) ? dec_elem(B, b_dtype, elem_index(b_layout, ldb, k, j)) : 0.0;
            partial += a * b;
          }
          acc[r * BN + c] += partial;
        }
      }
    }
    for (int64_t r = 0; r < BM; ++r)
      for (int64_t c = 0; c < BN; ++c) {
        const int64_t i = pid_m * BM + r, j = pid_n * BN + c;
        if (i < M && j < N) C[i * ldc + j] = acc[r * BN + c];
      }
  }
  free(acc);
  return OR_OK;
}

/*
 * The fp16 accumulator of "Chapter 13: The Blocked Matmul Kernel", section 13.3,
 * Worked Example 13.3.1: for every output element the running total is an fp16
 * value that starts at zero; each K-chunk of BK elements contributes its dot
 * product rounded to fp16, and the running total is rounded to fp16 after every
 * addition. The result (fp16 values held in doubles) goes to C[i*ldc + j].
 */
int oracle_gemm_f16acc(int64_t M, int64_t N, int64_t K,
                       const void *A, int64_t lda, int a_dtype, int a_layout,
                       const void *B, int64_t ldb, int b_dtype, int b_layout,
                       int64_t BK, double *C, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0 || BK <= 0) return OR_EINVAL;
  if (check_operand(M, K, lda, a_dtype, a_layout) ||
      check_operand(K, N, ldb, b_dtype, b_layout))
    return OR_EINVAL;
  if (ldc < (N > 0 ? N : 1)) return OR_EINVAL;
  for (int64_t i = 0; i < M; ++i)
    for (int64_t j = 0; j < N; ++j) {
      double acc = 0.0;
      for (int64_t k0 = 0; k0 < K; k0 += BK) {
        double partial = 0.0;
        for (int64_t k = k0; k < k0 + BK && k < K; ++k)
          partial += dec_elem(A, a_dtype, elem_index(a_layout, lda, i, k)) *
                     dec_elem(B, b_dtype, elem_index(b_layout, ldb, k, j));
        acc = round_to(OR_F16, acc + round_to(OR_F16, partial));
      }
      C[i * ldc + j] = acc;
    }
  return OR_OK;
}

/* ------------------------------------------------------------ row softmax */

/* Row softmax of an M x N row-major matrix X (leading dimension ldx, any stored
 * format), written as fp64 to Y (leading dimension ldy). Per row, in the order of
 * the homework's kernel: the maximum m over the row's N values, then
 * p_j = exp(x_j - m), their sum l, and y_j = p_j / l. Only the N logical values
 * of a row take part: the kernel's -inf padding of the tile's extra columns adds
 * nothing to the max or the sum. IEEE rules apply throughout: a row holding a NaN
 * or +inf, or only -inf values, gives NaN (m - m or x - m is NaN). */
int oracle_softmax_rows(int64_t M, int64_t N, const void *X, int64_t ldx, int x_dtype,
                        double *Y, int64_t ldy) {
  if (M < 0 || N < 0 || x_dtype < OR_F32 || x_dtype > OR_F64) return OR_EINVAL;
  if (ldx < (N > 0 ? N : 1) || ldy < (N > 0 ? N : 1)) return OR_EINVAL;
  if (N == 0) return OR_OK;
  double *p = (double *)malloc((size_t)N * sizeof(double));
  if (!p) return OR_ENOMEM;
  for (int64_t i = 0; i < M; ++i) {
    double m = -INFINITY;
    int nan = 0;
    for (int64_t j = 0; j < N; ++j) {
      const double x = dec_elem(X, x_dtype, i * ldx + j);
      if (isnan(x)) nan = 1;
      if (x > m) m = x;
    }
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
      p[j] = exp(dec_elem(X, x_dtype, i * ldx + j) - m);
      l += p[j];
    }
    for (int64_t j = 0; j < N; ++j) Y[i * ldy + j] = nan ? NAN : p[j] / l;
  }
  free(p);
  return OR_OK;
}
