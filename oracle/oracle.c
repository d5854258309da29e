/*
 * oracle.c -- plain fp64 CPU reference for the fgemm library.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
 * Python binding) links, loads or calls this file.  Only the tests, the smoke
 * check and the CPU-baseline leg of the benchmark use it.  It shares no code,
 * header, table or constant with the GPU path.
 *
 * What it computes, and where each piece comes from:
 *
 *  - Inputs are 16-bit floats (fp16 or bf16).  They are decoded bit by bit to
 *    double, exactly (sign, exponent, mantissa, subnormals, Inf/NaN).  The
 *    16-bit-input / wide-accumulator pattern is the one the CS336 Lecture 05
 *    notes describe on "Page 26. Low precision drives faster matrix
 *    multiplies"; here the accumulator is fp64, wider than the GPU's fp32.
 *
 *  - Classical product: C[i][j] = sum_k A[i][k] * B[k][j], a plain triple
 *    loop, k ascending (CS336 Lecture 05 notes, "Page 40. Trick 5: tiling",
 *    the definition P_ij = sum_k M_ik N_kj).
 *
 *  - Epilogue, applied to the accumulator before the store (PingPong GEMM /
 *    CODA note, opening section: mainloop, then scaling and elementwise ops in
 *    the epilogue; the CODA section names SwiGLU):
 *        v = alpha * acc + bias[j]        (bias optional)
 *        NONE / SCALE_BIAS : out = v
 *        SILU              : out = v / (1 + exp(-v))
 *        SWIGLU            : out[i][j] = silu(v[i][j]) * v[i][j + N/2],
 *                            output width N/2 (gate = first half, up = second).
 *
 *  - Strassen-like low-complexity product (FalconGEMM summary, "Methodology"
 *    items 1 and 4: Strassen-like LCMAs with a recursion depth).  The pages do
 *    not print the identities; the oracle uses the textbook one-level Strassen
 *    scheme (seven half-size products):
 *        M1 = (A11 + A22)(B11 + B22)     M5 = (A11 + A12) B22
 *        M2 = (A21 + A22) B11            M6 = (A21 - A11)(B11 + B12)
 *        M3 = A11 (B12 - B22)            M7 = (A12 - A22)(B21 + B22)
 *        M4 = A22 (B21 - B11)
 *        C11 = M1 + M4 - M5 + M7         C12 = M3 + M5
 *        C21 = M2 + M4                   C22 = M1 - M2 + M3 + M6
 *    applied recursively `depth` times, classical at the leaves.  In exact
 *    arithmetic it equals the classical product.
 *
 *  - RMSNorm statistics carried by the epilogue (PingPong GEMM / CODA note,
 *    CODA section: the epilogue also produces what the following
 *    normalisation needs).  RMSNorm of a row x of width n with gain g:
 *        y_j = x_j * g_j / sqrt(mean_j(x_j^2) + eps)
 *    The producing GEMM emits, per row and per block of 64 output columns,
 *    the sum of squares of its (rounded) outputs; the consuming GEMM forms
 *        r_i = 1 / sqrt(sum over blocks / n + eps)
 *    and since  y W = diag(r) x diag(g) W,  it multiplies its accumulator
 *    row i by r_i, with g folded into its weights once.
 *
 *  - Block-scaled 8-bit inputs (MX: CS336 Lecture 05 notes, "Page 27.
 *    Frontiers in low precision - FP8 and MXFP8").  An element is an 8-bit
 *    float, E4M3
 *    (bias 7, S.1111.111 is NaN, no infinity) or E5M2 (bias 15, IEEE-like
 *    infinities and NaNs), and every 32 consecutive elements along K share a
 *    power-of-two scale stored as E8M0 (value 2^(e - 127), e = 255 is NaN).
 *    Its value is element * scale; the MX product is the classical product
 *    of those values.
 *
 *  - Winograd's variant of Strassen (named beside Strassen among the
 *    Strassen-like LCMAs of the FalconGEMM summary, "Methodology" item 1; the
 *    pages print no formulas, so the oracle uses the standard variant).  It
 *    still multiplies seven half-size products but builds its operands and
 *    the output from shared partial sums:
 *        S1 = A21 + A22   S2 = S1 - A11   S3 = A11 - A21   S4 = A12 - S2
 *        T1 = B12 - B11   T2 = B22 - T1   T3 = B22 - B12   T4 = T2 - B21
 *        P1 = A11 B11   P2 = A12 B21   P3 = S4 B22   P4 = A22 T4
 *        P5 = S1 T1     P6 = S2 T2     P7 = S3 T3
 *        U1 = P1 + P2   U2 = P1 + P6   U3 = U2 + P7   U4 = U2 + P5
 *        U5 = U4 + P3   U6 = U3 - P4   U7 = U3 + P5
 *        C11 = U1   C12 = U5   C21 = U6   C22 = U7
 *    applied recursively `depth` times, classical at the leaves (15 block
 *    additions per level against Strassen's 18).
 *
 *  - Emulated Strassen: the same recursion, except that every leaf operand
 *    (an exact signed sum of source blocks) is rounded first to fp32 and then
 *    to the 16-bit input type, round-to-nearest-even, because a tensor core
 *    can only multiply 16-bit operands.  This predicts the rounding structure
 *    of a GPU implementation that forms each operand sum in fp32 and rounds
 *    it once.
 *
 * Compiled with -ffp-contract=off so that no multiply-add is fused and the
 * results are the same on every host architecture.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };
enum { ORACLE_EPI_NONE = 0, ORACLE_EPI_SCALE_BIAS = 1, ORACLE_EPI_SILU = 2,
       ORACLE_EPI_SWIGLU = 3 };

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- decoding */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double oracle_f16_value(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);              /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25); /* (1.m) * 2^(e-15) */
  return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits. */
double oracle_bf16_value(uint16_t b) {
  int sign = (b >> 15) & 1;
  int e = (b >> 7) & 0xff;
  int m = b & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)m, -133);             /* subnormal: m * 2^-133 */
  else if (e == 255)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x80), e - 134); /* (1.m) * 2^(e-127) */
  return sign ? -v : v;
}

static double decode_one(int dtype, uint16_t x) {
  return dtype == ORACLE_F16 ? oracle_f16_value(x) : oracle_bf16_value(x);
}

void oracle_decode(int dtype, int64_t n, const uint16_t* in, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = decode_one(dtype, in[i]);
}

/* ---------------------------------------------------------------- encoding */

/*
 * Round a double to a binary format with `p` significand bits (incl. the
 * hidden one), minimum normal exponent `emin`, exponent bias `bias` and
 * exponent field width `ebits`, round-to-nearest-even, and return its bits.
 */
static uint16_t encode_rne(double x, int p, int emin, int bias, int ebits) {
  const int mbits = p - 1;
  const uint16_t sign = signbit(x) ? (uint16_t)(1u << (mbits + ebits)) : 0;
  const uint16_t inf_bits = (uint16_t)(((1u << ebits) - 1u) << mbits);
  if (isnan(x)) return (uint16_t)(inf_bits | (1u << (mbits - 1)));
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | inf_bits);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);            /* a = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;           /* a in [2^E, 2^(E+1)) */
  int ulp_exp = (E < emin) ? (emin - mbits) : (E - mbits);
  double q = ldexp(a, -ulp_exp);   /* exact: power-of-two scaling */
  double r = nearbyint(q);         /* default mode: nearest, ties to even */
  if (r == 0.0) return sign;
  if (r >= ldexp(1.0, p)) {        /* carry into the next binade */
    r = ldexp(r, -1);
    ulp_exp += 1;
  }
  uint32_t ri = (uint32_t)r;
  if (ulp_exp == emin - mbits && ri < (1u << mbits)) {
    return (uint16_t)(sign | ri);  /* subnormal */
  }
  int efield = ulp_exp + mbits + bias;
  if (efield >= (1 << ebits) - 1) return (uint16_t)(sign | inf_bits);
  return (uint16_t)(sign | ((uint32_t)efield << mbits) | (ri - (1u << mbits)));
}

uint16_t oracle_f64_to_f16(double x) { return encode_rne(x, 11, -14, 15, 5); }
uint16_t oracle_f64_to_bf16(double x) { return encode_rne(x, 8, -126, 127, 8); }

void oracle_encode(int dtype, int64_t n, const double* in, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = dtype == ORACLE_F16 ? oracle_f64_to_f16(in[i])
                                 : oracle_f64_to_bf16(in[i]);
}

/* Round to the 16-bit type and back (identity for ORACLE_F64). */
static double round_to(int dtype, double x) {
  if (dtype == ORACLE_F64) return x;
  return dtype == ORACLE_F16 ? oracle_f16_value(oracle_f64_to_f16(x))
                             : oracle_bf16_value(oracle_f64_to_bf16(x));
}

/* ------------------------------------------------------- classical product */

/* C[M x N] = A[M x K] * B[K x N], all row-major with leading dimensions. */
void oracle_gemm_f64(int64_t M, int64_t N, int64_t K, const double* A,
                     int64_t lda, const double* B, int64_t ldb, double* C,
                     int64_t ldc) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double s = 0.0;
      for (int64_t k = 0; k < K; ++k) s += A[i * lda + k] * B[k * ldb + j];
      C[i * ldc + j] = s;
    }
  }
}

/*
 * Sampled entries of the raw product of 16-bit inputs:
 *   out[t] = sum_k A[rows[t]][k] * B[k][cols[t]]   (k ascending, fp64),
 * decoding A and B on the fly so that large inputs need no fp64 copy.
 */
void oracle_gemm_sampled(int dtype, int64_t K, const uint16_t* A, int64_t lda,
                         const uint16_t* B, int64_t ldb, int64_t n,
                         const int64_t* rows, const int64_t* cols,
                         double* out) {
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t t = 0; t < n; ++t) {
    const uint16_t* a = A + rows[t] * lda;
    const uint16_t* b = B + cols[t];
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
      s += decode_one(dtype, a[k]) * decode_one(dtype, b[k * ldb]);
    out[t] = s;
  }
}

/* ---------------------------------------------------------------- epilogue */

double oracle_silu(double v) { return v / (1.0 + exp(-v)); }

/*
 * out = epilogue(alpha * acc + bias).  acc is M x N (ld ldacc); bias has N
 * entries or is NULL.  For SWIGLU the output is M x N/2: silu of the first
 * half times the second half.
 */
void oracle_epilogue(int kind, int64_t M, int64_t N, const double* acc,
                     int64_t ldacc, double alpha, const double* bias,
                     double* out, int64_t ldo) {
  const int64_t Nout = (kind == ORACLE_EPI_SWIGLU) ? N / 2 : N;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < Nout; ++j) {
      double v = alpha * acc[i * ldacc + j] + (bias ? bias[j] : 0.0);
      double o;
      if (kind == ORACLE_EPI_SILU) {
        o = oracle_silu(v);
      } else if (kind == ORACLE_EPI_SWIGLU) {
        double u = alpha * acc[i * ldacc + j + Nout] +
                   (bias ? bias[j + Nout] : 0.0);
        o = oracle_silu(v) * u;
      } else {
        o = v;
      }
      out[i * ldo + j] = o;
    }
  }
}

/* ------------------------------------------------------ 8-bit MX inputs */

/* fmt 0: E4M3 (1 sign, 4 exponent bits, bias 7, 3 mantissa bits; exponent
 * and mantissa all ones is NaN, no infinity).  fmt 1: E5M2 (5 exponent bits,
 * bias 15, 2 mantissa bits; exponent all ones: infinity if the mantissa is 0,
 * else NaN).  Exponent 0: subnormal, mantissa * 2^(1 - bias - mbits). */
static double fp8_value(int fmt, uint8_t x) {
  const int ebits = fmt == 0 ? 4 : 5, mbits = fmt == 0 ? 3 : 2;
  const int bias = fmt == 0 ? 7 : 15;
  const int sign = x >> 7;
  const int e = (x >> mbits) & ((1 << ebits) - 1);
  const int m = x & ((1 << mbits) - 1);
  double v;
  if (fmt == 0 && e == 15 && m == 7) return NAN;
  if (fmt == 1 && e == 31) {
    if (m != 0) return NAN;
    v = INFINITY;
  } else if (e == 0) {
    v = ldexp((double)m, 1 - bias - mbits);
  } else {
    v = ldexp(1.0 + (double)m / (double)(1 << mbits), e - bias);
  }
  return sign ? -v : v;
}

void oracle_fp8_decode(int fmt, int64_t n, const uint8_t* in, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = fp8_value(fmt, in[i]);
}

/* E8M0 scale: 2^(e - 127); e = 255 is NaN. */
static double e8m0_value(uint8_t e) { return e == 255 ? NAN : ldexp(1.0, (int)e - 127); }

void oracle_e8m0_decode(int64_t n, const uint8_t* in, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e8m0_value(in[i]);
}

/* Value of a block-scaled matrix X (rows x cols, 8-bit elements, ld ldx).
 * along == 0: blocks of 32 run along a row, S[r * lds + c / 32];
 * along == 1: blocks of 32 run down a column, S[(r / 32) * lds + c]. */
void oracle_mx_values(int fmt, int along, int64_t rows, int64_t cols, const uint8_t* X,
                      int64_t ldx, const uint8_t* S, int64_t lds, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      const uint8_t e = along == 0 ? S[r * lds + c / 32] : S[(r / 32) * lds + c];
      out[r * cols + c] = fp8_value(fmt, X[r * ldx + c]) * e8m0_value(e);
    }
}

/* ------------------------------------------------------- RMSNorm pieces */

/* y = RMSNorm(x) row by row: y_ij = x_ij * g_j / sqrt(mean_j x_ij^2 + eps)
 * (g may be NULL: all ones). */
void oracle_rmsnorm(int64_t M, int64_t N, const double* x, int64_t ldx,
                    const double* g, double eps, double* y, int64_t ldy) {
  for (int64_t i = 0; i < M; ++i) {
    double ss = 0.0;
    for (int64_t j = 0; j < N; ++j) ss += x[i * ldx + j] * x[i * ldx + j];
    const double r = 1.0 / sqrt(ss / (double)N + eps);
    for (int64_t j = 0; j < N; ++j)
      y[i * ldy + j] = x[i * ldx + j] * r * (g ? g[j] : 1.0);
  }
}

/* Per row i and block p of 64 columns: out[p * M + i] = sum of x_ij^2 over
 * the block's columns j < N (the last block may be partial). */
void oracle_block_sumsq(int64_t M, int64_t N, const double* x, int64_t ldx,
                        double* out) {
  const int64_t parts = (N + 63) / 64;
  for (int64_t p = 0; p < parts; ++p)
    for (int64_t i = 0; i < M; ++i) {
      double ss = 0.0;
      for (int64_t j = p * 64; j < N && j < (p + 1) * 64; ++j)
        ss += x[i * ldx + j] * x[i * ldx + j];
      out[p * M + i] = ss;
    }
}

/* r_i = 1 / sqrt(sum_p sumsq[p * M + i] / n + eps). */
void oracle_row_scale(int64_t M, int64_t parts, const double* sumsq, double n,
                      double eps, double* r) {
  for (int64_t i = 0; i < M; ++i) {
    double ss = 0.0;
    for (int64_t p = 0; p < parts; ++p) ss += sumsq[p * M + i];
    r[i] = 1.0 / sqrt(ss / n + eps);
  }
}

/* ------------------------------------------------------ Strassen recursion */

/* A leaf operand: fp32 first, then the 16-bit type (no rounding for F64). */
static double round_leaf(int dtype, double x) {
  if (dtype == ORACLE_F64) return x;
  return round_to(dtype, (double)(float)x);
}

/* dst[r x c] = sa * X + sb * Y  (Y may be NULL: dst = sa * X). */
static void combine(int64_t r, int64_t c, double sa, const double* X,
                    int64_t ldx, double sb, const double* Y, int64_t ldy,
                    double* dst, int64_t ldd) {
  for (int64_t i = 0; i < r; ++i)
    for (int64_t j = 0; j < c; ++j)
      dst[i * ldd + j] =
          sa * X[i * ldx + j] + (Y ? sb * Y[i * ldy + j] : 0.0);
}

/*
 * Recursive Strassen.  `round_dtype` < 0: exact (every operand sum in fp64).
 * Otherwise every leaf operand is rounded to fp32 and then to that 16-bit
 * type before the classical leaf product (the emulated form).
 */
static void strassen_rec(int depth, int round_dtype, int64_t M, int64_t N,
                         int64_t K, const double* A, int64_t lda,
                         const double* B, int64_t ldb, double* C,
                         int64_t ldc) {
  if (depth == 0) {
    if (round_dtype < 0) {
      oracle_gemm_f64(M, N, K, A, lda, B, ldb, C, ldc);
      return;
    }
    double* Ar = (double*)malloc(sizeof(double) * (size_t)(M * K));
    double* Br = (double*)malloc(sizeof(double) * (size_t)(K * N));
    for (int64_t i = 0; i < M; ++i)
      for (int64_t k = 0; k < K; ++k)
        Ar[i * K + k] = round_leaf(round_dtype, A[i * lda + k]);
    for (int64_t k = 0; k < K; ++k)
      for (int64_t j = 0; j < N; ++j)
        Br[k * N + j] = round_leaf(round_dtype, B[k * ldb + j]);
    oracle_gemm_f64(M, N, K, Ar, K, Br, N, C, ldc);
    free(Ar);
    free(Br);
    return;
  }
  const int64_t m = M / 2, n = N / 2, k = K / 2;
  const double* A11 = A;
  const double* A12 = A + k;
  const double* A21 = A + m * lda;
  const double* A22 = A + m * lda + k;
  const double* B11 = B;
  const double* B12 = B + n;
  const double* B21 = B + k * ldb;
  const double* B22 = B + k * ldb + n;
  double* S = (double*)malloc(sizeof(double) * (size_t)(m * k));
  double* T = (double*)malloc(sizeof(double) * (size_t)(k * n));
  double* P[7];
  for (int q = 0; q < 7; ++q)
    P[q] = (double*)malloc(sizeof(double) * (size_t)(m * n));

  /* M1 = (A11 + A22)(B11 + B22) */
  combine(m, k, 1, A11, lda, 1, A22, lda, S, k);
  combine(k, n, 1, B11, ldb, 1, B22, ldb, T, n);
  strassen_rec(depth - 1, round_dtype, m, n, k, S, k, T, n, P[0], n);
  /* M2 = (A21 + A22) B11 */
  combine(m, k, 1, A21, lda, 1, A22, lda, S, k);
  combine(k, n, 1, B11, ldb, 0, NULL, 0, T, n);
  strassen_rec(depth - 1, round_dtype, m, n, k, S, k, T, n, P[1], n);
  /* M3 = A11 (B12 - B22) */
  combine(m, k, 1, A11, lda, 0, NULL, 0, S, k);
  combine(k, n, 1, B12, ldb, -1, B22, ldb, T, n);
  strassen_rec(depth - 1, round_dtype, m, n, k, S, k, T, n, P[2], n);
  /* M4 = A22 (B21 - B11) */
  combine(m, k, 1, A22, lda, 0, NULL, 0, S, k);
  combine(k, n, 1, B21, ldb, -1, B11, ldb, T, n);
  strassen_rec(depth - 1, round_dtype, m, n, k, S, k, T, n, P[3], n);
  /* M5 = (A11 + A12) B22 */
  combine(m, k, 1, A11, lda, 1, A12, lda, S, k);
  combine(k, n, 1, B22, ldb, 0, NULL, 0, T, n);
  strassen_rec(depth - 1, round_dtype, m, n, k, S, k, T, n, P[4], n);
  /* M6 = (A21 - A11)(B11 + B12) */
  combine(m, k, 1, A21, lda, -1, A11, lda, S, k);
  combine(k, n, 1, B11, ldb, 1, B12, ldb, T, n);
  strassen_rec(depth - 1, round_dtype, m, n, k, S, k, T, n, P[5], n);
  /* M7 = (A12 - A22)(B21 + B22) */
  combine(m, k, 1, A12, lda, -1, A22, lda, S, k);
  combine(k, n, 1, B21, ldb, 1, B22, ldb, T, n);
  strassen_rec(depth - 1, round_dtype, m, n, k, S, k, T, n, P[6], n);

  for (int64_t i = 0; i < m; ++i) {
    for (int64_t j = 0; j < n; ++j) {
      const int64_t t = i * n + j;
      C[i * ldc + j] = P[0][t] + P[3][t] - P[4][t] + P[6][t];           /* C11 */
      C[i * ldc + j + n] = P[2][t] + P[4][t];                           /* C12 */
      C[(i + m) * ldc + j] = P[1][t] + P[3][t];                         /* C21 */
      C[(i + m) * ldc + j + n] = P[0][t] - P[1][t] + P[2][t] + P[5][t]; /* C22 */
    }
  }
  for (int q = 0; q < 7; ++q) free(P[q]);
  free(S);
  free(T);
}

/*
 * Recursive Winograd variant, in the notation of the header.  The partial
 * sums S1..S4 and T1..T4 are formed exactly (fp64) at every level, so with
 * `round_dtype` >= 0 a leaf operand is rounded once, from the exact signed
 * sum of source blocks it stands for (S2 = A21 + A22 - A11, ...).
 */
static void winograd_rec(int depth, int round_dtype, int64_t M, int64_t N,
                         int64_t K, const double* A, int64_t lda,
                         const double* B, int64_t ldb, double* C,
                         int64_t ldc) {
  if (depth == 0) {
    strassen_rec(0, round_dtype, M, N, K, A, lda, B, ldb, C, ldc);
    return;
  }
  const int64_t m = M / 2, n = N / 2, k = K / 2;
  const double* A11 = A;
  const double* A12 = A + k;
  const double* A21 = A + m * lda;
  const double* A22 = A + m * lda + k;
  const double* B11 = B;
  const double* B12 = B + n;
  const double* B21 = B + k * ldb;
  const double* B22 = B + k * ldb + n;
  double* S1 = (double*)malloc(sizeof(double) * (size_t)(m * k));
  double* S2 = (double*)malloc(sizeof(double) * (size_t)(m * k));
  double* S3 = (double*)malloc(sizeof(double) * (size_t)(m * k));
  double* S4 = (double*)malloc(sizeof(double) * (size_t)(m * k));
  double* T1 = (double*)malloc(sizeof(double) * (size_t)(k * n));
  double* T2 = (double*)malloc(sizeof(double) * (size_t)(k * n));
  double* T3 = (double*)malloc(sizeof(double) * (size_t)(k * n));
  double* T4 = (double*)malloc(sizeof(double) * (size_t)(k * n));
  double* P[7];
  for (int q = 0; q < 7; ++q)
    P[q] = (double*)malloc(sizeof(double) * (size_t)(m * n));

  combine(m, k, 1, A21, lda, 1, A22, lda, S1, k);  /* S1 = A21 + A22 */
  combine(m, k, 1, S1, k, -1, A11, lda, S2, k);    /* S2 = S1 - A11 */
  combine(m, k, 1, A11, lda, -1, A21, lda, S3, k); /* S3 = A11 - A21 */
  combine(m, k, 1, A12, lda, -1, S2, k, S4, k);    /* S4 = A12 - S2 */
  combine(k, n, 1, B12, ldb, -1, B11, ldb, T1, n); /* T1 = B12 - B11 */
  combine(k, n, 1, B22, ldb, -1, T1, n, T2, n);    /* T2 = B22 - T1 */
  combine(k, n, 1, B22, ldb, -1, B12, ldb, T3, n); /* T3 = B22 - B12 */
  combine(k, n, 1, T2, n, -1, B21, ldb, T4, n);    /* T4 = T2 - B21 */

  winograd_rec(depth - 1, round_dtype, m, n, k, A11, lda, B11, ldb, P[0], n); /* P1 */
  winograd_rec(depth - 1, round_dtype, m, n, k, A12, lda, B21, ldb, P[1], n); /* P2 */
  winograd_rec(depth - 1, round_dtype, m, n, k, S4, k, B22, ldb, P[2], n);    /* P3 */
  winograd_rec(depth - 1, round_dtype, m, n, k, A22, lda, T4, n, P[3], n);    /* P4 */
  winograd_rec(depth - 1, round_dtype, m, n, k, S1, k, T1, n, P[4], n);       /* P5 */
  winograd_rec(depth - 1, round_dtype, m, n, k, S2, k, T2, n, P[5], n);       /* P6 */
  winograd_rec(depth - 1, round_dtype, m, n, k, S3, k, T3, n, P[6], n);       /* P7 */

  for (int64_t i = 0; i < m; ++i) {
    for (int64_t j = 0; j < n; ++j) {
      const int64_t t = i * n + j;
      const double u1 = P[0][t] + P[1][t];
      const double u2 = P[0][t] + P[5][t];
      const double u3 = u2 + P[6][t];
      const double u4 = u2 + P[4][t];
      const double u5 = u4 + P[2][t];
      const double u6 = u3 - P[3][t];
      const double u7 = u3 + P[4][t];
      C[i * ldc + j] = u1;                 /* C11 */
      C[i * ldc + j + n] = u5;             /* C12 */
      C[(i + m) * ldc + j] = u6;           /* C21 */
      C[(i + m) * ldc + j + n] = u7;       /* C22 */
    }
  }
  for (int q = 0; q < 7; ++q) free(P[q]);
  free(S1);
  free(S2);
  free(S3);
  free(S4);
  free(T1);
  free(T2);
  free(T3);
  free(T4);
}

/* Returns 0, or -1 if M, N, K are not divisible by 2^depth. */
int oracle_winograd_f64(int depth, int64_t M, int64_t N, int64_t K,
                        const double* A, int64_t lda, const double* B,
                        int64_t ldb, double* C, int64_t ldc) {
  const int64_t g = (int64_t)1 << depth;
  if (depth < 0 || M % g || N % g || K % g) return -1;
  winograd_rec(depth, -1, M, N, K, A, lda, B, ldb, C, ldc);
  return 0;
}

/* Same recursion with leaf operands rounded to `dtype` (0 f16, 1 bf16, 2 none). */
int oracle_winograd_emulated(int depth, int dtype, int64_t M, int64_t N,
                             int64_t K, const double* A, int64_t lda,
                             const double* B, int64_t ldb, double* C,
                             int64_t ldc) {
  const int64_t g = (int64_t)1 << depth;
  if (depth < 0 || M % g || N % g || K % g) return -1;
  if (dtype < 0 || dtype > 2) return -1;
  winograd_rec(depth, dtype, M, N, K, A, lda, B, ldb, C, ldc);
  return 0;
}

/* Returns 0, or -1 if M, N, K are not divisible by 2^depth. */
int oracle_strassen_f64(int depth, int64_t M, int64_t N, int64_t K,
                        const double* A, int64_t lda, const double* B,
                        int64_t ldb, double* C, int64_t ldc) {
  const int64_t g = (int64_t)1 << depth;
  if (depth < 0 || M % g || N % g || K % g) return -1;
  strassen_rec(depth, -1, M, N, K, A, lda, B, ldb, C, ldc);
  return 0;
}

/* Same recursion with leaf operands rounded to `dtype` (0 f16, 1 bf16, 2 none). */
int oracle_strassen_emulated(int depth, int dtype, int64_t M, int64_t N,
                             int64_t K, const double* A, int64_t lda,
                             const double* B, int64_t ldb, double* C,
                             int64_t ldc) {
  const int64_t g = (int64_t)1 << depth;
  if (depth < 0 || M % g || N % g || K % g) return -1;
  if (dtype < 0 || dtype > 2) return -1;
  strassen_rec(depth, dtype, M, N, K, A, lda, B, ldb, C, ldc);
  return 0;
}
