/*
 * oracle.c -- plain CPU reference for the dense GEMM path.
 *
 *   D = act(alpha * op(A) @ op(B) + beta * C)
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into liboracle.so and is
 * loaded by tests/, by __graft_entry__.smoke() and by the cpu_baseline /
 * reference legs of bench.py.  The GPU library never links, includes or calls
 * it, and it shares no code with dense_gemm_mma_gb300/csrc/.
 *
 * What it follows:
 *  - "Matrix Multiplication Background User's Guide", section 2 (Math and
 *    Memory Bounds): A is M x K, B is K x N, C is M x N; every output value is a
 *    dot product of K-element vectors (M*N*K fused multiply-adds).  The page's
 *    display formula for GEMM is lost in the extracted text; the reading taken
 *    is the BLAS one, D = alpha*A*B + beta*C.
 *  - "Learning Triton One Kernel at a Time: Matrix Multiplication", section
 *    Naive GEMM: one dot product per (row, column) pair, accumulated along the
 *    shared dimension; section Memory coalescing: row-major storage with a
 *    per-dimension stride, a transpose changes the strides, not the memory.
 *  - "OpenAI open-sources the Triton GPU language (part 2)", section Matrix
 *    multiplication: an output transform such as LeakyReLU fused after the
 *    product.  Reading taken: act is applied to alpha*AB + beta*C, and
 *    LeakyReLU(x) = x < 0 ? slope*x : x.  ReLU, GELU and SiLU are further
 *    transforms of the same kind, written from their definitions (apply_act).
 *  - "Matrix Multiplication Background User's Guide", section 2.2, Table 1:
 *    TF32 is one of the Tensor Core precisions.  Reading taken: a TF32
 *    operand is an fp32 word of which the sign, exponent and 10 highest
 *    fraction bits are used (the 13 lowest dropped, decode_tf32); products of
 *    two such values have at most 22 significant bits, so they are exact in
 *    fp32 as bf16/fp16 products are.
 *
 * Arithmetic: every bf16/fp16 input is decoded exactly to double; the dot
 * product is accumulated in double in ascending k; alpha, beta and the
 * activation are applied in double; the result is rounded ONCE to the output
 * format with round-to-nearest-even.  C is not read when beta == 0 (BLAS
 * convention).  Compile with -ffp-contract=off so that no multiply-add is
 * fused and the result is the same on every host.
 *
 * Pins (tests/test_oracle.py): the pages' worked (4,6)@(6,4) example split
 * into 3-element partial dot products and (2,2) blocks; identity and
 * permutation matrices; (A@B)^T = B^T@A^T through the transpose flags;
 * alpha/beta linearity; exact rational brute force for all M,N,K in 1..6;
 * the rounding and decoding routines against numpy and exact rationals;
 * the activations against tabulated values of the normal distribution
 * function and of exp, and the identity f(x) - f(-x) = x of GELU and SiLU.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* element formats */
enum { ORC_BF16 = 0, ORC_F16 = 1, ORC_F32 = 2, ORC_TF32 = 3 };

/* ---------------------------------------------------------------- decode */

/* bf16 is the top half of an IEEE binary32 word: widening is exact. */
static double decode_bf16(uint16_t h) {
  uint32_t w = (uint32_t)h << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m + 1024), e - 25); /* (1.m) * 2^(e-15) */
  return sign ? -v : v;
}

/* TF32 operand in an fp32 word: the tensor core uses the sign, the 8-bit
 * exponent and the 10 highest of the 23 fraction bits; the 13 lowest are
 * dropped (truncation of the significand toward zero). */
static double decode_tf32(uint32_t w) {
  w &= 0xFFFFE000u;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

double oracle_decode(uint32_t bits, int fmt) {
  if (fmt == ORC_BF16) return decode_bf16((uint16_t)bits);
  if (fmt == ORC_F16) return decode_f16((uint16_t)bits);
  if (fmt == ORC_TF32) return decode_tf32(bits);
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------- rounding */

/* Round x to a binary format with p significand bits (hidden bit included)
 * and minimum normal exponent emin, to nearest, ties to even.  Overflow is
 * not handled here.  x/q and r*q are exact because q is a power of two. */
static double round_to_precision(double x, int p, int emin) {
  if (x == 0.0 || !isfinite(x)) return x;
  int e;
  frexp(x, &e); /* |x| = f * 2^e with 0.5 <= f < 1, so floor(log2|x|) = e-1 */
  int ex = e - 1;
  if (ex < emin) ex = emin; /* subnormal range: fixed quantum */
  double q = ldexp(1.0, ex - (p - 1));
  return nearbyint(x / q) * q; /* default rounding mode: nearest-even */
}

uint16_t oracle_round_bf16(double x) {
  if (isnan(x)) return 0x7fc0;
  double r = round_to_precision(x, 8, -126);
  double maxf = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  if (fabs(r) > maxf) r = copysign(INFINITY, x);
  float f = (float)r; /* exact: r has at most 8 significant bits */
  uint32_t w;
  memcpy(&w, &f, sizeof w);
  return (uint16_t)(w >> 16);
}

uint16_t oracle_round_f16(double x) {
  if (isnan(x)) return 0x7e00;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double r = round_to_precision(x, 11, -14);
  double a = fabs(r);
  if (a > 65504.0) return sign | 0x7c00;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);
  int ex = e - 1;
  if (ex < -14) /* subnormal: a = m * 2^-24 */
    return sign | (uint16_t)ldexp(a, 24);
  uint16_t m = (uint16_t)(ldexp(a, 10 - ex) - 1024.0);
  return sign | (uint16_t)((ex + 15) << 10) | m;
}

float oracle_round_f32(double x) {
  return (float)x; /* C's double->float conversion rounds to nearest-even */
}

/* ---------------------------------------------------------------- access */

/* op(A)(i,k): transA == 0 -> A stored M x K row-major, A[i*lda + k];
 *             transA == 1 -> A stored K x M row-major, A[k*lda + i]. */
static double load_in(const void* p, int fmt, int64_t idx) {
  if (fmt == ORC_F32) return (double)((const float*)p)[idx];
  if (fmt == ORC_TF32) return decode_tf32(((const uint32_t*)p)[idx]);
  return oracle_decode(((const uint16_t*)p)[idx], fmt);
}

static double elem_a(const void* A, int64_t lda, int trans, int fmt, int64_t i, int64_t k) {
  return load_in(A, fmt, trans ? k * lda + i : i * lda + k);
}

/* op(B)(k,j): transB == 0 -> B stored K x N, B[k*ldb + j];
 *             transB == 1 -> B stored N x K, B[j*ldb + k]. */
static double elem_b(const void* B, int64_t ldb, int trans, int fmt, int64_t k, int64_t j) {
  return load_in(B, fmt, trans ? j * ldb + k : k * ldb + j);
}

static void store_out(void* D, int fmt, int64_t idx, double v) {
  if (fmt == ORC_F32)
    ((float*)D)[idx] = oracle_round_f32(v);
  else if (fmt == ORC_BF16)
    ((uint16_t*)D)[idx] = oracle_round_bf16(v);
  else
    ((uint16_t*)D)[idx] = oracle_round_f16(v);
}

/* ------------------------------------------------------------ the method */

/* The output transform, in double.  1: LeakyReLU, the pages' example of a
 * transform fused after the product.  2-4: further activations fused at the
 * same place, from their textbook definitions:
 *   ReLU(x) = x < 0 ? 0 : x              (-0 and NaN pass unchanged)
 *   GELU(x) = x * Phi(x),  Phi(x) = erfc(-x / sqrt(2)) / 2, the standard
 *             normal distribution function
 *   SiLU(x) = x * sigmoid(x) = x / (1 + exp(-x))
 * 0 (or any other code): identity. */
static double apply_act(double d, int act, double slope) {
  switch (act) {
    case 1: return d < 0.0 ? slope * d : d;
    case 2: return d < 0.0 ? 0.0 : d;
    case 3: return 0.5 * d * erfc(-d / sqrt(2.0));
    case 4: return d / (1.0 + exp(-d));
    default: return d;
  }
}

/* One output entry before output rounding: act(alpha * sum_k a(i,k) b(k,j) + beta * c(i,j)). */
double oracle_entry(int64_t i, int64_t j, int64_t K,
                    const void* A, int64_t lda, const void* B, int64_t ldb,
                    const void* C, int64_t ldc, double alpha, double beta,
                    int in_fmt, int c_fmt, int transA, int transB,
                    int act, double slope) {
  double s = 0.0;
  for (int64_t k = 0; k < K; ++k)
    s += elem_a(A, lda, transA, in_fmt, i, k) * elem_b(B, ldb, transB, in_fmt, k, j);
  double d = alpha * s;
  if (beta != 0.0) d += beta * load_in(C, c_fmt, i * ldc + j);
  return apply_act(d, act, slope);
}

/* Full product.  D_exact (M x N doubles, row stride N) receives the value
 * before output rounding; D_out (M x N in out_fmt, row stride N) receives it
 * rounded once.  Either may be NULL.  C is stored in c_fmt (the output's
 * format when C is updated in place; any format for a separate C).  Returns
 * 0, or -1 on a bad argument. */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, const void* B, int64_t ldb,
                const void* C, int64_t ldc, double alpha, double beta,
                int in_fmt, int out_fmt, int c_fmt, int transA, int transB,
                int act, double slope, double* D_exact, void* D_out) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (in_fmt != ORC_BF16 && in_fmt != ORC_F16 && in_fmt != ORC_TF32) return -1;
  if (out_fmt != ORC_BF16 && out_fmt != ORC_F16 && out_fmt != ORC_F32) return -1;
  if (c_fmt != ORC_BF16 && c_fmt != ORC_F16 && c_fmt != ORC_F32) return -1;
  if (beta != 0.0 && C == NULL) return -1;
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double d = oracle_entry(i, j, K, A, lda, B, ldb, C, ldc, alpha, beta,
                              in_fmt, c_fmt, transA, transB, act, slope);
      if (D_exact) D_exact[i * N + j] = d;
      if (D_out) store_out(D_out, out_fmt, i * N + j, d);
    }
  }
  return 0;
}

/* Sampled check: n entries (rows[t], cols[t]), same outputs as oracle_gemm. */
int oracle_sample(int64_t n, const int64_t* rows, const int64_t* cols, int64_t K,
                  const void* A, int64_t lda, const void* B, int64_t ldb,
                  const void* C, int64_t ldc, double alpha, double beta,
                  int in_fmt, int out_fmt, int c_fmt, int transA, int transB,
                  int act, double slope, double* D_exact, void* D_out) {
  if (n < 0 || K < 0) return -1;
  if (beta != 0.0 && C == NULL) return -1;
  for (int64_t t = 0; t < n; ++t) {
    double d = oracle_entry(rows[t], cols[t], K, A, lda, B, ldb, C, ldc, alpha, beta,
                            in_fmt, c_fmt, transA, transB, act, slope);
    if (D_exact) D_exact[t] = d;
    if (D_out) store_out(D_out, out_fmt, t, d);
  }
  return 0;
}
