/*
 * oracle_gemm.c -- the CPU oracle for dense GEMM.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
 * file.  The library never links, loads or calls it, and it shares no code,
 * header or constant with the library.
 *
 * What it computes is the plain definition of the operation described on
 * "bare-metal-bard" (ethanyanxu.com), first paragraph: the textbook matmul in
 * which one thread computes one output element, extended by the usual BLAS
 * scaling C = alpha * op(A) * op(B) + beta * C.  For every output element the
 * oracle walks k = 0 .. K-1 in ascending order and accumulates in IEEE double:
 *
 *     Cref[i][j] = alpha * sum_k r(opA[i][k]) * r(opB[k][j]) + beta * Cin[i][j]
 *     D[i][j]    =         sum_k |r(opA[i][k])| * |r(opB[k][j])|
 *
 * D is the scale used by the error metric err = |C - Cref| / D.
 *
 * r() is the precision of the mode's operands:
 *   FP32 : the fp32 value itself.
 *   TF32 : the fp32 value reduced to TF32 (sign, 8-bit exponent, 10 explicit
 *          mantissa bits).  The first paragraph of "bare-metal-bard" says TF32
 *          trades accuracy for speed but not how fp32 inputs are reduced; two
 *          readings are offered: dropping the 13 low mantissa bits
 *          (truncation toward zero) or rounding to nearest with ties away from
 *          zero.  The caller chooses.
 *   BF16 : the inputs arrive as bfloat16 bit patterns and are widened exactly.
 *   FP8  : the inputs arrive as 8-bit E4M3 codes and are decoded exactly.  The
 *          pages name FP8 among the tensor-core input types ("Tensor Cores:
 *          Matrix Instructions, Swizzling and FP8, Measured" and "Low-Precision
 *          Kernels: INT4, INT8 and FP8 Matmuls, Measured", their summaries)
 *          without defining it; the reading taken is the E4M3 format of the
 *          OCP 8-bit floating-point specification: 1 sign bit, 4 exponent bits
 *          with bias 7, 3 mantissa bits, subnormals at exponent 0, no
 *          infinities, and S.1111.111 the only NaN pattern (largest finite
 *          magnitude 448).  Per-tensor scale factors are the caller's alpha.
 *   FP8 E5M2 and the mixed pairs: E5M2 is the specification's other 8-bit
 *          format: 1 sign bit, 5 exponent bits with bias 15, 2 mantissa bits,
 *          subnormals at exponent 0, and exponent 31 holding the infinities
 *          (mantissa 0) and NaNs as in IEEE 754 (largest finite magnitude
 *          57344).  Mixed modes take A in one format and B in the other.
 *
 * Conventions the pages leave open (BLAS readings): when K == 0 or alpha == 0
 * A and B are not read; when beta == 0 Cin is not read, so a NaN there does
 * not reach the result.
 *
 * Matrices are row-major.  op(A) is M x K: stored M x K (lda >= K) when
 * transA == 0, or K x M (lda >= M) when transA == 1.  op(B) is K x N: stored
 * K x N (ldb >= N) when transB == 0, or N x K (ldb >= K) when transB == 1.
 *
 * Rows row0 .. row1-1 of the result are produced (a sample of rows for large
 * shapes); output row i is stored at Cref[(i - row0) * ldr + j].  Rows are
 * spread over OpenMP threads; each element is still a plain ascending-k loop.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORACLE_MODE_FP32 0
#define ORACLE_MODE_TF32 1
#define ORACLE_MODE_BF16 2
#define ORACLE_MODE_FP8_E4M3 3
#define ORACLE_MODE_FP8_E5M2 4
#define ORACLE_MODE_FP8_E4M3_E5M2 5 /* A E4M3, B E5M2 */
#define ORACLE_MODE_FP8_E5M2_E4M3 6 /* A E5M2, B E4M3 */

/* What one operand holds. */
enum { KIND_FP32, KIND_TF32, KIND_BF16, KIND_E4M3, KIND_E5M2 };

#define ORACLE_TF32_TRUNCATE 0
#define ORACLE_TF32_NEAREST_AWAY 1

static uint32_t float_bits(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  return u;
}

static float bits_float(uint32_t u) {
  float x;
  memcpy(&x, &u, sizeof x);
  return x;
}

/* TF32 keeps the top 19 bits of an fp32 pattern (1 sign, 8 exponent, 10
 * mantissa).  NaN and Inf pass through unchanged (a NaN keeps its payload so
 * that it stays a NaN). */
float oracle_tf32_truncate(float x) {
  uint32_t u = float_bits(x);
  if ((u & 0x7f800000u) == 0x7f800000u) return x;
  return bits_float(u & 0xffffe000u);
}

/* Round to the nearest TF32 value, ties away from zero: add half of the
 * dropped range (bit 12) to the magnitude, then drop the 13 low bits.  A carry
 * out of the mantissa steps the exponent, which is the correct rounding; a
 * carry into the all-ones exponent gives Inf, which is the correct overflow. */
float oracle_tf32_nearest_away(float x) {
  uint32_t u = float_bits(x);
  if ((u & 0x7f800000u) == 0x7f800000u) return x;
  uint32_t sign = u & 0x80000000u;
  uint32_t mag = (u & 0x7fffffffu) + 0x00001000u;
  return bits_float(sign | (mag & 0x7fffe000u));
}

/* A bfloat16 value is the upper half of an fp32 pattern; widening is exact. */
double oracle_bf16_to_double(uint16_t b) {
  return (double)bits_float((uint32_t)b << 16);
}

/* An E4M3 code as a double.  Fields: s = bit 7, e = bits 6..3, m = bits 2..0.
 *   e == 15 and m == 7 : NaN (either sign)
 *   e == 0             : (-1)^s * (m / 8) * 2^(1 - 7)       (zero and subnormals)
 *   otherwise          : (-1)^s * (1 + m / 8) * 2^(e - 7)
 * Every value is a small integer times a power of two, so ldexp is exact. */
double oracle_e4m3_to_double(uint8_t code) {
  const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = (e == 0) ? ldexp((double)m, 1 - 7 - 3) : ldexp((double)(8 + m), e - 7 - 3);
  return s ? -mag : mag;
}

/* An E5M2 code as a double.  Fields: s = bit 7, e = bits 6..2, m = bits 1..0.
 *   e == 31            : +-Inf when m == 0, NaN otherwise
 *   e == 0             : (-1)^s * (m / 4) * 2^(1 - 15)      (zero and subnormals)
 *   otherwise          : (-1)^s * (1 + m / 4) * 2^(e - 15) */
double oracle_e5m2_to_double(uint8_t code) {
  const int s = code >> 7, e = (code >> 2) & 31, m = code & 3;
  if (e == 31) return m ? NAN : (s ? -INFINITY : INFINITY);
  const double mag = (e == 0) ? ldexp((double)m, 1 - 15 - 2) : ldexp((double)(4 + m), e - 15 - 2);
  return s ? -mag : mag;
}

/* The kind of operand `side` (0 = A, 1 = B) in `mode`. */
static int operand_kind(int mode, int side) {
  switch (mode) {
    case ORACLE_MODE_TF32: return KIND_TF32;
    case ORACLE_MODE_BF16: return KIND_BF16;
    case ORACLE_MODE_FP8_E4M3: return KIND_E4M3;
    case ORACLE_MODE_FP8_E5M2: return KIND_E5M2;
    case ORACLE_MODE_FP8_E4M3_E5M2: return side == 0 ? KIND_E4M3 : KIND_E5M2;
    case ORACLE_MODE_FP8_E5M2_E4M3: return side == 0 ? KIND_E5M2 : KIND_E4M3;
    default: return KIND_FP32;
  }
}

static double operand(int kind, int tf32_rule, const void* base, int64_t idx) {
  if (kind == KIND_BF16) return oracle_bf16_to_double(((const uint16_t*)base)[idx]);
  if (kind == KIND_E4M3) return oracle_e4m3_to_double(((const uint8_t*)base)[idx]);
  if (kind == KIND_E5M2) return oracle_e5m2_to_double(((const uint8_t*)base)[idx]);
  float v = ((const float*)base)[idx];
  if (kind == KIND_TF32)
    v = (tf32_rule == ORACLE_TF32_NEAREST_AWAY) ? oracle_tf32_nearest_away(v) : oracle_tf32_truncate(v);
  return (double)v;
}

/* Elementwise TF32 reduction of an array (used by the tests to pin r()). */
void oracle_tf32_array(int tf32_rule, const float* in, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i)
    out[i] = (tf32_rule == ORACLE_TF32_NEAREST_AWAY) ? oracle_tf32_nearest_away(in[i]) : oracle_tf32_truncate(in[i]);
}

/* Elementwise exact widening of bfloat16 bit patterns (used by the tests). */
void oracle_bf16_array(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(in[i]);
}

/* Elementwise exact decoding of E4M3 / E5M2 codes (used by the tests). */
void oracle_e4m3_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_double(in[i]);
}

void oracle_e5m2_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e5m2_to_double(in[i]);
}

/* Returns 0 on success, a negative number for an argument it cannot take. */
int oracle_gemm(int mode, int tf32_rule, int transA, int transB,
                int64_t M, int64_t N, int64_t K, double alpha,
                const void* A, int64_t lda, const void* B, int64_t ldb,
                double beta, const float* Cin, int64_t ldc,
                int64_t row0, int64_t row1, double* Cref, double* D, int64_t ldr) {
  if (mode < ORACLE_MODE_FP32 || mode > ORACLE_MODE_FP8_E5M2_E4M3) return -1;
  const int kind_a = operand_kind(mode, 0), kind_b = operand_kind(mode, 1);
  if (M < 0 || N < 0 || K < 0) return -2;
  if (row0 < 0 || row1 < row0 || row1 > M) return -3;
  if (ldr < N) return -4;
  const int read_ab = (K > 0 && alpha != 0.0);
  const int read_c = (beta != 0.0);

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = row0; i < row1; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double acc = 0.0, mag = 0.0;
      if (read_ab) {
        for (int64_t k = 0; k < K; ++k) {
          int64_t ia = transA ? k * lda + i : i * lda + k;
          int64_t ib = transB ? j * ldb + k : k * ldb + j;
          double p = operand(kind_a, tf32_rule, A, ia) * operand(kind_b, tf32_rule, B, ib);
          acc += p;
          mag += fabs(p);
        }
      }
      double c = alpha * acc;
      if (read_c) c += beta * (double)Cin[i * ldc + j];
      Cref[(i - row0) * ldr + j] = c;
      if (D) D[(i - row0) * ldr + j] = mag;
    }
  }
  return 0;
}

/*
 * The fused epilogue of gemm_run_epilogue, in double, applied to the exact
 * pre-activation Y[i][j] = alpha * sum_k opA*opB + beta * Cin (as returned by
 * oracle_gemm) for a block of rows:
 *
 *   act 0:  out = Y + bias[j]
 *   act 1:  out = GELU(Y + bias[j])
 *   act 2:  out = Y * GELU'(Z[i][j])
 *
 * "bare-metal-bard" (second paragraph) trains a GPT whose GELU kernel is
 * written by hand; it does not say which GELU.  The reading taken is the
 * function's definition, GELU(x) = x * Phi(x) with Phi the standard normal
 * distribution function, Phi(x) = (1 + erf(x / sqrt 2)) / 2, and its
 * derivative GELU'(x) = Phi(x) + x * phi(x), phi(x) = exp(-x^2 / 2) / sqrt(2 pi).
 * bias may be NULL (no bias); Z is read only for act 2.
 */
double oracle_gelu(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }

double oracle_dgelu(double x) {
  const double Phi = 0.5 * (1.0 + erf(x / sqrt(2.0)));
  const double phi = exp(-0.5 * x * x) / sqrt(2.0 * 3.14159265358979323846);
  return Phi + x * phi;
}

int oracle_epilogue(int act, int64_t rows, int64_t N, const double* y, int64_t ldy, const float* bias,
                    const float* z, int64_t ldz, double* out, int64_t ldo) {
  if (act < 0 || act > 2 || rows < 0 || N < 0) return 1;
  if (act == 2 && (z == 0 || bias != 0)) return 2;
  for (int64_t i = 0; i < rows; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      const double v = y[i * ldy + j];
      double r;
      if (act == 2) {
        r = v * oracle_dgelu((double)z[i * ldz + j]);
      } else {
        const double pre = v + (bias ? (double)bias[j] : 0.0);
        r = (act == 1) ? oracle_gelu(pre) : pre;
      }
      out[i * ldo + j] = r;
    }
  }
  return 0;
}

/*
 * Block-scaled products: the MX formats and NVFP4.  "Low-Precision Kernels:
 * INT4, INT8 and FP8 Matmuls, Measured" (its summary) names FP8, MX and
 * NVFP4 scales without defining them; the reading taken is the OCP
 * Microscaling (MX) specification and NVIDIA's NVFP4 layout:
 *
 *   every run of `bs` consecutive K elements of a row of A (and of a row of
 *   the N x K-stored B) shares one scale; an element's value is its scale
 *   times its own decoded value, so
 *
 *   Cref[i][j] = alpha * sum_k (SA[i][k / bs] * a[i][k]) * (SB[j][k / bs] * b[j][k])
 *                + beta * Cin[i][j]
 *   D[i][j]    =         sum_k |SA[i][k / bs] * a[i][k]| * |SB[j][k / bs] * b[j][k]|
 *
 *   MXFP8: elements E4M3 or E5M2, bs = 32, scales E8M0.
 *   MXFP4: elements E2M1, bs = 32, scales E8M0.
 *   NVFP4: elements E2M1, bs = 16, scales UE4M3 (and a per-tensor factor,
 *          which is the caller's alpha).
 *
 * Element formats: 0 = E4M3, 1 = E5M2, 2 = E2M1.  E2M1 elements are packed
 * two to a byte, element 2t in the low four bits of byte t.
 * Scale formats: 0 = E8M0, 1 = UE4M3.
 * Both operands are K-major: A is M x K (row pitch lda bytes), B is N x K
 * (ldb bytes); SA is M x ceil(K / bs) bytes (pitch ldsa), SB N x ceil(K / bs)
 * (ldsb).  The last block of a row may be partial.
 */

/* E2M1: s = bit 3, e = bits 2..1 (bias 1), m = bit 0; no infinities or NaNs.
 *   e == 0 : (-1)^s * (m / 2) * 2^(1 - 1)
 *   else   : (-1)^s * (1 + m / 2) * 2^(e - 1)
 * giving the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double oracle_e2m1_to_double(uint8_t code) {
  const int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = (e == 0) ? ldexp((double)m, -1) : ldexp((double)(2 + m), e - 2);
  return s ? -mag : mag;
}

/* E8M0: an exponent alone, 2^(e - 127); 0xFF is NaN. */
double oracle_e8m0_to_double(uint8_t code) {
  if (code == 0xFF) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* UE4M3: the E4M3 magnitude of the code with its sign bit ignored. */
double oracle_ue4m3_to_double(uint8_t code) { return oracle_e4m3_to_double((uint8_t)(code & 0x7F)); }

static double block_element(int fmt, const uint8_t* row, int64_t k) {
  if (fmt == 2) {
    const uint8_t byte = row[k >> 1];
    return oracle_e2m1_to_double((uint8_t)((k & 1) ? (byte >> 4) : (byte & 15)));
  }
  return fmt == 1 ? oracle_e5m2_to_double(row[k]) : oracle_e4m3_to_double(row[k]);
}

static double block_scale(int scale_fmt, uint8_t code) {
  return scale_fmt == 1 ? oracle_ue4m3_to_double(code) : oracle_e8m0_to_double(code);
}

void oracle_e2m1_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e2m1_to_double(in[i]);
}

void oracle_e8m0_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e8m0_to_double(in[i]);
}

void oracle_ue4m3_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_ue4m3_to_double(in[i]);
}

/* Returns 0 on success, a negative number for an argument it cannot take. */
int oracle_gemm_block_scaled(int fmt_a, int fmt_b, int scale_fmt, int64_t bs, int64_t M, int64_t N, int64_t K,
                             double alpha, const uint8_t* A, int64_t lda, const uint8_t* SA, int64_t ldsa,
                             const uint8_t* B, int64_t ldb, const uint8_t* SB, int64_t ldsb, double beta,
                             const float* Cin, int64_t ldc, int64_t row0, int64_t row1, double* Cref, double* D,
                             int64_t ldr) {
  if (fmt_a < 0 || fmt_a > 2 || fmt_b < 0 || fmt_b > 2 || scale_fmt < 0 || scale_fmt > 1) return -1;
  if (M < 0 || N < 0 || K < 0 || bs < 1) return -2;
  if (row0 < 0 || row1 < row0 || row1 > M) return -3;
  if (ldr < N) return -4;
  const int read_ab = (K > 0 && alpha != 0.0);
  const int read_c = (beta != 0.0);

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = row0; i < row1; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      double acc = 0.0, mag = 0.0;
      if (read_ab) {
        for (int64_t k = 0; k < K; ++k) {
          const double a = block_scale(scale_fmt, SA[i * ldsa + k / bs]) * block_element(fmt_a, A + i * lda, k);
          const double b = block_scale(scale_fmt, SB[j * ldsb + k / bs]) * block_element(fmt_b, B + j * ldb, k);
          acc += a * b;
          mag += fabs(a * b);
        }
      }
      double c = alpha * acc;
      if (read_c) c += beta * (double)Cin[i * ldc + j];
      Cref[(i - row0) * ldr + j] = c;
      if (D) D[(i - row0) * ldr + j] = mag;
    }
  }
  return 0;
}

/*
 * Scaled dot-product attention, forward: the other GEMM-shaped operation of
 * the GPT step.  "bare-metal-bard" (third paragraph) reports a fused
 * attention kernel -- the score matrix never leaves the chip -- for the
 * model's causal self-attention; the operation it computes is the plain
 * definition, for every problem p (a batch element and head) and query row i:
 *
 *     s_j    = scale * sum_d q[i][d] * k[j][d]     for every key j that i sees
 *              (j <= i when causal, every j < T otherwise)
 *     p_j    = exp(s_j - max_j s_j),   l = sum_j p_j
 *     O[i][d] = (sum_j p_j * v[j][d]) / l
 *     W[i][d] = (sum_j p_j * |v[j][d]|) / l       (the error scale)
 *
 * Q, K and V are bfloat16 bit patterns of shape [problems][T][Dh], widened
 * exactly; sums run over d, then j, ascending, in IEEE double.  Problems
 * p0 .. p1-1 are produced, problem p's row i at O[((p - p0) * T + i) * Dh].
 */
int oracle_attention(int64_t problems, int64_t T, int64_t Dh, int causal, double scale, const uint16_t* Q,
                     const uint16_t* K, const uint16_t* V, int64_t p0, int64_t p1, double* O, double* W) {
  if (problems < 0 || T < 0 || Dh < 1 || p0 < 0 || p1 < p0 || p1 > problems) return 1;
  if (T > 0 && (Q == NULL || K == NULL || V == NULL || O == NULL || W == NULL)) return 2;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (int64_t p = p0; p < p1; ++p) {
    for (int64_t i = 0; i < T; ++i) {
      const uint16_t* q = Q + (p * T + i) * Dh;
      const int64_t keys = causal ? i + 1 : T;
      double smax = -INFINITY;
      for (int64_t j = 0; j < keys; ++j) {
        const uint16_t* k = K + (p * T + j) * Dh;
        double dot = 0.0;
        for (int64_t d = 0; d < Dh; ++d) dot += oracle_bf16_to_double(q[d]) * oracle_bf16_to_double(k[d]);
        const double s = scale * dot;
        if (s > smax) smax = s;
      }
      double l = 0.0;
      double* o = O + ((p - p0) * T + i) * Dh;
      double* w = W + ((p - p0) * T + i) * Dh;
      for (int64_t d = 0; d < Dh; ++d) o[d] = w[d] = 0.0;
      for (int64_t j = 0; j < keys; ++j) {
        const uint16_t* k = K + (p * T + j) * Dh;
        const uint16_t* v = V + (p * T + j) * Dh;
        double dot = 0.0;
        for (int64_t d = 0; d < Dh; ++d) dot += oracle_bf16_to_double(q[d]) * oracle_bf16_to_double(k[d]);
        const double pj = exp(scale * dot - smax);
        l += pj;
        for (int64_t d = 0; d < Dh; ++d) {
          const double vd = oracle_bf16_to_double(v[d]);
          o[d] += pj * vd;
          w[d] += pj * fabs(vd);
        }
      }
      for (int64_t d = 0; d < Dh; ++d) {
        o[d] /= l;
        w[d] /= l;
      }
    }
  }
  return 0;
}
