// epilogue.cuh -- the elementwise work of gemm_run_epilogue: a per-column
// bias, GELU, or the product with GELU' of a kept pre-activation (the
// backward pass through a GELU).  It is applied once per element, at the
// final store: in the tcgen05 kernel's epilogue warps when that kernel
// writes C itself (TF32 and BF16 with a K-major A, whole tiles or the tail
// slices with their reduction), in the split-K reduction when a call ends
// with one, in the beta-only update for K = 0, and otherwise in one pass over
// C after the GEMM kernels (the SIMT family, A moved through TMEM, the
// small-M kernels).
//
// "bare-metal-bard" (second paragraph) trains a GPT with hand-written
// matmul, layernorm and GELU kernels; the page does not say which GELU.  The
// reading taken here is the function's definition, GELU(x) = x * Phi(x) with
// Phi the standard normal distribution function, and GELU'(x) = Phi(x) +
// x * phi(x), phi(x) = exp(-x^2 / 2) / sqrt(2 pi).
//
// Phi comes from the complementary error function, Phi(x) = erfc(-x / sqrt 2)
// / 2, evaluated by the rational approximation of Abramowitz and Stegun,
// Handbook of Mathematical Functions, formula 7.1.26 (C. Hastings' fit):
// for z >= 0, erfc(z) = (a1 t + a2 t^2 + a3 t^3 + a4 t^4 + a5 t^5) e^(-z^2) +
// eps, t = 1 / (1 + p z), |eps| <= 1.5e-7.  Taking z = |x| / sqrt 2 and
// Phi(x) = 1 - erfc(z) / 2 for x >= 0, erfc(z) / 2 for x < 0 avoids the
// cancellation of 1 + erf(x) in the negative tail, and e^(-z^2) =
// e^(-x^2 / 2) is phi's exponential too, so GELU' costs no second one.
// The reciprocal and the power of two are the hardware's approximate
// instructions (rcp.approx, ex2.approx: a few units of 2^-23 relative), so
// |Phi - Phi_exact| stays near 1e-7.
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace dgt {

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float exp2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Phi(x) and e^(-x^2 / 2) together (7.1.26 above).  The constants are
// folded: t = 1 / (1 + (p / sqrt 2) |x|), the coefficients carry the 1/2 of
// erfc / 2, and the exponent's scale log2(e) / 2 is one multiply.
__device__ __forceinline__ void normal_cdf_exp(float x, float& Phi, float& e) {
  constexpr float kPs = 0.23164188f;  // 0.3275911 / sqrt(2)
  constexpr float kH1 = 0.127414796f, kH2 = -0.142248368f, kH3 = 0.7107068705f, kH4 = -0.7265760135f,
                  kH5 = 0.5307027145f;  // a1 .. a5 of 7.1.26, halved
  constexpr float kNegHalfLog2e = -0.72134752044448170f;  // -log2(e) / 2
  const float t = rcp_approx(fmaf(kPs, fabsf(x), 1.f));
  const float half_poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, kH5, kH4), kH3), kH2), kH1);
  e = exp2_approx((x * x) * kNegHalfLog2e);  // e^(-x^2 / 2) = e^(-z^2), z = |x| / sqrt 2
  const float half_erfc = half_poly * e;
  Phi = x >= 0.f ? 1.f - half_erfc : half_erfc;
}

__device__ __forceinline__ void normal_cdf_pdf(float x, float& Phi, float& phi) {
  constexpr float kInvSqrt2Pi = 0.39894228040143268f;
  float e;
  normal_cdf_exp(x, Phi, e);
  phi = kInvSqrt2Pi * e;
}

__device__ __forceinline__ float gelu_f(float x) {
  float Phi, e;
  normal_cdf_exp(x, Phi, e);
  return x * Phi;
}

__device__ __forceinline__ float dgelu_f(float x) {
  float Phi, phi;
  normal_cdf_pdf(x, Phi, phi);
  return fmaf(x, phi, Phi);
}

// The same functions on a pair of elements (a packed fp32 pair of ptx.cuh):
// the multiplies and adds of the pair are packed instructions, the
// reciprocal and the power of two stay per element.  normal_cdf_exp_x2 and
// dgelu_x2 take the steps of the scalar forms above in the same order, so
// each element comes out exactly as the scalar function gives it.
__device__ __forceinline__ uint64_t f2_splat(float c) { return f2_pack(c, c); }

__device__ __forceinline__ void normal_cdf_exp_x2(uint64_t x, uint64_t& Phi, uint64_t& e) {
  constexpr float kPs = 0.23164188f;
  constexpr float kH1 = 0.127414796f, kH2 = -0.142248368f, kH3 = 0.7107068705f, kH4 = -0.7265760135f,
                  kH5 = 0.5307027145f;
  constexpr float kNegHalfLog2e = -0.72134752044448170f;
  float x0, x1;
  f2_unpack(x, x0, x1);
  // (scalar: the absolute value folds into the multiply-add's operand)
  const uint64_t t = f2_pack(rcp_approx(fmaf(kPs, fabsf(x0), 1.f)), rcp_approx(fmaf(kPs, fabsf(x1), 1.f)));
  uint64_t q = f2_fma(t, f2_splat(kH5), f2_splat(kH4));
  q = f2_fma(t, q, f2_splat(kH3));
  q = f2_fma(t, q, f2_splat(kH2));
  q = f2_fma(t, q, f2_splat(kH1));
  const uint64_t half_poly = f2_mul(t, q);
  float a0, a1;
  f2_unpack(f2_mul(f2_mul(x, x), f2_splat(kNegHalfLog2e)), a0, a1);
  e = f2_pack(exp2_approx(a0), exp2_approx(a1));
  const uint64_t half_erfc = f2_mul(half_poly, e);
  float h0, h1, o0, o1;
  f2_unpack(half_erfc, h0, h1);
  f2_unpack(f2_fma(half_erfc, f2_splat(-1.f), f2_splat(1.f)), o0, o1);  // 1 - half_erfc, one rounding
  Phi = f2_pack(x0 >= 0.f ? o0 : h0, x1 >= 0.f ? o1 : h1);
}

// GELU of a pair, in the form GELU(x) = max(x, 0) - |x| erfc(|x| / sqrt 2) / 2
// (for x >= 0 it is x - x (1 - Phi(x)), for x < 0 it is x Phi(x)): the
// erfc term comes out of 7.1.26 with its coefficients negated, and one
// multiply-add with max(x, 0) finishes the element, so that no per-element
// sign test is needed; an element rounds once at the end, and in the
// negative tail the result keeps its relative accuracy.
__device__ __forceinline__ uint64_t gelu_x2(uint64_t x) {
  constexpr float kPs = 0.23164188f;
  constexpr float kH1 = 0.127414796f, kH2 = -0.142248368f, kH3 = 0.7107068705f, kH4 = -0.7265760135f,
                  kH5 = 0.5307027145f;
  constexpr float kNegHalfLog2e = -0.72134752044448170f;
  float x0, x1;
  f2_unpack(x, x0, x1);
  const uint64_t ax = f2_pack(fabsf(x0), fabsf(x1));
  float d0, d1;
  f2_unpack(f2_fma(f2_splat(kPs), ax, f2_splat(1.f)), d0, d1);
  const uint64_t t = f2_pack(rcp_approx(d0), rcp_approx(d1));
  uint64_t q = f2_fma(t, f2_splat(-kH5), f2_splat(-kH4));
  q = f2_fma(t, q, f2_splat(-kH3));
  q = f2_fma(t, q, f2_splat(-kH2));
  q = f2_fma(t, q, f2_splat(-kH1));
  const uint64_t neg_half_poly = f2_mul(t, q);
  float a0, a1;
  f2_unpack(f2_mul(f2_mul(x, x), f2_splat(kNegHalfLog2e)), a0, a1);
  const uint64_t e = f2_pack(exp2_approx(a0), exp2_approx(a1));
  return f2_fma(ax, f2_mul(neg_half_poly, e), f2_pack(fmaxf(x0, 0.f), fmaxf(x1, 0.f)));
}

__device__ __forceinline__ uint64_t dgelu_x2(uint64_t x) {
  constexpr float kInvSqrt2Pi = 0.39894228040143268f;
  uint64_t Phi, e;
  normal_cdf_exp_x2(x, Phi, e);
  return f2_fma(x, f2_mul(f2_splat(kInvSqrt2Pi), e), Phi);
}

// The epilogue's input for element (row, col) of the caller's C: Z there
// for DGELU, else the column's bias (0 without one).
__device__ __forceinline__ float epilogue_fetch(const EpiParams& e, int64_t row, int64_t col) {
  if (e.act == kActDGelu) return __ldg(e.aux + row * e.ld_aux + col);
  return e.bias != nullptr ? __ldg(e.bias + col) : 0.f;
}

// The same for columns col .. col + 3 of one row (columns from n on read
// nothing): one 16-byte load where the address allows.
__device__ __forceinline__ float4 epilogue_fetch4(const EpiParams& e, int64_t row, int64_t col, int64_t n) {
  const float* src = (e.act == kActDGelu) ? e.aux + row * e.ld_aux + col : e.bias + col;
  if (e.act != kActDGelu && e.bias == nullptr) return make_float4(0.f, 0.f, 0.f, 0.f);
  if (col + 3 < n && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) return __ldg(reinterpret_cast<const float4*>(src));
  float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
  if (col < n) r.x = __ldg(src);
  if (col + 1 < n) r.y = __ldg(src + 1);
  if (col + 2 < n) r.z = __ldg(src + 2);
  if (col + 3 < n) r.w = __ldg(src + 3);
  return r;
}

// v = alpha * (the product) + beta * C at an element whose fetched input is
// x; returns what is stored there.
__device__ __forceinline__ float epilogue_finish(const EpiParams& e, float v, float x) {
  if (e.act == kActDGelu) return v * dgelu_f(x);
  v += x;
  return e.act == kActGelu ? gelu_f(v) : v;
}

// epilogue_finish with the activation fixed at compile time (ACT: kActNone,
// kActGelu, kActDGelu), for loops that dispatch on it once.
template <int ACT>
__device__ __forceinline__ float epilogue_finish_t(float v, float x) {
  if constexpr (ACT == kActDGelu) return v * dgelu_f(x);
  v += x;
  if constexpr (ACT == kActGelu) return gelu_f(v);
  return v;
}

// Both steps for one element.
__device__ __forceinline__ float apply_epilogue(const EpiParams& e, float v, int64_t row, int64_t col) {
  return epilogue_finish(e, v, epilogue_fetch(e, row, col));
}

// Whether the epilogue does anything beyond alpha/beta.
__device__ __forceinline__ bool epilogue_active(const EpiParams& e) { return e.act != kActNone || e.bias != nullptr; }

}  // namespace dgt
