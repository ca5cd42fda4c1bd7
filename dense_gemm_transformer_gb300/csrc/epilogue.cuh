// epilogue.cuh -- the elementwise work of gemm_run_epilogue: a per-column
// bias, GELU, or the product with GELU' of a kept pre-activation (the
// backward pass through a GELU).  It runs where a call already touches every
// element of C after the GEMM kernels (the split-K reduction, the beta-only
// update), or else in one pass over C: computed inside the GEMM kernels'
// epilogues it measured slower than that pass on the GPT products (K = 384:
// the erf evaluations stall the tile pipeline more than the pass costs in
// HBM traffic), and it took registers from kernels that sit at their limit.
//
// "bare-metal-bard" (second paragraph) trains a GPT with hand-written
// matmul, layernorm and GELU kernels; the page does not say which GELU.  The
// reading taken here is the function's definition, GELU(x) = x * Phi(x) with
// Phi(x) = (1 + erf(x / sqrt 2)) / 2, and GELU'(x) = Phi(x) + x * phi(x),
// phi(x) = exp(-x^2 / 2) / sqrt(2 pi); erff and expf are CUDA's.
#pragma once

#include "kernels.h"

namespace dgt {

__device__ __forceinline__ float gelu_f(float x) {
  constexpr float kInvSqrt2 = 0.70710678118654752f;
  return 0.5f * x * (1.f + erff(x * kInvSqrt2));
}

__device__ __forceinline__ float dgelu_f(float x) {
  constexpr float kInvSqrt2 = 0.70710678118654752f;
  constexpr float kInvSqrt2Pi = 0.39894228040143268f;
  const float Phi = 0.5f * (1.f + erff(x * kInvSqrt2));
  return fmaf(x, kInvSqrt2Pi * expf(-0.5f * x * x), Phi);
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

// Both steps for one element.
__device__ __forceinline__ float apply_epilogue(const EpiParams& e, float v, int64_t row, int64_t col) {
  return epilogue_finish(e, v, epilogue_fetch(e, row, col));
}

// Whether the epilogue does anything beyond alpha/beta.
__device__ __forceinline__ bool epilogue_active(const EpiParams& e) { return e.act != kActNone || e.bias != nullptr; }

}  // namespace dgt
