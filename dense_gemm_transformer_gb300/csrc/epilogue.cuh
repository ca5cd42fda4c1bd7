// epilogue.cuh -- the elementwise work gemm_run_epilogue fuses into every
// kernel's final store: a per-column bias, GELU, or the product with GELU'
// of a kept pre-activation (the backward pass through a GELU).
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

// v = alpha * (the product) + beta * C at element (row, col) of the caller's
// C; returns what is stored there.
__device__ __forceinline__ float apply_epilogue(const EpiParams& e, float v, int64_t row, int64_t col) {
  if (e.act == kActDGelu) return v * dgelu_f(__ldg(e.aux + row * e.ld_aux + col));
  if (e.bias != nullptr) v += __ldg(e.bias + col);
  if (e.act == kActGelu) v = gelu_f(v);
  return v;
}

// Whether the epilogue does anything beyond alpha/beta.
__device__ __forceinline__ bool epilogue_active(const EpiParams& e) { return e.act != kActNone || e.bias != nullptr; }

}  // namespace dgt
