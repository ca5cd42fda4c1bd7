// calib.cu -- the FP32 FMA roof of this part, measured rather than derived.
//
// The FP32 mode's kernel is bound by the CUDA cores' fused multiply-adds, so
// its roofline fraction needs the rate those cores actually sustain here
// (clock under load included).  This kernel does nothing but independent
// FMA chains in registers: every thread runs 16 chains (scalar fma.rn.f32,
// or eight packed fma.rn.f32x2 pairs, the form the SIMT kernel issues) for
// `iters` steps and stores one sum so that nothing is optimised away.
// FLOPs per launch = grid x 256 threads x iters x 16 x 2.
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm.h"
#include "kernels.h"
#include "ptx.cuh"

namespace dgt {
namespace {

constexpr int kCalibThreads = 256;
constexpr int kChains = 16;

__device__ __forceinline__ uint64_t pack2f(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack2f(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

template <bool PACKED>
__global__ void __launch_bounds__(kCalibThreads) fma_peak_kernel(int64_t iters, float m, float c, float* out) {
  grid_dep_wait();
  grid_dep_launch();
  const float t = static_cast<float>(threadIdx.x) * 1e-3f;
  if constexpr (PACKED) {
    uint64_t acc[kChains / 2];
#pragma unroll
    for (int j = 0; j < kChains / 2; ++j) acc[j] = pack2f(t + j, t - j);
    const uint64_t mm = pack2f(m, m), cc = pack2f(c, c);
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
      for (int j = 0; j < kChains / 2; ++j) asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(acc[j]) : "l"(mm), "l"(cc));
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains / 2; ++j) {
      float lo, hi;
      unpack2f(acc[j], lo, hi);
      s += lo + hi;
    }
    out[blockIdx.x * kCalibThreads + threadIdx.x] = s;
  } else {
    float acc[kChains];
#pragma unroll
    for (int j = 0; j < kChains; ++j) acc[j] = t + j;
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
      for (int j = 0; j < kChains; ++j) asm volatile("fma.rn.f32 %0, %0, %1, %2;" : "+f"(acc[j]) : "f"(m), "f"(c));
    }
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kChains; ++j) s += acc[j];
    out[blockIdx.x * kCalibThreads + threadIdx.x] = s;
  }
}

}  // namespace
}  // namespace dgt

extern "C" gemm_status_t gemm_launch_fma_peak(int packed, int64_t grid, int64_t iters, float* out, void* stream) {
  if (grid < 1 || grid > (int64_t(1) << 20) || iters < 1 || out == nullptr || (packed != 0 && packed != 1))
    return GEMM_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0) return GEMM_ERR_MISALIGNED;
  const dim3 g(static_cast<unsigned>(grid)), b(dgt::kCalibThreads);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // m slightly below 1 and c small keep every chain finite for any iters
  const cudaError_t e = packed ? dgt::launch_pdl(dgt::fma_peak_kernel<true>, g, b, 0, s, iters, 0.9999999f, 1e-7f, out)
                               : dgt::launch_pdl(dgt::fma_peak_kernel<false>, g, b, 0, s, iters, 0.9999999f, 1e-7f, out);
  return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
