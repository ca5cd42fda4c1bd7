// tc_launch.cuh -- host-side launch of the tcgen05 kernel for one operand mode
// (included once by each of tc_tf32.cu and tc_bf16.cu so the two modes
// compile in parallel).
#pragma once

#include "tc_kernel.cuh"

namespace dgt {

template <int MODE, bool A_MN, bool B_MN, int BN, bool TRANS_C = false>
cudaError_t tc_launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const TcParams& p, int grid,
                          cudaStream_t s) {
  using Cfg = TcCfg<MODE, BN>;
  auto kern = tc_gemm_kernel<MODE, A_MN, B_MN, BN, TRANS_C>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, kTcThreads, Cfg::SMEM_BYTES, s>>>(ta, tb, tc, p);
  return cudaGetLastError();
}

// kind::tf32 takes K-major operands only (the planner transposes MN-major
// TF32 operands first), so only BF16 instantiates the MN-major forms.
template <int MODE, int BN>
cudaError_t tc_launch_bn(bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                         const TcParams& p, int grid, cudaStream_t s) {
  if (!a_mn && !b_mn) return tc_launch_one<MODE, false, false, BN>(ta, tb, tc, p, grid, s);
  if constexpr (MODE == 1) return cudaErrorInvalidValue;
  if (!a_mn && b_mn) return tc_launch_one<MODE, false, true, BN>(ta, tb, tc, p, grid, s);
  if (a_mn && !b_mn) return tc_launch_one<MODE, true, false, BN>(ta, tb, tc, p, grid, s);
  return tc_launch_one<MODE, true, true, BN>(ta, tb, tc, p, grid, s);
}

// tile_n == 16 is the swapped small-M form: the weights are the 128-row
// operand (K-major or MN-major), the activations a K-major 16-row operand,
// and C is written transposed.
template <int MODE>
cudaError_t tc_launch_mode(int tile_n, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t s) {
  if (tile_n == 256) return tc_launch_bn<MODE, 256>(a_mn, b_mn, ta, tb, tc, p, grid, s);
  if (tile_n == 128) return tc_launch_bn<MODE, 128>(a_mn, b_mn, ta, tb, tc, p, grid, s);
  if (tile_n == 16 && !b_mn) {
    if (!a_mn) return tc_launch_one<MODE, false, false, 16, true>(ta, tb, tc, p, grid, s);
    if constexpr (MODE == 2) return tc_launch_one<MODE, true, false, 16, true>(ta, tb, tc, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

// Defined in tc_tf32.cu (MODE 1) and tc_bf16.cu (MODE 2).
cudaError_t tc_launch_tf32(int tile_n, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t s);
cudaError_t tc_launch_bf16(int tile_n, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t s);

}  // namespace dgt
