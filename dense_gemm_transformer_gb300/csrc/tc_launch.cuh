// tc_launch.cuh -- host-side launch of the tcgen05 kernel for one operand mode
// (included once by each of tc_tf32.cu and tc_bf16.cu so the two modes
// compile in parallel).
#pragma once

#include "tc_kernel.cuh"

namespace dgt {

template <int MODE, bool A_MN, bool B_MN, int BN, bool TRANS_C = false, bool PAIR = false>
cudaError_t tc_launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const TcParams& p,
                          int grid, cudaStream_t s) {
  using Cfg = TcCfg<MODE, BN>;
  auto kern = tc_gemm_kernel<MODE, A_MN, B_MN, BN, TRANS_C, PAIR>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if constexpr (PAIR) {
    // Two-CTA clusters along x: CTAs 2c and 2c+1 form pair c.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, p);
  } else {
    kern<<<grid, kTcThreads, Cfg::SMEM_BYTES, s>>>(ta, tb, tc, p);
    return cudaGetLastError();
  }
}

// kind::tf32 takes K-major operands only (the planner transposes MN-major
// TF32 operands first), so only BF16 instantiates the MN-major forms.
template <int MODE, int BN, bool PAIR>
cudaError_t tc_launch_bn(bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                         const TcParams& p, int grid, cudaStream_t s) {
  if (!a_mn && !b_mn) return tc_launch_one<MODE, false, false, BN, false, PAIR>(ta, tb, tc, p, grid, s);
  if constexpr (MODE == 1) {
    return cudaErrorInvalidValue;
  } else {
    if (!a_mn && b_mn) return tc_launch_one<MODE, false, true, BN, false, PAIR>(ta, tb, tc, p, grid, s);
    if (a_mn && !b_mn) return tc_launch_one<MODE, true, false, BN, false, PAIR>(ta, tb, tc, p, grid, s);
    return tc_launch_one<MODE, true, true, BN, false, PAIR>(ta, tb, tc, p, grid, s);
  }
}

// tile_n == 16 is the swapped small-M form: the weights are the 128-row
// operand (K-major or MN-major), the activations a K-major 16-row operand,
// and C is written transposed.  `pair` selects the two-CTA form (tile_n 256).
template <int MODE>
cudaError_t tc_launch_mode(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t s) {
  if (tile_n == 256 && pair) return tc_launch_bn<MODE, 256, true>(a_mn, b_mn, ta, tb, tc, p, grid, s);
  if (tile_n == 256) return tc_launch_bn<MODE, 256, false>(a_mn, b_mn, ta, tb, tc, p, grid, s);
  if (tile_n == 128) return tc_launch_bn<MODE, 128, false>(a_mn, b_mn, ta, tb, tc, p, grid, s);
  if (tile_n == 16 && !b_mn) {
    if (!a_mn) return tc_launch_one<MODE, false, false, 16, true>(ta, tb, tc, p, grid, s);
    if constexpr (MODE == 2) return tc_launch_one<MODE, true, false, 16, true>(ta, tb, tc, p, grid, s);
  }
  return cudaErrorInvalidValue;
}

// Defined in tc_tf32.cu (MODE 1) and tc_bf16.cu (MODE 2).
cudaError_t tc_launch_tf32(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t s);
cudaError_t tc_launch_bf16(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const TcParams& p, int grid, cudaStream_t s);

}  // namespace dgt
