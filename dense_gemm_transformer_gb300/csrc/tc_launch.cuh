// tc_launch.cuh -- host-side launch of the tcgen05 kernel for one operand mode
// (included by each of tc_tf32.cu, tc_bf16.cu, tc_bf16_mid.cu, tc_fp8.cu and
// tc_fp8_mid.cu so that the modes compile in parallel).
#pragma once

#include "tc_kernel.cuh"

namespace dgt {

template <int MODE, bool A_MN, bool B_MN, int BN, bool TRANS_C = false, bool PAIR = false, bool EPI = false>
cudaError_t tc_launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                          const TcParams& p, int grid, cudaStream_t s) {
  using Cfg = TcCfg<MODE, BN, PAIR, EPI ? kTcEpiWarpsEpi : kTcEpiWarps>;
  auto kern = tc_gemm_kernel<MODE, A_MN, B_MN, BN, TRANS_C, PAIR, EPI>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  last_main_launch() = LaunchShape{dim3(static_cast<unsigned>(grid)), dim3(Cfg::THREADS),
                                   static_cast<size_t>(Cfg::SMEM_BYTES), PAIR ? 2 : 1, true};
  if constexpr (PAIR) {
    // Two-CTA clusters along x: CTAs 2c and 2c+1 form pair c.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tw, p);
  } else {
    return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(Cfg::THREADS), Cfg::SMEM_BYTES, s, ta, tb, tc, tw,
                      p);
  }
}

// Which operand layouts a tile width can take.  kind::tf32 reads K-major
// operands only from shared memory: the planner transposes an MN-major TF32
// B first, and an MN-major TF32 A too unless the 128-column, one-CTA kernel
// takes it through TMEM; an MN-major B is loaded in 128-byte column chunks,
// so its tile width must be a whole number of chunks, and an even number
// when each CTA of a pair loads one half.
template <int MODE, int BN, bool PAIR>
constexpr bool tc_mn_b_ok() {
  return MODE == 2 && BN % TcCfg<MODE, BN>::CH == 0 && (!PAIR || (BN / TcCfg<MODE, BN>::CH) % 2 == 0);
}

template <int MODE, int BN, bool PAIR, bool EPI = false>
cudaError_t tc_launch_bn(bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                         const CUtensorMap& tw, const TcParams& p, int grid, cudaStream_t s) {
  if (!a_mn && !b_mn) return tc_launch_one<MODE, false, false, BN, false, PAIR, EPI>(ta, tb, tc, tw, p, grid, s);
  if constexpr (EPI) {
    // the fused epilogue is built for a K-major A (the forward and dX
    // products that carry it), and in BF16 for an N-contiguous B too
    if constexpr (MODE == 2 && tc_mn_b_ok<MODE, BN, PAIR>()) {
      if (!a_mn) return tc_launch_one<MODE, false, true, BN, false, PAIR, true>(ta, tb, tc, tw, p, grid, s);
    }
    return cudaErrorNotSupported;
  } else {
    if constexpr (MODE == 1 && BN == 128 && !PAIR) {
      // an MN-major TF32 A goes to the MMA through TMEM
      if (a_mn && !b_mn) return tc_launch_one<1, true, false, 128>(ta, tb, tc, tw, p, grid, s);
    }
    if constexpr (MODE == 2) {
      if (a_mn && !b_mn) return tc_launch_one<MODE, true, false, BN, false, PAIR>(ta, tb, tc, tw, p, grid, s);
      if constexpr (tc_mn_b_ok<MODE, BN, PAIR>()) {
        if (!a_mn) return tc_launch_one<MODE, false, true, BN, false, PAIR>(ta, tb, tc, tw, p, grid, s);
        return tc_launch_one<MODE, true, true, BN, false, PAIR>(ta, tb, tc, tw, p, grid, s);
      }
    }
    return cudaErrorInvalidValue;
  }
}

// The 128- and 256-column tiles and the swapped small-M form (tile_n 16:
// the weights are the 128-row operand, K-major or MN-major, the activations
// a K-major 16-row operand, and C is written transposed).  `pair`: CTA
// pairs issuing one MMA of 256 rows (tcgen05 cta_group::2; 256 columns).
template <int MODE, bool EPI = false>
cudaError_t tc_launch_mode(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const CUtensorMap& tw, const TcParams& p, int grid,
                           cudaStream_t s) {
  if (tile_n == 256 && pair) return tc_launch_bn<MODE, 256, true, EPI>(a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  if (tile_n == 256) return tc_launch_bn<MODE, 256, false, EPI>(a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  if (tile_n == 128 && !pair) return tc_launch_bn<MODE, 128, false, EPI>(a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  if constexpr (EPI) {
    return cudaErrorNotSupported;
  } else {
    if (tile_n == 16 && !b_mn && !pair) {
      if (!a_mn) return tc_launch_one<MODE, false, false, 16, true>(ta, tb, tc, tw, p, grid, s);
      if constexpr (MODE == 2) return tc_launch_one<MODE, true, false, 16, true>(ta, tb, tc, tw, p, grid, s);
    }
    return cudaErrorInvalidValue;
  }
}

// The 192- and 224-column tiles, which let the planner fill whole waves
// where 256 would leave the last one mostly idle (4096 columns: 19 tiles of
// 224 instead of 16 of 256), alone or as CTA pairs issuing one MMA of 256
// rows (each CTA stages 96 or 112 rows of a K-major B).
template <int MODE, bool EPI = false>
cudaError_t tc_launch_mode_mid(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                               const TcParams& p, int grid, cudaStream_t s) {
  if (tile_n == 192 && pair) return tc_launch_bn<MODE, 192, true, EPI>(a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  if (tile_n == 192) return tc_launch_bn<MODE, 192, false, EPI>(a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  if (tile_n == 224 && pair) return tc_launch_bn<MODE, 224, true, EPI>(a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  if (tile_n == 224) return tc_launch_bn<MODE, 224, false, EPI>(a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  return cudaErrorInvalidValue;
}

// Defined in tc_tf32.cu (MODE 1), tc_bf16.cu (MODE 2: 16, 128 and 256
// columns), tc_bf16_mid.cu (MODE 2: 192 and 224 columns), tc_fp8.cu and
// tc_fp8_mid.cu (MODE 3, K-major operands only, the same widths).
cudaError_t tc_launch_tf32(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const CUtensorMap& tw, const TcParams& p, int grid,
                           cudaStream_t s);
cudaError_t tc_launch_bf16(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const CUtensorMap& tw, const TcParams& p, int grid,
                           cudaStream_t s);
cudaError_t tc_launch_bf16_mid(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                               const TcParams& p, int grid, cudaStream_t s);
cudaError_t tc_launch_fp8(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                          const CUtensorMap& tc, const CUtensorMap& tw, const TcParams& p, int grid, cudaStream_t s);
cudaError_t tc_launch_fp8_mid(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                              const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                              const TcParams& p, int grid, cudaStream_t s);
// Block-scaled operands (mode 4 MXFP8, 5 NVFP4), the swapped small-M form
// (tile_n 16) or 128 x 128 tiles: tc_bs.cu.
cudaError_t tc_launch_bs(int mode, int tile_n, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                         const CUtensorMap& tw, const TcParams& p, int grid, cudaStream_t s);

// The same kernels with the fused epilogue (EPI), K-major A: tc_tf32_epi.cu
// (TF32, every width), tc_bf16_epi.cu (BF16, 128 and 256 columns) and
// tc_bf16_epi_mid.cu (BF16, 192 and 224 columns).
cudaError_t tc_launch_tf32_epi(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                               const TcParams& p, int grid, cudaStream_t s);
cudaError_t tc_launch_bf16_epi(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                               const TcParams& p, int grid, cudaStream_t s);
cudaError_t tc_launch_bf16_epi_mid(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                                   const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                                   const TcParams& p, int grid, cudaStream_t s);

}  // namespace dgt
