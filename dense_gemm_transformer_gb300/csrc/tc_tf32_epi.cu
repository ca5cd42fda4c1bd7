// tc_tf32_epi.cu -- the tcgen05 kernel for TF32 operands with the fused
// epilogue (bias, GELU, GELU'), every tile width, K-major operands.
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_tf32_epi(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                               const TcParams& p, int grid, cudaStream_t s) {
  if (tile_n == 192 || tile_n == 224)
    return tc_launch_mode_mid<1, true>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  return tc_launch_mode<1, true>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
}
}  // namespace dgt
