// tc_bf16_epi_mid.cu -- the tcgen05 kernel for BF16 operands with the fused
// epilogue, 192- and 224-column tiles, K-major A (a translation unit of its
// own so that the instantiations compile in parallel).
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_bf16_epi_mid(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                                   const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                                   const TcParams& p, int grid, cudaStream_t s) {
  return tc_launch_mode_mid<2, true>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
}
}  // namespace dgt
