// tc_bf16_mid.cu -- instantiations of the tcgen05 kernel for BF16 operands
// with 192- and 224-column tiles (a translation unit of its own so that the
// BF16 instantiations compile in parallel).
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_bf16_mid(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                               const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                               const TcParams& p, int grid, cudaStream_t s) {
  return tc_launch_mode_mid<2>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
}
}  // namespace dgt
