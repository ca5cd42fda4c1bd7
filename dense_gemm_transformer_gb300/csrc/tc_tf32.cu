// tc_tf32.cu -- instantiations of the tcgen05 kernel for TF32 operands (kind::tf32).
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_tf32(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const CUtensorMap& tw, const TcParams& p, int grid,
                           cudaStream_t s) {
  if (tile_n == 192 || tile_n == 224) return tc_launch_mode_mid<1>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
  return tc_launch_mode<1>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
}
}  // namespace dgt
