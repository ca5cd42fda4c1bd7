// tc_bf16.cu -- instantiations of the tcgen05 kernel for BF16 operands (kind::f16).
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_bf16(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                           const CUtensorMap& tc, const CUtensorMap& tw, const TcParams& p, int grid,
                           cudaStream_t s) {
  return tc_launch_mode<2>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
}
}  // namespace dgt
