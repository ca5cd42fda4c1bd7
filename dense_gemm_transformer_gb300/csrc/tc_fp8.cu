// tc_fp8.cu -- instantiations of the tcgen05 kernel for FP8 E4M3 operands
// (kind::f8f6f4; both operands K-major), 16-, 128- and 256-column tiles.
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_fp8(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta, const CUtensorMap& tb,
                          const CUtensorMap& tc, const CUtensorMap& tw, const TcParams& p, int grid, cudaStream_t s) {
  if (a_mn || b_mn) return cudaErrorInvalidValue;
  return tc_launch_mode<3>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
}
}  // namespace dgt
