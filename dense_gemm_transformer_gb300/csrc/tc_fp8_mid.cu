// tc_fp8_mid.cu -- instantiations of the tcgen05 kernel for FP8 E4M3 operands
// with 192- and 224-column tiles (a translation unit of its own so that the
// FP8 instantiations compile in parallel).
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_fp8_mid(int tile_n, bool pair, bool a_mn, bool b_mn, const CUtensorMap& ta,
                              const CUtensorMap& tb, const CUtensorMap& tc, const CUtensorMap& tw,
                              const TcParams& p, int grid, cudaStream_t s) {
  if (a_mn || b_mn) return cudaErrorInvalidValue;
  return tc_launch_mode_mid<3>(tile_n, pair, a_mn, b_mn, ta, tb, tc, tw, p, grid, s);
}
}  // namespace dgt
