// tc_bs.cu -- the persistent tcgen05 kernel for block-scaled operands: MXFP8
// (kind::mxf8f6f4, E8M0 scales) and NVFP4 (kind::mxf4nvf4, UE4M3 scales),
// K-major operands, in the swapped small-M form (tile_n 16: the weights are
// the 128-row operand, C stored transposed) and on 128 x 128 tiles of one
// CTA (M > 16).
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_bs(int mode, int tile_n, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                         const CUtensorMap& tw, const TcParams& p, int grid, cudaStream_t s) {
  if (tile_n == 16) {
    if (mode == 4) return tc_launch_one<4, false, false, 16, true>(ta, tb, tc, tw, p, grid, s);
    if (mode == 5) return tc_launch_one<5, false, false, 16, true>(ta, tb, tc, tw, p, grid, s);
  } else if (tile_n == 128) {
    if (mode == 4) return tc_launch_one<4, false, false, 128, false>(ta, tb, tc, tw, p, grid, s);
    if (mode == 5) return tc_launch_one<5, false, false, 128, false>(ta, tb, tc, tw, p, grid, s);
  }
  return cudaErrorInvalidValue;
}
}  // namespace dgt
