// tc_bs.cu -- the persistent tcgen05 kernel in its swapped small-M form for
// block-scaled operands: MXFP8 (kind::mxf8f6f4, E8M0 scales) and NVFP4
// (kind::mxf4nvf4, UE4M3 scales), K-major weights and activations.
#include "tc_launch.cuh"

namespace dgt {
cudaError_t tc_launch_bs(int mode, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tc,
                         const CUtensorMap& tw, const TcParams& p, int grid, cudaStream_t s) {
  if (mode == 4) return tc_launch_one<4, false, false, 16, true>(ta, tb, tc, tw, p, grid, s);
  if (mode == 5) return tc_launch_one<5, false, false, 16, true>(ta, tb, tc, tw, p, grid, s);
  return cudaErrorInvalidValue;
}
}  // namespace dgt
