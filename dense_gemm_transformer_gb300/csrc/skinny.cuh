// skinny.cuh -- parameters and launcher of the small-M (decode-shaped) kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace dgt {

// The kernel computes C^T = W^T X^T for C = X W with X of M <= 16 rows: the
// weights W are its 128-row MMA operand ("A", tiles of 128 weight columns
// of C), the activations X its 16-column operand ("B", K-major, rows past M
// zero-filled by the TMA unit).  Tile t covers C[:, 128 t .. 128 t + 127].
struct SkParams {
  int M;        // rows of the kernel's A: the caller's N (columns of C)
  int N;        // rows of the kernel's B: the caller's M (<= 16)
  int num_kb;   // K blocks of 128 bytes
  int kb_per;   // K blocks per slice
  int cluster;  // K slices = CTAs per cluster (1: no split)
  float alpha, beta;
  float* C;     // caller's C, element (m, n) at C[m * ldc + n]
  int64_t ldc;
  int* status;  // device status word (bounded waits)
  uint32_t fmt8;  // mode 3: operand format bits of the instruction descriptor (E4M3 / E5M2)
  const uint8_t* sfa;  // modes 4 / 5: the weights' scale factors, tiled (gemm_block_scales_tile)
  const uint8_t* sfb;  // modes 4 / 5: the activations' scale factors, tiled
  int64_t sf_groups;   // modes 4 / 5: 512-byte scale atoms per 128-row tile of either operand
};

constexpr int kSkinnyThreads = 192;  // TMA producer warp, MMA warp, four epilogue warps
constexpr int kSkinnyMaxCluster = 16;

constexpr int kSkinnyStages = 5;  // with the 8 KB receive buffer ~100 KB of shared memory: two CTAs per SM
// Pipeline depth per mode: NVFP4 stages also carry 4 KB of scale atoms, so
// it keeps 4 of them to stay at two CTAs per SM.
constexpr int skinny_stages(int mode) { return mode == 5 ? 4 : kSkinnyStages; }

// Launch on `grid` = tiles * p.cluster CTAs, clusters of p.cluster CTAs
// along x, with programmatic dependent launch.  mode: 1 TF32, 2 BF16, 3 8-bit
// floats (p.fmt8), 4 MXFP8 (p.fmt8, E8M0 scales in p.sfa / p.sfb), 5 NVFP4
// (E2M1 codes, UE4M3 scales).  a_mn: the weights are stored with the caller's N contiguous
// (transB == 0); BF16 only.
cudaError_t skinny_launch(int mode, bool a_mn, const CUtensorMap& ta, const CUtensorMap& tb, const SkParams& p,
                          int grid, cudaStream_t s);
// Clusters of `cluster` CTAs of the kernel that can be resident at once
// (0 when that cluster size cannot be launched).
int skinny_max_active_clusters(int mode, bool a_mn, int cluster);

}  // namespace dgt
