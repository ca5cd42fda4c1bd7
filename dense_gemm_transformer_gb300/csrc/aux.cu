// aux.cu -- the small HBM-bound kernels around the GEMM kernels: the split-K
// reduction with the fused alpha/beta epilogue, the beta-only update used when
// K == 0 or alpha == 0, the operand re-pack that gives an operand with an
// unaligned leading dimension a 16-byte-aligned copy the TMA unit can read,
// and the transpose that turns an MN-major TF32 operand K-major.
// All are grid-stride loops sized to at most eight CTAs per SM.  Also here:
// the empty kernel that reproduces a GEMM kernel's launch configuration
// (the launch-cost floor a benchmark reports beside each shape).
#include <cuda_runtime.h>

#include <cstdint>

#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dgt {
namespace {

int grid_for(int64_t work, int threads) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t blocks = (work + threads - 1) / threads;
  int64_t cap = static_cast<int64_t>(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

// One thread per 4-column group of a row; the workspace rows are 16-byte
// aligned (ws_ld % 4 == 0), C is read/written by float4 only when CVEC.
template <bool CVEC>
__global__ void splitk_reduce_kernel(int64_t M, int64_t N, int splits, const float* __restrict__ ws, int64_t ws_ld,
                                     float* __restrict__ C, int64_t ldc, float alpha, float beta, EpiParams epi,
                                     int64_t row0) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t groups = (N + 3) / 4;
  const int64_t total = M * groups;
  const int64_t slice = M * ws_ld;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = g / groups, c = (g % groups) * 4;
    const float* src = ws + r * ws_ld + c;
    // Slices are loaded kBatch at a time (independent loads in flight: with
    // deep K there are dozens of slices and few output elements) and added in
    // ascending order.
    constexpr int kBatch = 8;
    float4 s = *reinterpret_cast<const float4*>(src);
    for (int k0 = 1; k0 < splits; k0 += kBatch) {
      float4 t[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (k0 + u < splits) t[u] = *reinterpret_cast<const float4*>(src + (k0 + u) * slice);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (k0 + u < splits) {
          s.x += t[u].x;
          s.y += t[u].y;
          s.z += t[u].z;
          s.w += t[u].w;
        }
      }
    }
    float v[4] = {alpha * s.x, alpha * s.y, alpha * s.z, alpha * s.w};
    float* dst = C + r * ldc + c;
    const bool epi_on = epilogue_active(epi);
    if (CVEC && c + 3 < N) {
      float4* d4 = reinterpret_cast<float4*>(dst);
      if (beta != 0.f) {
        const float4 old = *d4;
        v[0] = fmaf(beta, old.x, v[0]);
        v[1] = fmaf(beta, old.y, v[1]);
        v[2] = fmaf(beta, old.z, v[2]);
        v[3] = fmaf(beta, old.w, v[3]);
      }
      if (epi_on) {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = apply_epilogue(epi, v[j], row0 + r, c + j);
      }
      *d4 = make_float4(v[0], v[1], v[2], v[3]);
    } else {
      for (int j = 0; j < 4 && c + j < N; ++j) {
        float o = (beta != 0.f) ? fmaf(beta, dst[j], v[j]) : v[j];
        if (epi_on) o = apply_epilogue(epi, o, row0 + r, c + j);
        dst[j] = o;
      }
    }
  }
}

__global__ void scale_kernel(int64_t M, int64_t N, float* __restrict__ C, int64_t ldc, float beta, EpiParams epi) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t total = M * N;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = g / N, c = g % N;
    float* p = C + r * ldc + c;
    const float v = (beta != 0.f) ? beta * *p : 0.f;
    *p = apply_epilogue(epi, v, r, c);
  }
}

// C = epi(C): one thread per 4-column group of a row (16-byte accesses when
// the row allows), grid-stride; the epilogue's inputs come with the same
// coalesced pattern (a bias slice, or Z's row).  (Four groups per thread per
// iteration, for more loads in flight, measured slower: 56 registers halve
// the resident threads.)
template <bool CVEC>
__global__ void epilogue_kernel(int64_t M, int64_t N, float* __restrict__ C, int64_t ldc, EpiParams epi) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t groups = (N + 3) / 4;
  const int64_t total = M * groups;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = g / groups, c = (g % groups) * 4;
    float* dst = C + r * ldc + c;
    const float4 x = epilogue_fetch4(epi, r, c, N);
    if (CVEC && c + 3 < N) {
      float4 v = *reinterpret_cast<float4*>(dst);
      v.x = epilogue_finish(epi, v.x, x.x);
      v.y = epilogue_finish(epi, v.y, x.y);
      v.z = epilogue_finish(epi, v.z, x.z);
      v.w = epilogue_finish(epi, v.w, x.w);
      *reinterpret_cast<float4*>(dst) = v;
    } else {
      const float xs[4] = {x.x, x.y, x.z, x.w};
      for (int j = 0; j < 4 && c + j < N; ++j) dst[j] = epilogue_finish(epi, dst[j], xs[j]);
    }
  }
}

template <typename T>
__global__ void pack_kernel(const T* __restrict__ src, int64_t ld_src, T* __restrict__ dst, int64_t ld_dst,
                            int64_t rows, int64_t cols) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t total = rows * cols;
  for (int64_t g = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; g < total;
       g += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = g / cols, c = g % cols;
    dst[r * ld_dst + c] = src[r * ld_src + c];
  }
}

// 32 x 32 tiles through shared memory (one padding column keeps the
// transposed reads free of bank conflicts); reads and writes are both
// coalesced along rows.  Blocks of 32 x 8 threads loop over the tiles.
template <typename T>
__global__ void transpose_kernel(const T* __restrict__ src, int64_t ld_src, T* __restrict__ dst, int64_t ld_dst,
                                 int64_t rows, int64_t cols) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ T tile[32][33];
  const int64_t tiles_c = (cols + 31) / 32;
  const int64_t tiles = ((rows + 31) / 32) * tiles_c;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t r0 = (t / tiles_c) * 32, c0 = (t % tiles_c) * 32;
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int64_t r = r0 + i, c = c0 + threadIdx.x;
      if (r < rows && c < cols) tile[i][threadIdx.x] = src[r * ld_src + c];
    }
    __syncthreads();
    for (int i = threadIdx.y; i < 32; i += 8) {
      const int64_t c = c0 + i, r = r0 + threadIdx.x;
      if (c < cols && r < rows) dst[c * ld_dst + r] = tile[threadIdx.x][i];
    }
    __syncthreads();
  }
}

// fp32 with 16-byte aligned rows on both sides: 64 x 64 tiles, float4 loads
// and float4 stores (4 consecutive destination elements come from 4 source
// rows of the shared tile).  256 threads; each moves 4 float4 in and out.
__global__ void __launch_bounds__(256) transpose_f32x4_kernel(const float* __restrict__ src, int64_t ld_src,
                                                              float* __restrict__ dst, int64_t ld_dst, int64_t rows,
                                                              int64_t cols) {
  grid_dep_wait();
  grid_dep_launch();
  __shared__ float tile[64][65];
  const int64_t tiles_c = (cols + 63) / 64;
  const int64_t tiles = ((rows + 63) / 64) * tiles_c;
  const int t16 = threadIdx.x & 15, trow = threadIdx.x >> 4;  // 16 float4 per 64-wide row, 16 rows per pass
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int64_t r0 = (t / tiles_c) * 64, c0 = (t % tiles_c) * 64;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rr = trow + 16 * i;
      const int64_t r = r0 + rr, c = c0 + 4 * t16;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < rows) {
        const float* sp = src + r * ld_src + c;
        if (c + 3 < cols) {
          v = *reinterpret_cast<const float4*>(sp);
        } else {
          if (c + 0 < cols) v.x = sp[0];
          if (c + 1 < cols) v.y = sp[1];
          if (c + 2 < cols) v.z = sp[2];
        }
      }
      tile[rr][4 * t16 + 0] = v.x;
      tile[rr][4 * t16 + 1] = v.y;
      tile[rr][4 * t16 + 2] = v.z;
      tile[rr][4 * t16 + 3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int cc = trow + 16 * i;  // destination row = source column
      const int64_t c = c0 + cc, r = r0 + 4 * t16;
      if (c < cols && r < rows) {
        float* dp = dst + c * ld_dst + r;
        const float4 v = make_float4(tile[4 * t16 + 0][cc], tile[4 * t16 + 1][cc], tile[4 * t16 + 2][cc],
                                     tile[4 * t16 + 3][cc]);
        if (r + 3 < rows) {
          *reinterpret_cast<float4*>(dp) = v;
        } else {
          dp[0] = v.x;
          if (r + 1 < rows) dp[1] = v.y;
          if (r + 2 < rows) dp[2] = v.z;
        }
      }
    }
    __syncthreads();
  }
}

__global__ void null_kernel() {
  grid_dep_wait();
  grid_dep_launch();
}

// One thread per (atom, row within a quarter): the atom's 16 bytes for rows
// m0, m0 + 32, m0 + 64 and m0 + 96 of its tile, four blocks each.
__global__ void block_scales_tile_kernel(const uint8_t* __restrict__ S, int64_t rows, int64_t blocks, int64_t lds,
                                         uint8_t* __restrict__ T, int64_t groups, int64_t items) {
  grid_dep_wait();
  grid_dep_launch();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < items;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t atom = i / 32, m0 = i % 32;
    const int64_t rt = atom / groups, g = atom % groups;
    uint32_t w[4];
#pragma unroll
    for (int m1 = 0; m1 < 4; ++m1) {
      const int64_t r = rt * 128 + m1 * 32 + m0;
      uint32_t v = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int64_t b = g * 4 + j;
        const uint32_t x = (r < rows && b < blocks) ? S[r * lds + b] : 0u;
        v |= x << (8 * j);
      }
      w[m1] = v;
    }
    *reinterpret_cast<uint4*>(T + atom * 512 + m0 * 16) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

LaunchShape& last_main_launch() {
  thread_local LaunchShape shape;
  return shape;
}

cudaError_t launch_null(const LaunchShape& l, cudaStream_t stream) {
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = once_per_device(attr_done, [] {
    int dev = 0, optin = 0;
    cudaError_t r = cudaGetDevice(&dev);
    if (r == cudaSuccess) r = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (r == cudaSuccess) r = cudaFuncSetAttribute(null_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
    if (r == cudaSuccess) r = cudaFuncSetAttribute(null_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return r;
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = l.grid;
  cfg.blockDim = l.block;
  cfg.dynamicSmemBytes = l.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (l.cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(l.cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, null_kernel);
}

cudaError_t launch_transpose(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows, int64_t cols,
                             int elem_bytes, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const bool a16 = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0;
  if (elem_bytes == 4 && a16 && ld_src % 4 == 0 && ld_dst % 4 == 0) {
    const int64_t tiles64 = ((rows + 63) / 64) * ((cols + 63) / 64);
    return launch_pdl(transpose_f32x4_kernel, dim3(grid_for(tiles64 * 256, 256)), dim3(256), 0, stream,
                      static_cast<const float*>(src), ld_src, static_cast<float*>(dst), ld_dst, rows, cols);
  }
  const int64_t tiles = ((rows + 31) / 32) * ((cols + 31) / 32);
  const dim3 blocks(grid_for(tiles * 256, 256));
  const dim3 block(32, 8);
  if (elem_bytes == 1)
    return launch_pdl(transpose_kernel<uint8_t>, blocks, block, 0, stream, static_cast<const uint8_t*>(src), ld_src,
                      static_cast<uint8_t*>(dst), ld_dst, rows, cols);
  if (elem_bytes == 2)
    return launch_pdl(transpose_kernel<uint16_t>, blocks, block, 0, stream, static_cast<const uint16_t*>(src),
                      ld_src, static_cast<uint16_t*>(dst), ld_dst, rows, cols);
  return launch_pdl(transpose_kernel<float>, blocks, block, 0, stream, static_cast<const float*>(src), ld_src,
                    static_cast<float*>(dst), ld_dst, rows, cols);
}

cudaError_t launch_splitk_reduce(int64_t M, int64_t N, int splits, const float* ws, int64_t ws_ld, float* C,
                                 int64_t ldc, float alpha, float beta, const EpiParams& epi, int64_t row0,
                                 cudaStream_t stream) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int threads = 256;
  const dim3 blocks(grid_for(M * ((N + 3) / 4), threads));
  const bool cvec = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) && (ldc % 4 == 0);
  if (cvec)
    return launch_pdl(splitk_reduce_kernel<true>, blocks, dim3(threads), 0, stream, M, N, splits, ws, ws_ld, C, ldc,
                      alpha, beta, epi, row0);
  return launch_pdl(splitk_reduce_kernel<false>, blocks, dim3(threads), 0, stream, M, N, splits, ws, ws_ld, C, ldc,
                    alpha, beta, epi, row0);
}

cudaError_t launch_scale(int64_t M, int64_t N, float* C, int64_t ldc, float beta, const EpiParams& epi,
                         cudaStream_t stream) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int threads = 256;
  return launch_pdl(scale_kernel, dim3(grid_for(M * N, threads)), dim3(threads), 0, stream, M, N, C, ldc, beta, epi);
}

cudaError_t launch_epilogue(int64_t M, int64_t N, float* C, int64_t ldc, const EpiParams& epi, cudaStream_t stream) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int threads = 256;
  const dim3 blocks(grid_for(M * ((N + 3) / 4), threads));
  const bool cvec = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0) && (ldc % 4 == 0);
  if (cvec) return launch_pdl(epilogue_kernel<true>, blocks, dim3(threads), 0, stream, M, N, C, ldc, epi);
  return launch_pdl(epilogue_kernel<false>, blocks, dim3(threads), 0, stream, M, N, C, ldc, epi);
}

cudaError_t launch_pack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows, int64_t cols,
                        int elem_bytes, cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int threads = 256;
  const dim3 blocks(grid_for(rows * cols, threads));
  if (elem_bytes == 1)
    return launch_pdl(pack_kernel<uint8_t>, blocks, dim3(threads), 0, stream, static_cast<const uint8_t*>(src),
                      ld_src, static_cast<uint8_t*>(dst), ld_dst, rows, cols);
  if (elem_bytes == 2)
    return launch_pdl(pack_kernel<uint16_t>, blocks, dim3(threads), 0, stream, static_cast<const uint16_t*>(src),
                      ld_src, static_cast<uint16_t*>(dst), ld_dst, rows, cols);
  return launch_pdl(pack_kernel<float>, blocks, dim3(threads), 0, stream, static_cast<const float*>(src), ld_src,
                    static_cast<float*>(dst), ld_dst, rows, cols);
}

}  // namespace dgt

namespace dgt {
cudaError_t launch_block_scales_tile(const uint8_t* S, int64_t rows, int64_t blocks, int64_t lds, uint8_t* T,
                                     cudaStream_t stream) {
  const int64_t groups = block_scale_groups(blocks);
  const int64_t items = (rows + 127) / 128 * groups * 32;
  if (items == 0) return cudaSuccess;
  return launch_pdl(block_scales_tile_kernel, dim3(grid_for(items, 256)), dim3(256), 0, stream, S, rows, blocks, lds, T,
                    groups, items);
}
}  // namespace dgt
