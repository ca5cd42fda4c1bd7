// simt.cu -- exact-FP32 GEMM on the CUDA cores.
//
// The fp32 kernel of "bare-metal-bard" (first paragraph) climbs from one
// thread per output to coalesced loads, shared-memory tiling, register
// tiling, float4 loads, warp-level blocking and double buffering.  This is
// that end point, re-sized for a 152-SM part with 64K registers per SM:
//   * a 128 x 128 block tile, BK = 16, 256 threads, two CTAs per SM;
//   * warps tile the block 4 (M) x 2 (N) with 32 x 64 warp tiles, lanes tile a
//     warp 4 x 8, and every thread owns an 8 x 8 register tile split into
//     four 4 x 4 quadrants so each of its shared-memory reads is one float4
//     that the lanes sharing a row or column receive by broadcast;
//   * A is stored k-major in shared memory (transposed on the way in when the
//     operand is stored M x K) so both operands are read as float4 along M / N;
//   * the next K tile is copied global -> shared with cp.async (no register
//     staging) into the second buffer while the current one is multiplied;
//   * products are single-rounded FFMA in fp32, the accumulation order along
//     K is ascending, and the alpha/beta epilogue is fused into the stores.
#include <cuda_runtime.h>

#include "kernels.h"

namespace dgt {
namespace {

constexpr int BM = kSimtTileM, BN = kSimtTileN, BK = kSimtTileK, NT = kSimtThreads;
constexpr int PAD = 4;  // keeps rows 16-byte aligned and staggers the transposed copies across banks
constexpr int LDS = BM + PAD;

// cp.async copies global -> shared without staging in registers.  A source
// size of 0 copies nothing and fills the destination with zeros, which is how
// rows and columns outside the matrix enter the tile.
__device__ __forceinline__ void cp_async4(float* dst, const float* src, bool ok) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(d), "l"(src), "r"(ok ? 4 : 0) : "memory");
}

__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool ok) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(ok ? 16 : 0) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copies successive K tiles of a 128-wide operand into s[k][mn], keeping only
// two running source pointers per thread.
// K_CONTIG: the operand is stored with K contiguous (A as M x K, or B as N x K);
// each element lands transposed, so it is copied 4 bytes at a time (thread ->
// rows tid/4 and tid/4 + 64, k quad (tid%4)*4).  Otherwise the rows of the
// tile are contiguous in memory and are copied 16 bytes at a time when aligned
// (thread -> k rows tid/32 and tid/32 + 8, quad (tid%32)*4).
template <bool K_CONTIG, bool VEC>
struct TileCopier {
  const float* ptr[2];
  int avail;  // columns of this thread's quad inside the matrix (non-K_CONTIG)
  bool row_ok[2];

  __device__ __forceinline__ void init(const float* __restrict__ base, int64_t ld, int64_t mn0, int64_t lim,
                                       int64_t kbeg, int tid) {
    if (K_CONTIG) {
      const int row = tid >> 2, kq = (tid & 3) * 4;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t r = mn0 + row + 64 * h;
        row_ok[h] = r < lim;
        ptr[h] = base + (row_ok[h] ? r : 0) * ld + kbeg + kq;
      }
    } else {
      const int kr = tid >> 5, q = (tid & 31) * 4;
      const int64_t mn = mn0 + q;
      const int64_t left = lim - mn;
      avail = left <= 0 ? 0 : (left >= 4 ? 4 : static_cast<int>(left));
#pragma unroll
      for (int h = 0; h < 2; ++h) ptr[h] = base + (kbeg + kr + 8 * h) * ld + mn;
    }
  }

  // k_rem: how many K indices of this tile exist (>= BK except at the tail).
  // safe: any valid address, handed to copies of size 0; ld: leading dimension.
  __device__ __forceinline__ void issue(float (*s)[LDS], int k_rem, int tid, const float* safe, int64_t ld) {
    if (K_CONTIG) {
      const int row = tid >> 2, kq = (tid & 3) * 4;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool ok = row_ok[h] && kq + j < k_rem;
          cp_async4(&s[kq + j][row + 64 * h], ok ? ptr[h] + j : safe, ok);
        }
        ptr[h] += BK;
      }
    } else {
      const int kr = tid >> 5, q = (tid & 31) * 4;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const bool k_ok = kr + 8 * h < k_rem;
        if (VEC && avail == 4) {
          cp_async16(&s[kr + 8 * h][q], k_ok ? ptr[h] : safe, k_ok);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const bool ok = k_ok && j < avail;
            cp_async4(&s[kr + 8 * h][q + j], ok ? ptr[h] + j : safe, ok);
          }
        }
        ptr[h] += BK * ld;
      }
    }
  }
};

template <bool TA, bool TB, bool VEC, bool CVEC>
__global__ void __launch_bounds__(NT, 2) simt_gemm_kernel(SimtArgs p) {
  __shared__ __align__(16) float As[2][BK][LDS];
  __shared__ __align__(16) float Bs[2][BK][LDS];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;  // 4 x 2 warps
  const int lm = lane >> 3, ln = lane & 7;  // 4 x 8 lanes
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;

  const int64_t kbeg = static_cast<int64_t>(blockIdx.z) * p.k_per_split;
  const int64_t kend = (kbeg + p.k_per_split < p.K) ? kbeg + p.k_per_split : p.K;
  const int kspan = static_cast<int>(kend - kbeg);  // K elements of this slice (< 2^31)
  const int ntiles = (kspan + BK - 1) / BK;

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  // op(A) is K-contiguous when A is stored M x K (TA == 0); op(B) is
  // K-contiguous when B is stored N x K (TB == 1).
  TileCopier<!TA, VEC> ca;
  TileCopier<TB, VEC> cb;
  ca.init(p.A, p.lda, m0, p.M, kbeg, tid);
  cb.init(p.B, p.ldb, n0, p.N, kbeg, tid);
  if (ntiles > 0) {
    ca.issue(As[0], kspan, tid, p.A, p.lda);
    cb.issue(Bs[0], kspan, tid, p.B, p.ldb);
  }
  cp_async_commit();

  const int am = wm * 32 + lm * 4;  // A rows of quadrant 0 (quadrant 1: +16)
  const int bn = wn * 64 + ln * 4;  // B cols of quadrant 0 (quadrant 1: +32)

  for (int t = 0; t < ntiles; ++t) {
    const int cur = t & 1;
    if (t + 1 < ntiles) {
      const int k_rem = kspan - (t + 1) * BK;
      ca.issue(As[cur ^ 1], k_rem, tid, p.A, p.lda);
      cb.issue(Bs[cur ^ 1], k_rem, tid, p.B, p.ldb);
      cp_async_commit();
      cp_async_wait<1>();  // tile t has landed, tile t+1 may still be in flight
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][k][am]);
      const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][k][am + 16]);
      const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][k][bn]);
      const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][k][bn + 32]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();  // every warp is done with buffer `cur` before it is refilled
  }

  // Epilogue.  Rows: am + {0..3} and am + 16 + {0..3}; cols: bn + {0..3} and bn + 32 + {0..3}.
  const bool partial = p.splits > 1;
  float* __restrict__ out = partial ? p.ws + static_cast<int64_t>(blockIdx.z) * p.M * p.ws_ld : p.C;
  const int64_t ldo = partial ? p.ws_ld : p.ldc;
  const bool read_c = !partial && p.beta != 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = m0 + am + (i & 3) + (i >> 2) * 16;
    if (row >= p.M) continue;
    float* __restrict__ crow = out + row * ldo;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t col = n0 + bn + h * 32;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = partial ? acc[i][h * 4 + j] : p.alpha * acc[i][h * 4 + j];
      // the workspace is always 16-byte aligned with ws_ld % 4 == 0
      const bool vec = (partial || CVEC) && col + 3 < p.N;
      if (vec) {
        float4* dst = reinterpret_cast<float4*>(crow + col);
        if (read_c) {
          const float4 c = *dst;
          v[0] = fmaf(p.beta, c.x, v[0]);
          v[1] = fmaf(p.beta, c.y, v[1]);
          v[2] = fmaf(p.beta, c.z, v[2]);
          v[3] = fmaf(p.beta, c.w, v[3]);
        }
        *dst = make_float4(v[0], v[1], v[2], v[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (col + j < p.N) {
            float r = v[j];
            if (read_c) r = fmaf(p.beta, crow[col + j], r);
            crow[col + j] = r;
          }
        }
      }
    }
  }
}

template <bool TA, bool TB, bool VEC>
cudaError_t launch_cvec(const SimtArgs& a, dim3 grid, cudaStream_t s, bool cvec) {
  if (cvec)
    simt_gemm_kernel<TA, TB, VEC, true><<<grid, NT, 0, s>>>(a);
  else
    simt_gemm_kernel<TA, TB, VEC, false><<<grid, NT, 0, s>>>(a);
  return cudaGetLastError();
}

template <bool TA, bool TB>
cudaError_t launch_vec(const SimtArgs& a, dim3 grid, cudaStream_t s, bool vec, bool cvec) {
  return vec ? launch_cvec<TA, TB, true>(a, grid, s, cvec) : launch_cvec<TA, TB, false>(a, grid, s, cvec);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

cudaError_t launch_simt(const SimtArgs& a, cudaStream_t stream) {
  const int64_t gx = (a.N + BN - 1) / BN, gy = (a.M + BM - 1) / BM;
  if (gy > 65535 || a.splits > 65535) return cudaErrorInvalidConfiguration;
  dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(gy), static_cast<unsigned>(a.splits));
  const bool vec = aligned16(a.A) && aligned16(a.B) && (a.lda % 4 == 0) && (a.ldb % 4 == 0);
  const bool cvec = aligned16(a.C) && (a.ldc % 4 == 0);
  if (!a.transA && !a.transB) return launch_vec<false, false>(a, grid, stream, vec, cvec);
  if (!a.transA && a.transB) return launch_vec<false, true>(a, grid, stream, vec, cvec);
  if (a.transA && !a.transB) return launch_vec<true, false>(a, grid, stream, vec, cvec);
  return launch_vec<true, true>(a, grid, stream, vec, cvec);
}

}  // namespace dgt
