// simt.cu -- exact-FP32 GEMM on the CUDA cores.
//
// The fp32 kernel of "bare-metal-bard" (first paragraph) climbs from one
// thread per output to coalesced loads, shared-memory tiling, register
// tiling, float4 loads, warp-level blocking and double buffering.  This is
// that end point, re-sized for a 152-SM part with 64K registers per SM:
//   * a 128 x TBN block tile (TBN = 128: two CTAs per SM, 8 x 8 outputs per
//     thread, the planner's choice; TBN = 256: one CTA per SM, 8 x 16
//     outputs per thread, which halves the shared-memory reads per FFMA but
//     leaves no second CTA to cover each tile's fill and stores), BK = 16,
//     256 threads;
//   * warps tile the block 4 (M) x 2 (N), lanes tile a warp 4 x 8, and every
//     thread's register tile is split into 4 x 4 quadrants so each of its
//     shared-memory reads is one float4 that the lanes sharing a row or column
//     receive by broadcast;
//   * both operands sit k-major in shared memory so they are read as float4
//     along M / N.  A K-contiguous A (stored M x K, 16-byte aligned) is
//     copied row by row with 16-byte copies into its stage and transposed in
//     shared memory (two 16-byte reads and eight 4-byte writes per thread per
//     K tile, then one more barrier); a K-contiguous operand that is not
//     aligned, or a K-contiguous B, is transposed on the way in with 4-byte
//     copies;
//   * K tiles are copied global -> shared with cp.async (no register
//     staging) into a ring of 3 (TBN = 128) or 4 (TBN = 256) stages, with one
//     barrier per tile; the register fragments of step k+1 are loaded while
//     step k is multiplied;
//   * work is scheduled as whole tiles when they fill whole waves of the
//     resident CTAs, and otherwise as whole-tile waves followed by stream-K
//     for the rest: the remaining (tile, k-tile) iterations are cut into one
//     equal contiguous run per resident CTA, runs that cover part of a tile
//     store a raw partial tile, and each such tile's partials are summed in
//     ascending k order (deterministic) by the last CTA to store one when a
//     tile has about two parts, else by a fixup kernel;
//   * products are single-rounded FFMA in fp32, the accumulation order along
//     K is ascending, and the alpha/beta epilogue is fused into the stores.
#include <cuda_runtime.h>

#include <type_traits>

#include "kernels.h"
#include "ptx.cuh"

namespace dgt {
namespace {

constexpr int BM = kSimtTileM, BK = kSimtTileK, NT = kSimtThreads;
constexpr int PAD = 4;  // keeps rows 16-byte aligned and staggers the transposed copies across banks

template <int TBN>
struct SimtCfg {
  static constexpr int LDA = BM + PAD;
  static constexpr int LDB = TBN + PAD;
  static constexpr int STAGES = (TBN == 256) ? 4 : 3;
  static constexpr int MIN_BLOCKS = (TBN == 256) ? 1 : 2;
  static constexpr int TN = TBN / 16;  // outputs per thread along N
  static constexpr int QN = TN / 4;    // float4 quadrants along N
  static constexpr int A_STAGE = BK * LDA;
  static constexpr int B_STAGE = BK * LDB;
  static constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;
  // A stored M x K with K contiguous: each K tile lands row by row (rows of
  // BK floats, padded to LDK) and is transposed in shared memory into one
  // k-major buffer of A_STAGE floats.
  static constexpr int LDK = BK + 4;
  static constexpr int A_RAW_STAGE = BM * LDK;
  static constexpr int SMEM_BYTES_RAW = (STAGES * (A_RAW_STAGE + B_STAGE) + A_STAGE) * 4;
};

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

// 16-byte copy of which the first `bytes` (0, 4, 8, 12 or 16) come from src
// and the rest are zero-filled.
__device__ __forceinline__ void cp_async16n(float* dst, const float* src, int bytes) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Packed pairs of fp32: fma.rn.f32x2 performs two independent
// round-to-nearest FMAs (the same results as two scalar fmaf) in one
// instruction, halving the issue slots the outer product needs.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ void ffma2(uint64_t& d, uint64_t a, uint64_t b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Copies successive K tiles of a ROWS-wide operand into s[k * LD + mn],
// keeping only a few running source pointers per thread.
// K_CONTIG: the operand is stored with K contiguous (A as M x K, or B as N x K);
// each element lands transposed, so it is copied 4 bytes at a time (thread ->
// rows tid/4 + 64h, k quad (tid%4)*4).  Otherwise the rows of the tile are
// contiguous in memory and are copied 16 bytes at a time when aligned
// (thread -> k rows tid/32 and tid/32 + 8, quads (tid%32)*4 + 128g).
template <bool K_CONTIG, bool VEC, int ROWS, int LD>
struct TileCopier {
  static constexpr int H = K_CONTIG ? ROWS / 64 : 2;
  static constexpr int G = K_CONTIG ? 1 : ROWS / 128;
  const float* ptr[H];
  int avail[G];  // columns of each quad inside the matrix (non-K_CONTIG)
  bool row_ok[H];

  __device__ __forceinline__ void init(const float* __restrict__ base, int64_t ld, int64_t mn0, int64_t lim,
                                       int64_t kbeg, int tid) {
    if (K_CONTIG) {
      const int row = tid >> 2, kq = (tid & 3) * 4;
#pragma unroll
      for (int h = 0; h < H; ++h) {
        const int64_t r = mn0 + row + 64 * h;
        row_ok[h] = r < lim;
        ptr[h] = base + (row_ok[h] ? r : 0) * ld + kbeg + kq;
      }
    } else {
      const int kr = tid >> 5, q = (tid & 31) * 4;
      const int64_t mn = mn0 + q;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int64_t left = lim - (mn + 128 * g);
        avail[g] = left <= 0 ? 0 : (left >= 4 ? 4 : static_cast<int>(left));
      }
#pragma unroll
      for (int h = 0; h < H; ++h) ptr[h] = base + (kbeg + kr + 8 * h) * ld + mn;
    }
  }

  // k_rem: how many K indices of this tile exist (>= BK except at the tail).
  // safe: any valid address, handed to copies of size 0; ld: leading dimension.
  __device__ __forceinline__ void issue(float* s, int k_rem, int tid, const float* safe, int64_t ld) {
    if (K_CONTIG) {
      const int row = tid >> 2, kq = (tid & 3) * 4;
#pragma unroll
      for (int h = 0; h < H; ++h) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool ok = row_ok[h] && kq + j < k_rem;
          cp_async4(s + (kq + j) * LD + row + 64 * h, ok ? ptr[h] + j : safe, ok);
        }
        ptr[h] += BK;
      }
    } else {
      const int kr = tid >> 5, q = (tid & 31) * 4;
#pragma unroll
      for (int h = 0; h < H; ++h) {
        const bool k_ok = kr + 8 * h < k_rem;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float* d = s + (kr + 8 * h) * LD + q + 128 * g;
          const float* src = ptr[h] + 128 * g;
          if (VEC && avail[g] == 4) {
            cp_async16(d, k_ok ? src : safe, k_ok);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const bool ok = k_ok && j < avail[g];
              cp_async4(d + j, ok ? src + j : safe, ok);
            }
          }
        }
        ptr[h] += BK * ld;
      }
    }
  }
};

// Copies successive K tiles of a K-contiguous, 16-byte-aligned operand of
// ROWS rows into s[row * LDK + k] (rows as stored): thread -> rows tid/4 and
// tid/4 + 64h, K quad tid%4; a quad that runs past K is zero-filled.
template <int ROWS, int LDK>
struct RowTileCopier {
  static constexpr int H = ROWS / 64;
  const float* ptr[H];
  bool row_ok[H];

  __device__ __forceinline__ void init(const float* __restrict__ base, int64_t ld, int64_t mn0, int64_t lim,
                                       int64_t kbeg, int tid) {
    const int row = tid >> 2, kq = (tid & 3) * 4;
#pragma unroll
    for (int h = 0; h < H; ++h) {
      const int64_t r = mn0 + row + 64 * h;
      row_ok[h] = r < lim;
      ptr[h] = base + (row_ok[h] ? r : 0) * ld + kbeg + kq;
    }
  }

  __device__ __forceinline__ void issue(float* s, int k_rem, int tid, const float* safe) {
    const int row = tid >> 2, kq = (tid & 3) * 4;
    const int left = k_rem - kq;
    const int bytes = left >= 4 ? 16 : left > 0 ? 4 * left : 0;
#pragma unroll
    for (int h = 0; h < H; ++h) {
      const int b = row_ok[h] ? bytes : 0;
      cp_async16n(s + (row + 64 * h) * LDK + kq, b > 0 ? ptr[h] : safe, b);
      ptr[h] += BK;
    }
  }
};

// The k-tile range [ks, ke) of one tile that a CTA accumulates in one go, and
// where the result goes.
struct Segment {
  int64_t tile;
  int ks, ke;
  int dest;       // kToC: finished tile; kToSlice: split-K slice; kToSlot: stream-K partial
  int64_t index;  // slice (kToSlice) or slot (kToSlot)
};
enum { kToC = 0, kToSlice = 1, kToSlot = 2 };

// First k-tile iteration of stream-K CTA c: iterations are the (tile, k-tile)
// pairs in tile-major order, split evenly over the grid.
__host__ __device__ __forceinline__ int64_t sk_begin(int64_t c, int64_t iters, int64_t grid) {
  return c * iters / grid;
}

// The stream-K CTA whose run holds iteration x.
__device__ __forceinline__ int64_t sk_owner(int64_t x, int64_t iters, int64_t grid) {
  int64_t c = x * grid / iters;
  while (c + 1 < grid && sk_begin(c + 1, iters, grid) <= x) ++c;
  while (c > 0 && sk_begin(c, iters, grid) > x) --c;
  return c;
}

template <int TBN, bool TA, bool TB, bool VEC, bool CVEC>
__global__ void __launch_bounds__(NT, SimtCfg<TBN>::MIN_BLOCKS) simt_gemm_kernel(SimtArgs p) {
  using Cfg = SimtCfg<TBN>;
  constexpr int S = Cfg::STAGES, TN = Cfg::TN, QN = Cfg::QN, LDA = Cfg::LDA, LDB = Cfg::LDB;
  grid_dep_wait();
  grid_dep_launch();
  extern __shared__ __align__(16) float smem[];
  // A K-contiguous A lands row by row and is transposed in shared memory.
  constexpr bool A_RAW = !TA && VEC;
  constexpr int A_RING = A_RAW ? Cfg::A_RAW_STAGE : Cfg::A_STAGE;
  float* As = smem;                      // [S][BK][LDA], or [S][BM][LDK] rows as stored
  float* Bs = smem + S * A_RING;         // [S][BK][LDB]
  float* Ax = Bs + S * Cfg::B_STAGE;     // [BK][LDA]: the transposed tile (A_RAW)

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;  // 4 x 2 warps
  const int lm = lane >> 3, ln = lane & 7;  // 4 x 8 lanes
  const int am = wm * 32 + lm * 4;          // A rows of quadrant 0 (quadrant 1: +16)
  const int bn = wn * (TBN / 2) + ln * 4;   // B cols of quadrant 0 (quadrant q: +32q)
  const int64_t tiles_n = (p.N + TBN - 1) / TBN;
  const int kt = static_cast<int>((p.K + BK - 1) / BK);  // k-tiles of a whole tile

  // The CTA's work: one segment (whole tile / split-K slice); or, for
  // stream-K, first whole tiles dp, dp + grid, ... below dp_tiles, then a
  // contiguous run of the (tile, k-tile) iterations of the remaining tiles,
  // which may span several tiles.  Thread 0 decodes each segment into shared
  // memory, so the scheduling state occupies no registers in the mainloop.
  struct SegState {
    Segment sg;
    int64_t it, it_end, dp;
    int valid;
    int last, nparts;        // inline stream-K fixup: this CTA sums the tile; its parts
    int64_t part0, owner0;   // slot of the first part, and the CTA that stored it
  };
  __shared__ SegState sh;
  if (tid == 0) {
    if (p.schedule == kSimtStreamK) {
      sh.it = sk_begin(blockIdx.x, p.iters, p.grid);
      sh.it_end = sk_begin(blockIdx.x + 1, p.iters, p.grid);
    } else {
      sh.it = 0;
      sh.it_end = 1;
    }
    sh.dp = blockIdx.x;
  }

  for (;;) {
    __syncthreads();  // every thread is done with the previous segment's descriptor
    if (tid == 0) {
      Segment sg;
      sh.valid = 1;
      if (p.schedule == kSimtStreamK && sh.dp < p.dp_tiles) {
        sg.tile = sh.dp;
        sg.ks = 0;
        sg.ke = kt;
        sg.dest = kToC;
        sh.dp += gridDim.x;
      } else if (p.schedule == kSimtStreamK && sh.it < sh.it_end) {
        const int64_t it = sh.it;
        sg.tile = p.dp_tiles + it / kt;
        sg.ks = static_cast<int>(it % kt);
        const int64_t left = sh.it_end - it;
        sg.ke = (kt - sg.ks <= left) ? kt : sg.ks + static_cast<int>(left);
        if (sg.ks == 0 && sg.ke == kt) {
          sg.dest = kToC;
        } else {
          sg.dest = kToSlot;
          sg.index = 2 * static_cast<int64_t>(blockIdx.x) +
                     (it == sk_begin(blockIdx.x, p.iters, p.grid) ? 0 : 1);
        }
        sh.it += sg.ke - sg.ks;
      } else if (p.schedule != kSimtStreamK && sh.it < sh.it_end) {
        sg.tile = static_cast<int64_t>(blockIdx.y) * tiles_n + blockIdx.x;
        if (p.schedule == kSimtSplitK) {
          const int per = static_cast<int>(p.k_per_split / BK);
          sg.ks = blockIdx.z * per;
          sg.ke = (sg.ks + per < kt) ? sg.ks + per : kt;
          sg.dest = kToSlice;
          sg.index = blockIdx.z;
        } else {
          sg.ks = 0;
          sg.ke = kt;
          sg.dest = kToC;
        }
        sh.it = sh.it_end;
      } else {
        sh.valid = 0;
      }
      sh.sg = sg;
    }
    __syncthreads();
    if (!sh.valid) break;
    const int64_t m0 = (sh.sg.tile / tiles_n) * BM;
    const int64_t n0 = (sh.sg.tile % tiles_n) * TBN;
    const int n = sh.sg.ke - sh.sg.ks;

    // Accumulators in pairs of adjacent columns (acc2[i][j] holds columns
    // 2j and 2j + 1 of row i), multiplied with packed FMAs; each element
    // still sums its products in ascending k with one fp32 FMA per product.
    uint64_t acc2[8][TN / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < TN / 2; ++j) acc2[i][j] = 0ull;  // +0.0f, +0.0f

    // op(A) is K-contiguous when A is stored M x K (TA == 0); op(B) is
    // K-contiguous when B is stored N x K (TB == 1).
    std::conditional_t<A_RAW, RowTileCopier<BM, Cfg::LDK>, TileCopier<!TA, VEC, BM, LDA>> ca;
    TileCopier<TB, VEC, TBN, LDB> cb;
    const int64_t kbeg = static_cast<int64_t>(sh.sg.ks) * BK;
    ca.init(p.A, p.lda, m0, p.M, kbeg, tid);
    cb.init(p.B, p.ldb, n0, p.N, kbeg, tid);
    auto issue_a = [&](float* dst, int k_rem) {
      if constexpr (A_RAW)
        ca.issue(dst, k_rem, tid, p.A);
      else
        ca.issue(dst, k_rem, tid, p.A, p.lda);
    };
    // The ring: tiles t+1 .. t+S-1 are in flight while tile t is multiplied;
    // one barrier per tile both publishes tile t and frees the stage that
    // tile t+S-1 overwrites (it held tile t-1).
#pragma unroll
    for (int st = 0; st < S - 1; ++st) {
      if (st < n) {
        const int k_rem = static_cast<int>(p.K - (kbeg + st * BK));
        issue_a(As + st * A_RING, k_rem);
        cb.issue(Bs + st * Cfg::B_STAGE, k_rem, tid, p.B, p.ldb);
      }
      cp_async_commit();
    }
    for (int t = 0; t < n; ++t) {
      cp_async_wait<S - 2>();
      __syncthreads();
      if (t + S - 1 < n) {
        const int nx = (t + S - 1) % S;
        const int k_rem = static_cast<int>(p.K - (kbeg + static_cast<int64_t>(t + S - 1) * BK));
        issue_a(As + nx * A_RING, k_rem);
        cb.issue(Bs + nx * Cfg::B_STAGE, k_rem, tid, p.B, p.ldb);
      }
      cp_async_commit();
      const float* a_s = As + (t % S) * A_RING;
      const float* b_s = Bs + (t % S) * Cfg::B_STAGE;
      if constexpr (A_RAW) {
        // Transpose tile t into Ax (each thread: rows m = tid % 128, K quads
        // tid / 128 and tid / 128 + 2), then publish it.  Ax was last read by
        // the previous tile's FMAs, which every thread finished before the
        // barrier above.
        const int m = tid & (BM - 1), kh = tid >> 7;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int kq = kh + 2 * j;
          const float4 v = *reinterpret_cast<const float4*>(a_s + m * Cfg::LDK + 4 * kq);
          Ax[(4 * kq + 0) * LDA + m] = v.x;
          Ax[(4 * kq + 1) * LDA + m] = v.y;
          Ax[(4 * kq + 2) * LDA + m] = v.z;
          Ax[(4 * kq + 3) * LDA + m] = v.w;
        }
        __syncthreads();
        a_s = Ax;
      }
      // Fragments of step k + 1 are loaded while step k is multiplied.
      float af[2][8];
      uint64_t bf[2][TN / 2];  // B fragment as column pairs, loaded as such
      auto load = [&](int k, int buf) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float4 v = *reinterpret_cast<const float4*>(a_s + k * LDA + am + 16 * r);
          af[buf][4 * r + 0] = v.x;
          af[buf][4 * r + 1] = v.y;
          af[buf][4 * r + 2] = v.z;
          af[buf][4 * r + 3] = v.w;
        }
#pragma unroll
        for (int q = 0; q < QN; ++q) {
          const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(b_s + k * LDB + bn + 32 * q);
          bf[buf][2 * q + 0] = v.x;
          bf[buf][2 * q + 1] = v.y;
        }
      };
      load(0, 0);
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        if (k + 1 < BK) load(k + 1, (k + 1) & 1);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint64_t a2 = pack2(af[k & 1][i], af[k & 1][i]);
#pragma unroll
          for (int j = 0; j < TN / 2; ++j) ffma2(acc2[i][j], a2, bf[k & 1][j]);
        }
      }
    }
    float acc[8][TN];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < TN / 2; ++j) unpack2(acc2[i][j], acc[i][2 * j], acc[i][2 * j + 1]);
    cp_async_wait<0>();
    __syncthreads();  // the ring is idle before the next segment refills it

    // Epilogue.  Rows am + {0..3}, am + 16 + {0..3}; cols bn + 32q + {0..3}.
    int dest = sh.sg.dest;
    const int64_t index = sh.sg.index;
    const int64_t em0 = (sh.sg.tile / tiles_n) * BM;  // re-read: the mainloop kept no copy
    const int64_t en0 = (sh.sg.tile % tiles_n) * TBN;
    if (dest == kToSlot) {
      // A stream-K partial: the raw 128 x TBN tile, rows of TBN floats
      // (quadrants wholly past column N are neither stored nor read back).
      float* __restrict__ slot = p.ws + index * (BM * TBN);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float* rowp = slot + (am + (i & 3) + (i >> 2) * 16) * TBN + bn;
#pragma unroll
        for (int q = 0; q < QN; ++q)
          if (en0 + bn + 32 * q < p.N)
            *reinterpret_cast<float4*>(rowp + 32 * q) =
                make_float4(acc[i][4 * q], acc[i][4 * q + 1], acc[i][4 * q + 2], acc[i][4 * q + 3]);
      }
      if (!p.sk_inline) continue;
      // Inline fixup: the partial is published (fence, then one arrival on
      // the tile's counter); the CTA whose arrival completes the count sums
      // every part of the tile, in ascending k order as the fixup kernel
      // does, and stores the tile through the normal epilogue.  It also
      // resets the counter for the next call.
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const int64_t t = sh.sg.tile - p.dp_tiles;
        const int64_t f = t * kt, l = f + kt - 1;
        const int64_t cf = sk_owner(f, p.iters, p.grid), cl = sk_owner(l, p.iters, p.grid);
        const int n = static_cast<int>(cl - cf + 1);
        const int prev = atomicAdd(p.sk_cnt + t, 1);
        sh.last = prev == n - 1;
        if (sh.last) atomicExch(p.sk_cnt + t, 0);
        sh.nparts = n;
        sh.owner0 = cf;
        sh.part0 = 2 * cf + (sk_begin(cf, p.iters, p.grid) >= f ? 0 : 1);
      }
      __syncthreads();
      if (!sh.last) continue;
      __threadfence();
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
      // Four rows at a time, one part at a time: at most 4 x QN float4 loads
      // in flight, so the sum needs no more registers than the mainloop.
#pragma unroll
      for (int g = 0; g < 2; ++g) {
#pragma unroll 1
        for (int j = 0; j < sh.nparts; ++j) {
          // parts after the first start their CTA's run: slot 2c
          const int64_t sl = j == 0 ? sh.part0 : 2 * (sh.owner0 + j);
          const float* __restrict__ src = p.ws + sl * (BM * TBN) + (am + 16 * g) * TBN + bn;
#pragma unroll
          for (int r = 0; r < 4; ++r) {
#pragma unroll
            for (int q = 0; q < QN; ++q) {
              if (en0 + bn + 32 * q >= p.N) continue;
              const float4 v = __ldcg(reinterpret_cast<const float4*>(src + r * TBN + 32 * q));
              float* a = acc[4 * g + r] + 4 * q;
              a[0] += v.x;
              a[1] += v.y;
              a[2] += v.z;
              a[3] += v.w;
            }
          }
        }
      }
      dest = kToC;
    }
    const bool partial = dest == kToSlice;
    float* __restrict__ out = partial ? p.ws + index * p.M * p.ws_ld : p.C;
    const int64_t ldo = partial ? p.ws_ld : p.ldc;
    const bool read_c = !partial && p.beta != 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t row = em0 + am + (i & 3) + (i >> 2) * 16;
      if (row >= p.M) continue;
      float* __restrict__ crow = out + row * ldo;
#pragma unroll
      for (int q = 0; q < QN; ++q) {
        const int64_t col = en0 + bn + 32 * q;
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = partial ? acc[i][4 * q + j] : p.alpha * acc[i][4 * q + j];
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
}

// Stream-K fixup: each output tile is handled by kFixupChunks CTAs (so that
// tiles summed from many partials -- deep K, few tiles -- still spread over
// the SMs).  A tile that one CTA finished in one segment was stored already;
// otherwise its partial tiles (one per CTA that touched it, in ascending k
// order) are summed in that fixed order and the alpha/beta epilogue applied.
constexpr int kFixupChunks = 16;

template <int TBN>
__global__ void __launch_bounds__(NT) simt_streamk_fixup_kernel(SimtArgs p) {
  constexpr int kMaxParts = 512;  // > the most resident CTAs that can share one tile
  __shared__ int64_t slots[kMaxParts];
  __shared__ int nparts;
  grid_dep_wait();
  grid_dep_launch();
  const int64_t tile = p.dp_tiles + blockIdx.x / kFixupChunks;  // tiles below dp_tiles were stored whole
  const int chunk = blockIdx.x % kFixupChunks;
  if (threadIdx.x == 0) {
    const int64_t kt = (p.K + BK - 1) / BK;
    const int64_t f = (tile - p.dp_tiles) * kt, l = f + kt - 1;
    const int64_t cf = sk_owner(f, p.iters, p.grid), cl = sk_owner(l, p.iters, p.grid);
    int n = 0;
    if (cf != cl) {
      for (int64_t c = cf; c <= cl && n < kMaxParts; ++c)
        slots[n++] = 2 * c + (sk_begin(c, p.iters, p.grid) >= f ? 0 : 1);
    }
    nparts = n;
  }
  __syncthreads();
  const int n = nparts;
  if (n == 0) return;  // one CTA finished this tile in one segment and stored it
  const int64_t tiles_n = (p.N + TBN - 1) / TBN;
  const int64_t m0 = (tile / tiles_n) * BM, n0 = (tile % tiles_n) * TBN;
  constexpr int kChunkVec = BM * TBN / 4 / kFixupChunks;  // float4 groups per chunk
  for (int e = chunk * kChunkVec + threadIdx.x; e < (chunk + 1) * kChunkVec; e += NT) {
    const int r = e / (TBN / 4), c4 = (e % (TBN / 4)) * 4;
    const int64_t row = m0 + r;
    if (row >= p.M || n0 + c4 >= p.N) continue;
    // Partials are loaded kBatch at a time (independent loads in flight: a
    // deep-K tile has dozens of partials, and one dependent L2 round trip per
    // partial would dominate) and added in ascending order.
    constexpr int kBatch = 8;
    const float* __restrict__ src = p.ws + r * TBN + c4;
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q0 = 0; q0 < n; q0 += kBatch) {
      float4 v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (q0 + u < n) v[u] = *reinterpret_cast<const float4*>(src + slots[q0 + u] * (BM * TBN));
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (q0 + u < n) {
          sum.x += v[u].x;
          sum.y += v[u].y;
          sum.z += v[u].z;
          sum.w += v[u].w;
        }
      }
    }
    float* crow = p.C + row * p.ldc + n0 + c4;
    const int64_t left = p.N - (n0 + c4);
    if (left > 0) crow[0] = (p.beta != 0.f) ? fmaf(p.beta, crow[0], p.alpha * sum.x) : p.alpha * sum.x;
    if (left > 1) crow[1] = (p.beta != 0.f) ? fmaf(p.beta, crow[1], p.alpha * sum.y) : p.alpha * sum.y;
    if (left > 2) crow[2] = (p.beta != 0.f) ? fmaf(p.beta, crow[2], p.alpha * sum.z) : p.alpha * sum.z;
    if (left > 3) crow[3] = (p.beta != 0.f) ? fmaf(p.beta, crow[3], p.alpha * sum.w) : p.alpha * sum.w;
  }
}

template <int TBN, bool TA, bool TB, bool VEC>
cudaError_t launch_cvec(const SimtArgs& a, dim3 grid, cudaStream_t s, bool cvec) {
  constexpr int smem = (!TA && VEC) ? SimtCfg<TBN>::SMEM_BYTES_RAW : SimtCfg<TBN>::SMEM_BYTES;
  auto kern = cvec ? simt_gemm_kernel<TBN, TA, TB, VEC, true> : simt_gemm_kernel<TBN, TA, TB, VEC, false>;
  static std::atomic<uint64_t> done[2] = {};
  cudaError_t e = once_per_device(done[cvec ? 1 : 0], [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, grid, dim3(NT), smem, s, a);
}

template <int TBN, bool TA, bool TB>
cudaError_t launch_vec(const SimtArgs& a, dim3 grid, cudaStream_t s, bool vec, bool cvec) {
  return vec ? launch_cvec<TBN, TA, TB, true>(a, grid, s, cvec) : launch_cvec<TBN, TA, TB, false>(a, grid, s, cvec);
}

template <int TBN>
cudaError_t launch_tbn(const SimtArgs& a, cudaStream_t stream) {
  dim3 grid;
  if (a.schedule == kSimtStreamK) {
    grid = dim3(static_cast<unsigned>(a.grid));
  } else {
    const int64_t gx = (a.N + TBN - 1) / TBN, gy = (a.M + BM - 1) / BM;
    if (gy > 65535 || a.splits > 65535) return cudaErrorInvalidConfiguration;
    grid = dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy),
                static_cast<unsigned>(a.schedule == kSimtSplitK ? a.splits : 1));
  }
  const auto aligned16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  const bool vec = aligned16(a.A) && aligned16(a.B) && (a.lda % 4 == 0) && (a.ldb % 4 == 0);
  const bool cvec = aligned16(a.C) && (a.ldc % 4 == 0);
  last_main_launch() = LaunchShape{
      grid, dim3(NT),
      static_cast<size_t>((!a.transA && vec) ? SimtCfg<TBN>::SMEM_BYTES_RAW : SimtCfg<TBN>::SMEM_BYTES), 1, true};
  cudaError_t e;
  if (!a.transA && !a.transB)
    e = launch_vec<TBN, false, false>(a, grid, stream, vec, cvec);
  else if (!a.transA && a.transB)
    e = launch_vec<TBN, false, true>(a, grid, stream, vec, cvec);
  else if (a.transA && !a.transB)
    e = launch_vec<TBN, true, false>(a, grid, stream, vec, cvec);
  else
    e = launch_vec<TBN, true, true>(a, grid, stream, vec, cvec);
  if (e != cudaSuccess || a.schedule != kSimtStreamK || a.sk_inline) return e;
  const int64_t tiles = ((a.M + BM - 1) / BM) * ((a.N + TBN - 1) / TBN);
  return launch_pdl(simt_streamk_fixup_kernel<TBN>, dim3(static_cast<unsigned>((tiles - a.dp_tiles) * kFixupChunks)),
                    dim3(NT), 0, stream, a);
}

}  // namespace

int64_t simt_streamk_slot_floats(int tile_n) { return static_cast<int64_t>(BM) * tile_n; }

cudaError_t launch_simt(const SimtArgs& a, cudaStream_t stream) {
  if (a.tile_n == 256) return launch_tbn<256>(a, stream);
  if (a.tile_n == 128) return launch_tbn<128>(a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace dgt
