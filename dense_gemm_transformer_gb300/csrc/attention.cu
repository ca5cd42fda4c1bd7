// attention.cu -- fused scaled dot-product attention, forward, on tcgen05.
//
// "bare-metal-bard" (third paragraph) reports a fused attention kernel for
// the GPT's causal self-attention: the scores never travel to global memory,
// and memory grows linearly with the context.  This kernel computes, for
// every problem (a batch element and head) and query row i,
//
//     O[i] = sum_j softmax_j(scale * q_i . k_j) v_j     (j <= i when causal)
//
// with bf16 Q, K, V ([problems][T][64], rows of 64 contiguous elements) and
// an fp32 O of the same shape.  The work items are (problem, tile of 128
// queries), the tiles with the most key blocks first; a persistent grid of
// two CTAs per SM takes them in turn, so that the copies for the next blocks
// and the next item run while the current one computes.  Per CTA:
//
//   warp 0      TMA producer: per item the Q tile (two buffers), then per
//               block of 64 keys the K and V blocks (rings of four), all as
//               128-byte swizzled rows of 64 bf16;
//   warp 1      allocates TMEM (two S buffers of 64 fp32 columns, O: 64,
//               two P buffers of 32); one lane issues S = Q K^T (M 128, N
//               64, K 64) into the S buffers, up to two blocks ahead;
//   warp 6      one lane issues O += P V (M 128, N 64, K 64: P read from
//               TMEM, V from shared memory MN-major) once the softmax has
//               written P; the two chains are independent, and one lane
//               issuing both spent most of every block issuing;
//   warps 2-5   the softmax: warp w owns TMEM lane quarter w % 4, one query
//               row per thread.  Per key block: read the row of S from TMEM
//               into registers (and release S), take its maximum (scale,
//               causal mask), write P = 2^(scale s - m) as bf16 pairs into
//               TMEM, and add the fp32 weights to the row sum l.  The
//               running maximum m is raised only when a block's maximum
//               exceeds it by more than kSlack (then O in TMEM and l are
//               rescaled by 2^(m_old - m_new)); otherwise the weights stay
//               below 2^kSlack, which bf16 and fp32 hold without loss of
//               relative precision, and O / l is unchanged.  At the end of
//               an item O / l is read from TMEM and stored.
//
// Exponentials are base 2 with log2(e) folded into the scale.  The row sum
// l adds the fp32 weights; the P V product uses them rounded to bf16.
// Every wait is bounded; on a timeout the CTA records the cause in the
// device status word, drains its copies and MMAs, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace dgt {
namespace {

constexpr int kAttnThreads = 224;  // producer, S issuer, four softmax warps, P V issuer
constexpr int kAttnD = 64;         // head dimension (one 128-byte bf16 row)
constexpr int kAttnBQ = 128;       // queries per item (UMMA M)
constexpr int kAttnBK = 64;        // keys per block (UMMA N of S, K of P V)
constexpr int kQBytes = kAttnBQ * 128;   // 128 rows x 128 bytes
constexpr int kKVBytes = kAttnBK * 128;  // 64 rows x 128 bytes
constexpr int kQBufs = 2;                // Q buffers
constexpr int kKVStages = 4;             // K and V ring stages
constexpr int kNumBars = 2 * kQBufs + 4 * kKVStages + 11;
constexpr int kSmemBytes = kQBufs * kQBytes + 2 * kKVStages * kKVBytes + 1024 + 8 * kNumBars + 16;
constexpr int kCtasPerSm = 2;
constexpr int kTmemCols = 256;  // S0 [0, 64), S1 [64, 128), O [128, 192), P0 [192, 224), P1 [224, 256)
constexpr int kSCol = 0;         // S of block n: kSCol + 64 (n % 2)
constexpr int kOCol = 128;
constexpr int kPCol = 192;       // P of block n: kPCol + 32 (n % 2)
constexpr float kSlack = 8.f;   // log2 of the largest weight a stale maximum allows

struct AttnParams {
  int problems, T, q_tiles, k_blocks, causal, items;
  float scale_log2;  // scale * log2(e)
  float* O;
  int o_v8;  // O is 32-byte aligned: rows are stored 32 bytes (one DRAM sector) per instruction
  int* status;
  uint64_t wait_ns;
};

struct Item {
  int problem, qt, blocks;
};

__device__ __forceinline__ Item decode_item(const AttnParams& p, int w) {
  Item it;
  it.problem = w % p.problems;
  it.qt = p.q_tiles - 1 - w / p.problems;
  const int seen = (it.qt + 1) * (kAttnBQ / kAttnBK);  // blocks up to the tile's last query
  it.blocks = (p.causal && seen < p.k_blocks) ? seen : p.k_blocks;
  return it;
}

// The k-th work item of this CTA.  Items are numbered longest first (the
// causal tiles with the most key blocks); round k of the grid takes items
// k G .. k G + G - 1 (G CTAs), in CTA order on even rounds and in reverse
// order on odd ones, so that the CTA given one of the longest items of a
// round is given one of the shortest of the next ("snake" order).  In CTA
// order on every round the CTAs that start with the longest tiles also
// drew the longest of every later round: 60 key blocks against 28 for the
// last CTA at T = 2048 (a mean of 43); the snake takes the most to 48.
// Each role of the CTA walks the same sequence.
__device__ __forceinline__ int item_of(int k) {
  const int G = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return k * G + ((k & 1) ? G - 1 - c : c);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The whole warp waits on `bar`; false for every lane when any lane gave up
// (so that the warp-collective TMEM accesses after it stay converged).
// Between tries the warp sleeps 32 ns (`nanosleep`), leaving the issue slots
// to the other softmax warps of its sub-partition: measured 2 % faster than
// tries with a suspend-time hint at T = 256, 1024 and 2048.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status, int code,
                                          uint64_t limit) {
  bool ok = mbar_try_wait(bar, parity);
  if (!ok) {
    const uint64_t t0 = globaltimer();
    for (;;) {
      __nanosleep(32);
      if (mbar_try_wait(bar, parity)) {
        ok = true;
        break;
      }
      if (*abort) break;
      if (globaltimer() - t0 > limit) {
        *abort = 1;
        if (status) atomicExch(status, code);
        break;
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

// One full 32-byte sector of a row of O (32-byte aligned address).
__device__ __forceinline__ void st_global_v8(float* dst, const uint32_t* v, float scale) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst),
               "f"(__uint_as_float(v[0]) * scale), "f"(__uint_as_float(v[1]) * scale),
               "f"(__uint_as_float(v[2]) * scale), "f"(__uint_as_float(v[3]) * scale),
               "f"(__uint_as_float(v[4]) * scale), "f"(__uint_as_float(v[5]) * scale),
               "f"(__uint_as_float(v[6]) * scale), "f"(__uint_as_float(v[7]) * scale)
               : "memory");
}

// Three-input max / min (with the packed fp32 pairs of ptx.cuh: fewer
// instructions per score in the softmax).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float exp2_fast(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Bounded drain of the last of `n` phases of `bar` (nothing when n == 0).
__device__ __forceinline__ void drain_last(uint32_t bar, uint32_t n, int* status, uint64_t limit) {
  if (n > 0) drain_wait(bar, (n - 1) & 1u, status, limit);
}

__global__ void __launch_bounds__(kAttnThreads, kCtasPerSm)
    attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_s = smem_u32(smem), k_s = q_s + kQBufs * kQBytes, v_s = k_s + kKVStages * kKVBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kQBufs * kQBytes + 2 * kKVStages * kKVBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  auto q_full = [&](uint32_t b) { return bar0 + 8 * b; };
  auto q_empty = [&](uint32_t b) { return bar0 + 8 * (kQBufs + b); };
  const uint32_t kv0 = bar0 + 8 * (2 * kQBufs);
  auto k_full = [&](uint32_t s) { return kv0 + 8 * s; };
  auto k_empty = [&](uint32_t s) { return kv0 + 8 * (kKVStages + s); };
  auto v_full = [&](uint32_t s) { return kv0 + 8 * (2 * kKVStages + s); };
  auto v_empty = [&](uint32_t s) { return kv0 + 8 * (3 * kKVStages + s); };
  // per S / P buffer x (block n uses x = n % 2, phase n / 2): S written,
  // S read, P written, P V done; then the item's O read out, and the drain
  const uint32_t sp0 = kv0 + 8 * (4 * kKVStages);
  auto s_full = [&](uint32_t x) { return sp0 + 8 * x; };
  auto s_free = [&](uint32_t x) { return sp0 + 8 * (2 + x); };
  auto p_full = [&](uint32_t x) { return sp0 + 8 * (4 + x); };
  auto pv_done = [&](uint32_t x) { return sp0 + 8 * (6 + x); };
  const uint32_t o_empty = sp0 + 64, drain = sp0 + 72, drain2 = sp0 + 80;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int b = 0; b < kQBufs; ++b) {
      mbar_init(q_full(b), 1);
      mbar_init(q_empty(b), 1);
    }
    for (int s = 0; s < kKVStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(s_free(x), 4);
      mbar_init(p_full(x), 4);
      mbar_init(pv_done(x), 1);
    }
    mbar_init(o_empty, 4);
    mbar_init(drain, 1);
    mbar_init(drain2, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t nq = 0, nk = 0, nv = 0;  // copies issued
      bool ok = true;
      for (int k = 0, w = item_of(0); w < p.items && ok; w = item_of(++k)) {
        const Item it = decode_item(p, w);
        const uint32_t qb = nq % kQBufs;
        if (!mbar_wait(q_empty(qb), ((nq / kQBufs) & 1u) ^ 1u, abort_flag, p.status, kDevTimeoutEmpty,
                             p.wait_ns))
          break;
        mbar_arrive_expect_tx(q_full(qb), kQBytes);
        tma_load_3d(q_s + qb * kQBytes, &tmQ, q_full(qb), 0, it.qt * kAttnBQ, it.problem);
        ++nq;
        for (int j = 0; j < it.blocks; ++j) {
          const uint32_t st = nk % kKVStages, ph = ((nk / kKVStages) & 1u) ^ 1u;
          if (!mbar_wait(k_empty(st), ph, abort_flag, p.status, kDevTimeoutEmpty, p.wait_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(k_full(st), kKVBytes);
          tma_load_3d(k_s + st * kKVBytes, &tmK, k_full(st), 0, j * kAttnBK, it.problem);
          ++nk;
          if (!mbar_wait(v_empty(st), ph, abort_flag, p.status, kDevTimeoutEmpty, p.wait_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(v_full(st), kKVBytes);
          tma_load_3d(v_s + st * kKVBytes, &tmV, v_full(st), 0, j * kAttnBK, it.problem);
          ++nv;
        }
      }
      // every copy lands before the CTA exits: the last phase of each buffer
      for (uint32_t b = 0; b < kQBufs; ++b) drain_last(q_full(b), (nq + kQBufs - 1 - b) / kQBufs, p.status, p.wait_ns);
      for (uint32_t s = 0; s < kKVStages; ++s) {
        drain_last(k_full(s), (nk + kKVStages - 1 - s) / kKVStages, p.status, p.wait_ns);
        drain_last(v_full(s), (nv + kKVStages - 1 - s) / kKVStages, p.status, p.wait_ns);
      }
    }
  } else if (warp == 1 || warp == 6) {
    // ------------------------------------------------------------ MMA issuers
    // Two lanes issue the two independent chains: warp 1's S = Q K^T of
    // every block into its S buffer (two blocks ahead at most, as the
    // buffers allow), warp 6's O += P V once the softmax has written P.  A
    // single lane issuing both spent most of each block issuing.  Each chain
    // of four MMAs goes out back to back from descriptors built once (a K
    // step of 16 elements advances a K-major descriptor by 32 bytes, 2 in
    // its address field, and V's MN-major one by 16 rows, 2048 bytes, 128).
    if (lane == 0) {
      const bool s_lane = warp == 1;
      const uint32_t idesc = s_lane ? make_idesc(1, false, false, kAttnBQ, kAttnBK)  // bf16, both K-major
                                    : make_idesc(1, false, true, kAttnBQ, kAttnD);   // V read MN-major
      const uint32_t my_drain = s_lane ? drain : drain2;
      uint32_t n = 0, ni = 0;  // blocks and items begun so far
      bool ok = true;
      for (int k = 0, w = item_of(0); w < p.items && ok; w = item_of(++k), ++ni) {
        const Item it = decode_item(p, w);
        const uint32_t qb = ni % kQBufs;
        for (int j = 0; j < it.blocks; ++j, ++n) {
          const uint32_t st = n % kKVStages, kph = (n / kKVStages) & 1u, x = n & 1u, xph = (n >> 1) & 1u;
          if (s_lane) {
            // Q of a new item, K of the block, and its S buffer read (block n - 2)
            if ((j == 0 && !mbar_wait(q_full(qb), (ni / kQBufs) & 1u, abort_flag, p.status, kDevTimeoutFull,
                                      p.wait_ns)) ||
                !mbar_wait(k_full(st), kph, abort_flag, p.status, kDevTimeoutFull, p.wait_ns) ||
                !mbar_wait(s_free(x), xph ^ 1u, abort_flag, p.status, kDevTimeoutAccEmpty, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = smem_desc_sw128(q_s + qb * kQBytes, 16, 1024);
            const uint64_t bd = smem_desc_sw128(k_s + st * kKVBytes, 16, 1024);
            const uint32_t d = tmem + kSCol + 64 * x;
            mma_bf16(d, ad, bd, idesc, 0u);
#pragma unroll
            for (int k = 1; k < kAttnD / 16; ++k) mma_bf16(d, ad + 2 * k, bd + 2 * k, idesc, 1u);
            mma_commit(k_empty(st));
            mma_commit(s_full(x));
            if (j == it.blocks - 1) mma_commit(q_empty(qb));  // the item's last S has read its Q
          } else {
            // the previous item's O read out, P of the block written (and O
            // rescaled), V of the block in
            if ((j == 0 && !mbar_wait(o_empty, (ni & 1u) ^ 1u, abort_flag, p.status, kDevTimeoutAccEmpty,
                                      p.wait_ns)) ||
                !mbar_wait(p_full(x), xph, abort_flag, p.status, kDevTimeoutFull, p.wait_ns) ||
                !mbar_wait(v_full(st), kph, abort_flag, p.status, kDevTimeoutFull, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t vd = smem_desc_sw128(v_s + st * kKVBytes, kKVBytes, 1024);
            const uint32_t a = tmem + kPCol + 32 * x, d = tmem + kOCol;
            mma_bf16_tmem_a(d, a, vd, idesc, j > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 1; k < kAttnBK / 16; ++k) mma_bf16_tmem_a(d, a + 8 * k, vd + 128 * k, idesc, 1u);
            mma_commit(v_empty(st));
            mma_commit(pv_done(x));
          }
        }
      }
      // every MMA this lane issued has completed once its drain barrier flips
      mma_commit(my_drain);
      drain_wait(my_drain, 0, p.status, p.wait_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax
    // Warp w (2..5) owns TMEM lane quarter w % 4: rows 32 (w % 4) .. of the
    // tile, one per thread.
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // this thread's query row in the tile
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const float c = p.scale_log2;
    const float kNegInf = -__int_as_float(0x7f800000);
    uint32_t nb = 0;
    bool ok = true;
    for (int k = 0, w = item_of(0); w < p.items && ok; w = item_of(++k)) {
      const Item it = decode_item(p, w);
      const int q_row = it.qt * kAttnBQ + r;
      float m = kNegInf, l = 0.f;
      for (int j = 0; j < it.blocks; ++j, ++nb) {
        const uint32_t x = nb & 1u, xph = (nb >> 1) & 1u;
        if (!warp_wait(s_full(x), xph, abort_flag, p.status, kDevTimeoutAccFull, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // the row of S: two loads, one wait; then release S for block n + 2
        uint32_t s[kAttnBK];
        {
          uint32_t lo[32], hi[32];
          tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kSCol + 64 * x), lo);
          tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kSCol + 64 * x + 32), hi);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) {
            s[t] = lo[t];
            s[32 + t] = hi[t];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_free(x));
        // keys this row sees in block j: [0, limit)
        const int key0 = j * kAttnBK;
        int limit = p.T - key0;
        if (p.causal && q_row - key0 + 1 < limit) limit = q_row - key0 + 1;
        limit = limit < 0 ? 0 : (limit > kAttnBK ? kAttnBK : limit);
        const bool whole = __all_sync(0xffffffffu, limit == kAttnBK);
        // the block's maximum of c s (log2 units): the largest s for c >= 0,
        // the smallest for c < 0 (masked keys never win), in eight chains
        float e8[8];
        if (whole) {
#pragma unroll
          for (int q = 0; q < 8; ++q) e8[q] = __uint_as_float(s[q]);
          if (c >= 0.f) {
#pragma unroll
            for (int t = 8; t < kAttnBK; t += 2)
              e8[(t >> 1) & 7] = max3f(e8[(t >> 1) & 7], __uint_as_float(s[t]), __uint_as_float(s[t + 1]));
          } else {
#pragma unroll
            for (int t = 8; t < kAttnBK; t += 2)
              e8[(t >> 1) & 7] = min3f(e8[(t >> 1) & 7], __uint_as_float(s[t]), __uint_as_float(s[t + 1]));
          }
        } else {
          const float none = c >= 0.f ? kNegInf : -kNegInf;
#pragma unroll
          for (int q = 0; q < 8; ++q) e8[q] = none;
#pragma unroll
          for (int t = 0; t < kAttnBK; ++t) {
            const float v = t < limit ? __uint_as_float(s[t]) : none;
            e8[t & 7] = c >= 0.f ? fmaxf(e8[t & 7], v) : fminf(e8[t & 7], v);
          }
        }
#pragma unroll
        for (int q = 4; q > 0; q >>= 1)
#pragma unroll
          for (int i = 0; i < q; ++i) e8[i] = c >= 0.f ? fmaxf(e8[i], e8[i + q]) : fminf(e8[i], e8[i + q]);
        const float bmax = limit > 0 ? e8[0] * c : kNegInf;
        // raise the running maximum only past the slack (always on the
        // first block, where m = -inf); the warp decides together, since
        // the rescale of O is warp-collective
        const bool raise = __any_sync(0xffffffffu, bmax > m + kSlack);
        const float m_new = raise ? fmaxf(m, bmax) : m;
        const float alpha = raise ? exp2_fast(m - m_new) : 1.f;  // 0 when m = -inf
        // P = 2^(c s - m_new) as bf16 pairs (key 2u in the low half of word
        // u) and the row sum of the fp32 weights (four partial sums)
        // (the exponent c s - m_new and the sums as packed pairs)
        const uint64_t cc = f2_pack(c, c), mm = f2_pack(-m_new, -m_new);
        uint64_t ps2[2] = {0ull, 0ull};  // +0.0f pairs
        uint32_t pk[kAttnBK / 2];
#pragma unroll
        for (int u = 0; u < kAttnBK / 2; ++u) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(s[2 * u]), __uint_as_float(s[2 * u + 1])), cc, mm), x0, x1);
          float p0 = exp2_fast(x0);
          float p1 = exp2_fast(x1);
          if (!whole) {
            p0 = 2 * u < limit ? p0 : 0.f;
            p1 = 2 * u + 1 < limit ? p1 : 0.f;
          }
          ps2[u & 1] = f2_add(ps2[u & 1], f2_pack(p0, p1));
          pk[u] = pack_bf16x2(p0, p1);
        }
        float sa, sb, sc, sd;
        f2_unpack(ps2[0], sa, sb);
        f2_unpack(ps2[1], sc, sd);
        const float bsum = (sa + sb) + (sc + sd);
        // P buffer x is free once P V of block n - 2 is done; O may be
        // rescaled once P V of block n - 1 is done
        if (!warp_wait(pv_done(x), xph ^ 1u, abort_flag, p.status, kDevTimeoutAccFull, p.wait_ns) ||
            (raise && j > 0 &&
             !warp_wait(pv_done(x ^ 1u), ((nb - 1) >> 1) & 1u, abort_flag, p.status, kDevTimeoutAccFull, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kPCol + 32 * x), pk);
        l = l * alpha + bsum;
        m = m_new;
        // O *= alpha when the maximum was raised after the first block
        if (raise && j > 0) {
#pragma unroll
          for (int h = 0; h < kAttnD; h += 32) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kOCol + h), o);
            tmem_wait_ld();
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
            tmem_st_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kOCol + h), o);
          }
        }
        // P and O visible to the next MMAs
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(x));
      }
      if (!ok) break;
      // the item's last P V, then O / l to global memory; O's columns are
      // free for the next item once read
      if (!warp_wait(pv_done((nb - 1) & 1u), ((nb - 1) >> 1) & 1u, abort_flag, p.status, kDevTimeoutAccFull,
                     p.wait_ns))
        break;
      tc_fence_after();
      uint32_t o[2][32];
      tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kOCol), o[0]);
      tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kOCol + 32), o[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_empty);
      if (q_row < p.T) {
        const float inv_l = 1.f / l;
        float* out = p.O + (static_cast<int64_t>(it.problem) * p.T + q_row) * kAttnD;
        // each thread writes its own row: whole 32-byte sectors when O
        // allows (half sectors, 16 bytes a store, measured four times the
        // DRAM write traffic of O), else 16 bytes a store
        if (p.o_v8) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int t = 0; t < 32; t += 8) st_global_v8(out + 32 * h + t, &o[h][t], inv_l);
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int t = 0; t < 32; t += 4)
              *reinterpret_cast<float4*>(out + 32 * h + t) =
                  make_float4(__uint_as_float(o[h][t]) * inv_l, __uint_as_float(o[h][t + 1]) * inv_l,
                              __uint_as_float(o[h][t + 2]) * inv_l, __uint_as_float(o[h][t + 3]) * inv_l);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// [problems][T][64] bf16 as a 3-D tensor map, boxes of 64 x `rows` x 1,
// 128-byte swizzle; rows past T read as zeros.
CUresult encode_qkv(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* m, const void* ptr, int64_t problems,
                    int64_t T, uint32_t rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kAttnD), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(problems)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kAttnD) * 2, static_cast<cuuint64_t>(T) * kAttnD * 2};
  cuuint32_t box[3] = {kAttnD, rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

int attention_grid(int64_t problems, int64_t T, int sms) {
  const int64_t items = problems * ((T + kAttnBQ - 1) / kAttnBQ);
  const int64_t slots = static_cast<int64_t>(kCtasPerSm) * (sms > 0 ? sms : 1);
  return static_cast<int>(items < slots ? items : slots);
}

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  cudaError_t e = tc_init_driver();
  if (e != cudaSuccess) return e;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tc_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tq, tk, tv;
  if (encode_qkv(encode, &tq, a.Q, a.problems, a.T, kAttnBQ) != CUDA_SUCCESS ||
      encode_qkv(encode, &tk, a.K, a.problems, a.T, kAttnBK) != CUDA_SUCCESS ||
      encode_qkv(encode, &tv, a.V, a.problems, a.T, kAttnBK) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  static std::atomic<uint64_t> attr_done{0};
  e = once_per_device(attr_done, [] {
    return cudaFuncSetAttribute(attention_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  AttnParams p;
  p.problems = static_cast<int>(a.problems);
  p.T = static_cast<int>(a.T);
  p.q_tiles = static_cast<int>((a.T + kAttnBQ - 1) / kAttnBQ);
  p.k_blocks = static_cast<int>((a.T + kAttnBK - 1) / kAttnBK);
  p.causal = a.causal ? 1 : 0;
  p.items = static_cast<int>(a.problems * p.q_tiles);
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.O = a.O;
  p.o_v8 = (reinterpret_cast<uintptr_t>(a.O) & 31u) == 0 ? 1 : 0;
  p.status = a.status;
  p.wait_ns = a.wait_ns > 0 ? a.wait_ns : kWaitLimitNs;
  const int grid = attention_grid(a.problems, a.T, a.sms);
  last_main_launch() = LaunchShape{dim3(static_cast<unsigned>(grid)), dim3(kAttnThreads), kSmemBytes, 1, true};
  return launch_pdl(attention_fwd_kernel, dim3(static_cast<unsigned>(grid)), dim3(kAttnThreads), kSmemBytes, stream,
                    tq, tk, tv, p);
}

}  // namespace dgt
