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
// an fp32 O of the same shape.  One CTA per (problem, tile of 128 queries):
//
//   warp 0      TMA producer: the Q tile once, then per block of 128 keys the
//               K block and the V block (128-byte swizzled rows of 64 bf16);
//   warp 1      allocates TMEM (S: 128 fp32 columns, O: 64), then one lane
//               issues S = Q K^T (M 128, N 128, K 64) and O += P V (M 128,
//               N 64, K 128: P from shared memory, V read MN-major);
//   warps 2-5   the softmax: warp w owns TMEM lane quarter w % 4, one query
//               row per thread.  Per key block: read S from TMEM (scale,
//               causal mask), update the running maximum m and sum l, rescale
//               O in TMEM by 2^(m_old - m_new) when m grew (after the previous
//               P V has completed), and write P = 2^(s - m) as bf16 into the
//               K-major, 128-byte-swizzled layout the P V MMA reads.  At the
//               end O / l is read from TMEM and stored.
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

constexpr int kAttnThreads = 192;  // producer, MMA, four softmax warps
constexpr int kAttnD = 64;         // head dimension (one 128-byte bf16 row)
constexpr int kAttnBQ = 128;       // queries per CTA (UMMA M)
constexpr int kAttnBK = 128;       // keys per block (UMMA N of S, K of P V)
constexpr int kTileBytes = kAttnBQ * 128;             // 128 rows x 128 bytes
constexpr int kSmemBytes = 5 * kTileBytes + 1024 + 256;  // Q, K, V, P (two tiles), align, barriers
constexpr int kTmemCols = 256;                         // S [0, 128), O [128, 192)
constexpr int kOCol = 128;

struct AttnParams {
  int problems, T, q_tiles, causal;
  float scale_log2;  // scale * log2(e)
  float* O;
  int* status;
  uint64_t wait_ns;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// The whole warp waits on `bar`; false for every lane when any lane gave up
// (so that the warp-collective TMEM accesses after it stay converged).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status, int code,
                                          uint64_t limit) {
  const bool ok = mbar_wait(bar, parity, abort, status, code, limit);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float exp2_fast(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// 3-D tiled load (one box of the [problems][T][64] tensor) completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t c0, int32_t c1,
                                            int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attention_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_s = smem_u32(smem), k_s = q_s + kTileBytes, v_s = k_s + kTileBytes, p_s = v_s + kTileBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 5 * kTileBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 10);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
  const uint32_t q_full = bar0, k_full = bar0 + 8, k_empty = bar0 + 16, v_full = bar0 + 24, v_empty = bar0 + 32,
                 s_full = bar0 + 40, s_free = bar0 + 48, p_full = bar0 + 56, o_full = bar0 + 64, drain = bar0 + 72;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the grid runs the last query tiles of every problem first: under the
  // causal mask they have the most key blocks (longest work first)
  const int problem = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.problems));
  const int qt = p.q_tiles - 1 - static_cast<int>(blockIdx.x / static_cast<unsigned>(p.problems));
  const int key_blocks = p.causal ? qt + 1 : (p.T + kAttnBK - 1) / kAttnBK;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(o_full, 1);
    mbar_init(drain, 1);
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
      uint32_t k_issued = 0, v_issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(q_full, kTileBytes);
      tma_load_3d(q_s, &tmQ, q_full, 0, qt * kAttnBQ, problem);
      for (int j = 0; j < key_blocks && ok; ++j) {
        const uint32_t ph = static_cast<uint32_t>(j) & 1u;
        // K block j once S_{j-1} has read K_{j-1}; V block j once P_{j-1} V_{j-1} has read V_{j-1}
        if (!mbar_wait(k_empty, ph ^ 1u, abort_flag, p.status, kDevTimeoutEmpty, p.wait_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(k_full, kTileBytes);
        tma_load_3d(k_s, &tmK, k_full, 0, j * kAttnBK, problem);
        ++k_issued;
        if (!mbar_wait(v_empty, ph ^ 1u, abort_flag, p.status, kDevTimeoutEmpty, p.wait_ns)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(v_full, kTileBytes);
        tma_load_3d(v_s, &tmV, v_full, 0, j * kAttnBK, problem);
        ++v_issued;
      }
      // every copy lands before the CTA exits (the consumers normally waited
      // for all of them already)
      drain_wait(q_full, 0, p.status, p.wait_ns);
      if (k_issued > 0) drain_wait(k_full, (k_issued - 1) & 1u, p.status, p.wait_ns);
      if (v_issued > 0) drain_wait(v_full, (v_issued - 1) & 1u, p.status, p.wait_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc(1, false, false, kAttnBQ, kAttnBK);  // bf16, both K-major
      const uint32_t idesc_o = make_idesc(1, false, true, kAttnBQ, kAttnD);    // V read MN-major
      bool ok = mbar_wait(q_full, 0, abort_flag, p.status, kDevTimeoutFull, p.wait_ns);
      for (int j = 0; j < key_blocks && ok; ++j) {
        const uint32_t ph = static_cast<uint32_t>(j) & 1u;
        // S_j = Q K_j^T, once K_j is in and the softmax has read S_{j-1}
        if (!mbar_wait(k_full, ph, abort_flag, p.status, kDevTimeoutFull, p.wait_ns) ||
            (j > 0 && !mbar_wait(s_free, ph ^ 1u, abort_flag, p.status, kDevTimeoutAccEmpty, p.wait_ns))) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kAttnD / 16; ++k)
          mma_bf16(tmem, smem_desc_sw128(q_s + 32 * k, 16, 1024), smem_desc_sw128(k_s + 32 * k, 16, 1024), idesc_s,
                   k > 0 ? 1u : 0u);
        mma_commit(k_empty);
        mma_commit(s_full);
        // O += P_j V_j, once the softmax has written P_j (and rescaled O)
        if (!mbar_wait(p_full, ph, abort_flag, p.status, kDevTimeoutFull, p.wait_ns) ||
            !mbar_wait(v_full, ph, abort_flag, p.status, kDevTimeoutFull, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int k = 0; k < kAttnBK / 16; ++k)
          mma_bf16(tmem + kOCol,
                   smem_desc_sw128(p_s + (k >> 2) * kTileBytes + 32 * (k & 3), 16, 1024),
                   smem_desc_sw128(v_s + 16 * 128 * k, kTileBytes, 1024), idesc_o, (j > 0 || k > 0) ? 1u : 0u);
        mma_commit(v_empty);
        mma_commit(o_full);
      }
      // every MMA this thread issued has completed once drain flips
      mma_commit(drain);
      drain_wait(drain, 0, p.status, p.wait_ns);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // this thread's query row in the tile
    const int q_row = qt * kAttnBQ + r;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    float m = -__int_as_float(0x7f800000), l = 0.f;
    bool ok = true;
    for (int j = 0; j < key_blocks; ++j) {
      const uint32_t ph = static_cast<uint32_t>(j) & 1u;
      if (!warp_wait(s_full, ph, abort_flag, p.status, kDevTimeoutAccFull, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // keys this row sees in block j: [0, limit)
      const int key0 = j * kAttnBK;
      int limit = p.T - key0;
      if (p.causal && q_row - key0 + 1 < limit) limit = q_row - key0 + 1;
      limit = limit < 0 ? 0 : (limit > kAttnBK ? kAttnBK : limit);
      // pass 1: the row maximum of this block (scaled, log2 units)
      float bmax = -__int_as_float(0x7f800000);
#pragma unroll 1
      for (int c = 0; c < kAttnBK; c += 32) {
        uint32_t s[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(c), s);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 32; ++t)
          if (c + t < limit) bmax = fmaxf(bmax, __uint_as_float(s[t]) * p.scale_log2);
      }
      const float m_new = fmaxf(m, bmax);
      const float alpha = exp2_fast(m - m_new);  // 0 on the first block (m = -inf)
      // P_{j-1} V_{j-1} must be done before O is rescaled and P is rewritten
      if (j > 0 && !warp_wait(o_full, ph ^ 1u, abort_flag, p.status, kDevTimeoutAccFull, p.wait_ns)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // pass 2: P = 2^(s - m_new) as bf16 into the P tile (K-major, 128-byte
      // swizzle: keys 64 h .. 64 h + 63 in tile h, row r at r * 128, 16-byte
      // chunk u at (u ^ (r % 8)) * 16), and the row sum
      float bsum = 0.f;
#pragma unroll 1
      for (int c = 0; c < kAttnBK; c += 32) {
        uint32_t s[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(c), s);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int t = 0; t < 32; t += 2) {
          const float p0 = (c + t < limit) ? exp2_fast(__uint_as_float(s[t]) * p.scale_log2 - m_new) : 0.f;
          const float p1 = (c + t + 1 < limit) ? exp2_fast(__uint_as_float(s[t + 1]) * p.scale_log2 - m_new) : 0.f;
          bsum += p0 + p1;
          pk[t / 2] = pack_bf16x2(p0, p1);
        }
        const uint32_t tile = p_s + static_cast<uint32_t>((c >> 6) * kTileBytes + r * 128);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ((c & 63) >> 3) + u;  // 16-byte chunk of the 128-byte row
          st_shared_v4(tile + static_cast<uint32_t>(((chunk ^ (r & 7)) << 4)), pk[4 * u], pk[4 * u + 1],
                       pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      // S may be overwritten now
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);
      l = l * alpha + bsum;
      m = m_new;
      // O *= alpha (O holds the previous blocks' P V; skip when no row of
      // this warp grew its maximum)
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c = 0; c < kAttnD; c += 32) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kOCol + c), o);
          tmem_wait_ld();
#pragma unroll
          for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
          tmem_st_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kOCol + c), o);
        }
        tmem_wait_st();
      }
      // P (generic-proxy stores) and O visible to the next MMAs
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // the last P V, then O / l to global memory
    if (ok && key_blocks > 0 &&
        warp_wait(o_full, static_cast<uint32_t>(key_blocks - 1) & 1u, abort_flag, p.status, kDevTimeoutAccFull,
                  p.wait_ns)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      float* out = p.O + (static_cast<int64_t>(problem) * p.T + q_row) * kAttnD;
#pragma unroll
      for (int c = 0; c < kAttnD; c += 32) {
        uint32_t o[32];
        __syncwarp();
        tmem_ld_32x32b_x32(tmem + lane_addr + static_cast<uint32_t>(kOCol + c), o);
        tmem_wait_ld();
        if (q_row < p.T) {
#pragma unroll
          for (int t = 0; t < 32; t += 4)
            *reinterpret_cast<float4*>(out + c + t) =
                make_float4(__uint_as_float(o[t]) * inv_l, __uint_as_float(o[t + 1]) * inv_l,
                            __uint_as_float(o[t + 2]) * inv_l, __uint_as_float(o[t + 3]) * inv_l);
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

// [problems][T][64] bf16 as a 3-D tensor map, boxes of 64 x 128 x 1,
// 128-byte swizzle; rows past T read as zeros.
CUresult encode_qkv(PFN_cuTensorMapEncodeTiled_v12000 encode, CUtensorMap* m, const void* ptr, int64_t problems,
                    int64_t T) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kAttnD), static_cast<cuuint64_t>(T),
                        static_cast<cuuint64_t>(problems)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kAttnD) * 2, static_cast<cuuint64_t>(T) * kAttnD * 2};
  cuuint32_t box[3] = {kAttnD, kAttnBQ, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  cudaError_t e = tc_init_driver();
  if (e != cudaSuccess) return e;
  PFN_cuTensorMapEncodeTiled_v12000 encode = tc_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  CUtensorMap tq, tk, tv;
  if (encode_qkv(encode, &tq, a.Q, a.problems, a.T) != CUDA_SUCCESS ||
      encode_qkv(encode, &tk, a.K, a.problems, a.T) != CUDA_SUCCESS ||
      encode_qkv(encode, &tv, a.V, a.problems, a.T) != CUDA_SUCCESS)
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
  p.causal = a.causal ? 1 : 0;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.O = a.O;
  p.status = a.status;
  p.wait_ns = a.wait_ns > 0 ? a.wait_ns : kWaitLimitNs;
  const int64_t grid = a.problems * p.q_tiles;
  last_main_launch() = LaunchShape{dim3(static_cast<unsigned>(grid)), dim3(kAttnThreads), kSmemBytes, 1, true};
  return launch_pdl(attention_fwd_kernel, dim3(static_cast<unsigned>(grid)), dim3(kAttnThreads), kSmemBytes, stream,
                    tq, tk, tv, p);
}

}  // namespace dgt
