// skinny.cu -- the small-M (decode-shaped) GEMM on the tensor cores.
//
// "bare-metal-bard" uses one matmul for every projection of its GPT; at
// generation time those projections see a handful of token rows against
// a full weight matrix, and the multiply is bound by reading the weights
// from HBM once.  This kernel is built for that case on this part:
//
//   * the weights are the 128-row side of a tcgen05 MMA (128 x 16 x K per
//     tile) and stream through a TMA ring; the activations are the
//     16-column operand (rows past M are zero fill);
//   * one (tile, K slice) per CTA, small enough (5 stages and an 8 KB
//     receive buffer, ~100 KB of shared memory, 192 threads, 32 TMEM
//     columns) for two CTAs per SM:
//     clusters of up to 16 CTAs then fit twice into a GPC, and the next
//     call's CTAs can start while this one finishes (one CTA per SM with
//     twice the stages measured slower: its 12-CTA clusters fit only once
//     per GPC, so a third of them waited for a second wave);
//   * K is split across the CTAs of a thread-block cluster, and the slices
//     are summed through distributed shared memory: CTA r owns the r-th
//     share of the tile's elements; each CTA pushes the other owners' shares
//     of its 128 x 16 partial tile into their receive buffers with st.async
//     (counted on the owner's barrier), and each owner, once its barrier has
//     all the bytes, adds its share over all slices in ascending order and
//     writes C.  No workspace, no atomics, no second kernel, and no barrier
//     across the cluster after the MMAs (pulling the shares instead needed
//     two, and measured 6-8% slower);
//   * programmatic dependent launch: set-up (barriers, TMEM, descriptor
//     prefetch) and an L2 warm-up of this CTA's weight slice run before
//     griddepcontrol.wait, i.e. while the previous kernel in the stream is
//     still finishing.  Only L2 is touched before the wait, and L2 is where
//     global memory is kept coherent, so no stale value can be read.
//
// Every mbarrier wait is bounded; on a timeout the CTA records the cause in
// the status word, drains its own copies and MMAs, and an owner whose shares
// never arrive gives up its receive wait the same way.
#include "skinny.cuh"

#include "kernels.h"
#include "ptx.cuh"

namespace dgt {
namespace {

// MODE: 1 TF32 (fp32 operands), 2 BF16, 3 8-bit floats (E4M3 / E5M2 codes,
// the formats named at run time in SkParams::fmt8).
// MODE 4 / 5: block-scaled 8-bit (MXFP8: E4M3 / E5M2 with an E8M0 scale per
// 32 K) and 4-bit (NVFP4: E2M1 packed two per byte with a UE4M3 scale per 16
// K) codes; their TMA maps and K coordinates are in bytes.  Each stage then
// also carries both operands' scale factors for its 128 bytes of K, as
// 512-byte atoms (128 rows x 4 scale blocks) in the layout tcgen05.cp
// replicates into the TMEM cells the block-scaled MMA reads.
template <int MODE>
struct SkCfg {
  static constexpr bool BS = MODE >= 4;  // block-scaled
  static constexpr int ES = (MODE >= 3) ? 1 : (MODE == 2) ? 2 : 4;  // operand bytes (coordinate units)
  static constexpr int BM = 128;                   // weight rows per tile (UMMA M)
  static constexpr int BN = 16;                    // activation rows (UMMA N)
  static constexpr int BK = 128 / ES;              // K units per stage (one 128-byte swizzle row)
  static constexpr int UK = 32 / ES;                // K units of one MMA (32 bytes)
  static constexpr int CH = 128 / ES;              // weight rows in one 128-byte MN-major row
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN * 128;
  static constexpr int SF_ATOMS = (MODE == 5) ? 4 : (MODE == 4) ? 1 : 0;  // scale atoms per operand per stage
  static constexpr int SF_BYTES = SF_ATOMS * 512;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + 2 * SF_BYTES;
  static constexpr int STAGES = skinny_stages(MODE);
  // TMEM: the 16-column accumulator, then (block-scaled) one ring slot of
  // scale columns per stage: 4 columns per atom, A's atoms then B's.
  static constexpr int SF_COL0 = 32;
  static constexpr int SF_COLS = 2 * SF_ATOMS * 4;
  static constexpr int TMEM_NEED = BS ? SF_COL0 + STAGES * SF_COLS : 16;
  static constexpr int TMEM_COLS = TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : 256;
  static constexpr int NUM_BARS = 2 * STAGES + 3;     // full/empty per stage, accumulator full, drain, receive
  static constexpr int RECV_BYTES = (BN * BM / 4 + kSkinnyMaxCluster) * 16;  // shares pushed by the peers
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + RECV_BYTES + 1024 /*align*/ + 256 /*barriers*/;
  static constexpr int PREFETCH_KB = 16;              // K blocks of weights warmed in L2 before the wait
  static constexpr uint32_t FORMAT = (MODE == 3) ? 0u : (MODE == 2) ? 1u : 2u;  // 8-bit (fmt8) / bf16 / tf32
  static_assert(!BS || TMEM_NEED <= 256, "block-scaled: two CTAs per SM");
  static_assert(2 * (SMEM_BYTES + 1024) <= 233472, "two CTAs per SM (228 KB, 1 KB reserved per CTA)");
  static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
  static_assert(BM * BN * 4 <= STAGES * STAGE_BYTES, "the partial tile fits in the drained stages");
  static_assert(NUM_BARS * 8 + 8 <= 256, "barrier area");
};

template <int MODE>
__device__ __forceinline__ void sk_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  static_assert(MODE <= 3, "block-scaled kinds take scale factors (sk_mma_bs)");
  if (MODE == 3)
    mma_f8f6f4(d, a, b, idesc, acc);
  else if (MODE == 2)
    mma_bf16(d, a, b, idesc, acc);
  else
    mma_tf32(d, a, b, idesc, acc);
}

template <int MODE, bool A_MN>
__global__ void __launch_bounds__(kSkinnyThreads, 2)
    skinny_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const SkParams p) {
  using Cfg = SkCfg<MODE>;
  constexpr int S = Cfg::STAGES;
  // MODE 3 names its operand formats at run time (the FORMAT fields are 0);
  // the block-scaled modes build theirs per MMA.
  const uint32_t IDESC = make_idesc(Cfg::FORMAT, A_MN, false, Cfg::BM, Cfg::BN) | (MODE == 3 ? p.fmt8 : 0u);
  static_assert(!Cfg::BS || !A_MN, "block-scaled operands are K-major");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* recv = reinterpret_cast<float*>(smem + S * Cfg::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::STAGE_BYTES + Cfg::RECV_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  const uint32_t accf_bar = bar0 + 8u * (2 * S);
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 1);
  const uint32_t recv_bar = bar0 + 8u * (2 * S + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cs = p.cluster;
  const int rank = (cs > 1) ? static_cast<int>(cluster_ctarank()) : 0;
  const int tile = static_cast<int>(blockIdx.x) / cs;
  const int kb0 = rank * p.kb_per;
  const int kb1 = (kb0 + p.kb_per < p.num_kb) ? kb0 + p.kb_per : p.num_kb;
  const int row0 = tile * Cfg::BM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(accf_bar, 1);
    mbar_init(drain_bar, 1);
    mbar_init(recv_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    // Warm L2 with the first K blocks of this CTA's weight slice.
    const int pf_end = (kb0 + Cfg::PREFETCH_KB < kb1) ? kb0 + Cfg::PREFETCH_KB : kb1;
    for (int kb = kb0; kb < pf_end; ++kb) {
      if (A_MN) {
#pragma unroll
        for (int c = 0; c < Cfg::BM / Cfg::CH; ++c) tma_prefetch_l2_2d(&tmA, row0 + c * Cfg::CH, kb * Cfg::BK);
      } else {
        tma_prefetch_l2_2d(&tmA, kb * Cfg::BK, row0);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  // Every CTA's receive barrier exists before any peer can push to it.
  if (cs > 1) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // From here on global memory written by earlier kernels is read or written.
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.status, kDevTimeoutEmpty)) {
          ok = false;
          break;
        }
        const uint32_t fb = full_bar(stage);
        mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
        const uint32_t a_dst = smem0 + stage * Cfg::STAGE_BYTES;
        const int k0 = kb * Cfg::BK;
        if (A_MN) {
#pragma unroll
          for (int c = 0; c < Cfg::BM / Cfg::CH; ++c)
            tma_load_2d(a_dst + c * Cfg::BK * 128, &tmA, fb, row0 + c * Cfg::CH, k0);
        } else {
          tma_load_2d(a_dst, &tmA, fb, k0, row0);
        }
        tma_load_2d(a_dst + Cfg::A_BYTES, &tmB, fb, k0, 0);
        if constexpr (Cfg::BS) {
          // both operands' scale atoms for this stage's 128 bytes of K
          const uint32_t sf_dst = a_dst + Cfg::A_BYTES + Cfg::B_BYTES;
          bulk_copy_g2s(sf_dst, p.sfa + (static_cast<int64_t>(tile) * p.sf_groups + kb * Cfg::SF_ATOMS) * 512,
                        Cfg::SF_BYTES, fb);
          bulk_copy_g2s(sf_dst + Cfg::SF_BYTES, p.sfb + static_cast<int64_t>(kb) * Cfg::SF_ATOMS * 512, Cfg::SF_BYTES,
                        fb);
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) {
        const uint32_t n = issued < static_cast<uint32_t>(S) ? issued : static_cast<uint32_t>(S);
        for (uint32_t i = issued - n; i < issued; ++i) drain_wait(full_bar(i % S), (i / S) & 1u, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      // Stage 0's descriptors; a stage's are these plus its byte offset in
      // the address field (bits 0-13, address >> 4: every shared address
      // here is below 256 KB, so the field cannot carry).  Rebuilding the
      // 64-bit descriptors between these small MMAs is what would pace the
      // single issuing thread.
      const uint64_t a_desc0 = smem_desc_sw128(smem0, A_MN ? Cfg::BK * 128 : 16, 1024);
      const uint64_t b_desc0 = smem_desc_sw128(smem0 + Cfg::A_BYTES, 16, 1024);
      [[maybe_unused]] const uint64_t sf_desc0 = smem_desc_noswizzle(smem0 + Cfg::A_BYTES + Cfg::B_BYTES, 128);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(full_bar(stage), phase, abort_flag, p.status, kDevTimeoutFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t soff = static_cast<uint64_t>((stage * Cfg::STAGE_BYTES) >> 4);
        if constexpr (Cfg::BS) {
          // This stage's scale atoms into its TMEM ring slot (the slot's
          // previous MMAs are complete: this stage's copies could only be
          // issued after they released it), then four block-scaled MMAs of
          // 32 bytes of K each: MXFP8 picks its byte of the 32-bit scale
          // cells by scale-factor ID j; NVFP4 takes atom j's four bytes.
          const uint32_t sf_col = tmem_base + static_cast<uint32_t>(Cfg::SF_COL0 + stage * Cfg::SF_COLS);
#pragma unroll
          for (int a = 0; a < 2 * Cfg::SF_ATOMS; ++a) tmem_cp_32x128b_x4(sf_col + 4 * a, sf_desc0 + soff + 32 * a);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t ad = a_desc0 + soff + 2 * j;
            const uint64_t bd = b_desc0 + soff + 2 * j;
            const uint32_t acc = (kb > kb0 || j > 0) ? 1u : 0u;
            if constexpr (MODE == 4)
              mma_mxf8f6f4_bs(tmem_base, ad, bd,
                              make_idesc_bs(0, 0, true, Cfg::BM, Cfg::BN, static_cast<uint32_t>(j),
                                            static_cast<uint32_t>(j)) | p.fmt8,
                              sf_col, sf_col + 4, acc);
            else
              mma_mxf4nvf4_bs(tmem_base, ad, bd, make_idesc_bs(1, 1, false, Cfg::BM, Cfg::BN, 0, 0),
                              sf_col + 4 * j, sf_col + 4 * (Cfg::SF_ATOMS + j), acc);
          }
        } else {
#pragma unroll
          for (int j = 0; j < Cfg::BK / Cfg::UK; ++j) {
            const uint64_t ad = a_desc0 + soff + ((A_MN ? j * Cfg::UK * 128 : j * Cfg::UK * Cfg::ES) >> 4);
            const uint64_t bd = b_desc0 + soff + ((j * Cfg::UK * Cfg::ES) >> 4);
            sk_mma<MODE>(tmem_base, ad, bd, IDESC, (kb > kb0 || j > 0) ? 1u : 0u);
          }
        }
        mma_commit(empty_bar(stage));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) mma_commit(accf_bar);
      // Every MMA this thread issued has finished once drain_bar flips.
      mma_commit(drain_bar);
      drain_wait(drain_bar, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lanes 32*(w%4)..+31: rows sub*32 + lane of the tile.
    const int sub = warp & 3;
    const int rt = sub * 32 + lane;
    const bool got = __all_sync(0xffffffffu, mbar_wait(accf_bar, 0, abort_flag, p.status, kDevTimeoutAccFull));
    float v[Cfg::BN];
    if (got && kb1 > kb0) {
      tc_fence_after();
      uint32_t r[Cfg::BN];
      tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(sub * 32) << 16), r);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < Cfg::BN; ++j) v[j] = __uint_as_float(r[j]);
    } else {
#pragma unroll
      for (int j = 0; j < Cfg::BN; ++j) v[j] = 0.f;
    }
    if (cs == 1) {
      const int64_t row = static_cast<int64_t>(row0) + rt;
      if (got && row < p.M) {
        // Lanes hold consecutive columns of C: each store of the warp is contiguous.
#pragma unroll
        for (int j = 0; j < Cfg::BN; ++j) {
          if (j < p.N) {
            float* dst = p.C + static_cast<int64_t>(j) * p.ldc + row;
            float out = p.alpha * v[j];
            if (p.beta != 0.f) out = fmaf(p.beta, *dst, out);
            *dst = out;
          }
        }
      }
    } else {
      // The partial tile, column-major (element (rt, j) at j * BM + rt), in
      // the first stage: every MMA has read its operands by now.
      float* red = reinterpret_cast<float*>(smem);
#pragma unroll
      for (int j = 0; j < Cfg::BN; ++j) red[j * Cfg::BM + rt] = v[j];
      asm volatile("bar.sync 1, 128;" ::: "memory");  // the four epilogue warps
      // Groups of four rows of one column; CTA q owns groups [q per, (q+1) per).
      // Push every other owner's groups into its receive buffer (slot of this
      // rank), counted on its receive barrier.
      constexpr int G = Cfg::BM / 4;
      const int total = p.N * G;
      const int per = (total + cs - 1) / cs;
      const int et = static_cast<int>(threadIdx.x) - 64;
      const uint32_t recv0 = smem_u32(recv);
      for (int g = et; g < total; g += 128) {
        const int q = g / per;
        if (q == rank) continue;
        const float4 val = *reinterpret_cast<const float4*>(red + 4 * g);
        const uint32_t dst = dsmem_map(recv0 + 16u * static_cast<uint32_t>(rank * per + (g - q * per)),
                                       static_cast<uint32_t>(q));
        st_async_f32x4(dst, val, dsmem_map(recv_bar, static_cast<uint32_t>(q)));
      }
      const int g0 = rank * per;
      const int g1 = (g0 + per < total) ? g0 + per : total;
      const int mine = (g1 > g0) ? g1 - g0 : 0;
      if (et == 0) mbar_arrive_expect_tx(recv_bar, static_cast<uint32_t>((cs - 1) * mine * 16));
      const bool all_in = mbar_wait_cluster(recv_bar, 0, abort_flag, p.status, kDevTimeoutFull);
      if (all_in) {
        for (int g = g0 + et; g < g1; g += 128) {
          float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
          for (int q = 0; q < cs; ++q) {
            const float4 x = (q == rank) ? *reinterpret_cast<const float4*>(red + 4 * g)
                                         : *reinterpret_cast<const float4*>(recv + 4 * (q * per + (g - g0)));
            if (q == 0) {
              s4 = x;
            } else {
              s4.x += x.x;
              s4.y += x.y;
              s4.z += x.z;
              s4.w += x.w;
            }
          }
          const float sum[4] = {s4.x, s4.y, s4.z, s4.w};
          const int col = g / G;
          const int64_t row = static_cast<int64_t>(row0) + 4 * (g % G);
          float* dst = p.C + static_cast<int64_t>(col) * p.ldc + row;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (row + i < p.M) {
              float out = p.alpha * sum[i];
              if (p.beta != 0.f) out = fmaf(p.beta, dst[i], out);
              dst[i] = out;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

template <int MODE>
cudaLaunchConfig_t make_config(const SkParams& p, int grid, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kSkinnyThreads);
  cfg.dynamicSmemBytes = SkCfg<MODE>::SMEM_BYTES;
  cfg.stream = s;
  int n = 0;
  if (p.cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  cfg.attrs = attr;
  cfg.numAttrs = static_cast<unsigned>(n);
  return cfg;
}

template <int MODE, bool A_MN>
cudaError_t set_attributes() {
  static std::atomic<uint64_t> done{0};
  return once_per_device(done, [] {
    auto kern = skinny_gemm_kernel<MODE, A_MN>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SkCfg<MODE>::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
}

template <int MODE, bool A_MN>
cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const SkParams& p, int grid, cudaStream_t s) {
  cudaError_t e = set_attributes<MODE, A_MN>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_config<MODE>(p, grid, s, attr);
  last_main_launch() = LaunchShape{cfg.gridDim, cfg.blockDim, cfg.dynamicSmemBytes, p.cluster, true};
  return cudaLaunchKernelEx(&cfg, skinny_gemm_kernel<MODE, A_MN>, ta, tb, p);
}

template <int MODE, bool A_MN>
int active_clusters(int cluster) {
  if (set_attributes<MODE, A_MN>() != cudaSuccess) return 0;
  SkParams p{};
  p.cluster = cluster;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_config<MODE>(p, cluster, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, skinny_gemm_kernel<MODE, A_MN>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

}  // namespace

cudaError_t skinny_launch(int mode, bool a_mn, const CUtensorMap& ta, const CUtensorMap& tb, const SkParams& p,
                          int grid, cudaStream_t s) {
  if (p.cluster < 1 || p.cluster > kSkinnyMaxCluster || grid % p.cluster != 0 || p.N < 1 || p.N > 16)
    return cudaErrorInvalidValue;
  if (mode == 2) return a_mn ? launch_one<2, true>(ta, tb, p, grid, s) : launch_one<2, false>(ta, tb, p, grid, s);
  if (mode == 1 && !a_mn) return launch_one<1, false>(ta, tb, p, grid, s);
  if (mode == 3 && !a_mn) return launch_one<3, false>(ta, tb, p, grid, s);
  if (mode == 4 && !a_mn) return launch_one<4, false>(ta, tb, p, grid, s);
  if (mode == 5 && !a_mn) return launch_one<5, false>(ta, tb, p, grid, s);
  return cudaErrorInvalidValue;  // kind::tf32 and the 8- and 4-bit forms take K-major operands only
}

int skinny_max_active_clusters(int mode, bool a_mn, int cluster) {
  if (cluster < 1 || cluster > kSkinnyMaxCluster) return 0;
  if (mode == 2) return a_mn ? active_clusters<2, true>(cluster) : active_clusters<2, false>(cluster);
  if (mode == 1 && !a_mn) return active_clusters<1, false>(cluster);
  if (mode == 3 && !a_mn) return active_clusters<3, false>(cluster);
  if (mode == 4 && !a_mn) return active_clusters<4, false>(cluster);
  if (mode == 5 && !a_mn) return active_clusters<5, false>(cluster);
  return 0;
}

}  // namespace dgt
