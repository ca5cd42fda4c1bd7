// tc_kernel.cuh -- the persistent TMA + tcgen05 GEMM kernel (TF32 and BF16).
//
// "bare-metal-bard" (first paragraph) ends its ladder with a tensor-core
// kernel in TF32.  On this part the tensor cores are driven by tcgen05: one
// thread issues asynchronous 128 x N x K MMAs whose operands are read from
// shared memory through descriptors and whose fp32 accumulator lives in TMEM.
// The kernel is organised around that:
//
//   warp 0      TMA producer: fills a ring of shared-memory stages (one A box
//               of 128 rows and one B box of tile_n rows, 128-byte swizzled,
//               128 bytes of K per row) and arms each stage's "full" mbarrier
//               with the bytes it expects;
//   warp 1      allocates TMEM (two accumulators of tile_n fp32 columns), then
//               one lane issues the MMAs of a stage and commits them to the
//               stage's "empty" mbarrier, and commits a finished tile to its
//               accumulator's "full" mbarrier;
//   warps 2-9   epilogue: tcgen05.ld of the accumulator (warp w reads TMEM
//               lanes 32*(w%4)..+31, i.e. those rows of the tile; warps w
//               and w+4 split the tile's columns), the fused alpha/beta
//               update, and the stores; then they release the accumulator
//               so the next tile's MMAs can start.  Two accumulators let the
//               epilogue of tile i overlap the mainloop of tile i+1.  The
//               builds with the fused epilogue (EPI) have twelve epilogue
//               warps, 2-13, three per lane quarter, each group of four
//               taking a third of the tile's columns (128 registers a
//               thread, one stage fewer where their staging needs room).
//   TF32 with an MN-major A (128-column tiles, one CTA): kind::tf32 reads
//               only K-major operands from shared memory, so warps 2-5 read
//               each stage's A tile there (one row of A per lane, down the
//               MN-major rows) and store it into TMEM, whose lanes are the
//               rows the MMA takes A from; warps 6-9 are the epilogue.
//   Block-scaled builds (MXFP8 / NVFP4, the swapped small-M form): warp 10
//               copies each stage's scale atoms into the stage's TMEM slot
//               with tcgen05.cp once its data has arrived, and the MMA lane
//               waits for that; the activations' atoms, the same for every
//               weight tile, are copied once per CTA when they fit.  A lane
//               issuing both the copies and the MMAs paced the stages.
//
// Work units are tiles, or (tile, K slice) pairs, handed out round-robin to
// a persistent grid of one CTA per SM (or one CTA pair per two SMs, see PAIR
// below), in a grouped raster order (group_m tiles of M walk all
// tiles of N) so that CTAs running at the same time share A and B tiles in
// L2.  Whole tiles come first; the last rows of tiles may be cut into K
// slices to fill the final wave (or every tile, for plain split-K), and each
// such unit writes raw partial sums to the workspace, which a separate kernel
// reduces in a fixed slice order.  The kernel waits for the previous kernel
// in the stream (programmatic dependent launch) only after its set-up.
//
// Every mbarrier wait is bounded (ptx.cuh); on a timeout the CTA records the
// cause in the device status word, waits (bounded) for its own copies and
// MMAs in flight, frees its TMEM and returns.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "epilogue.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dgt {

// Work units.  Rows of units below tail_tm0 are whole tiles (dp_units of
// them, full K, written to C); the rows from tail_tm0 on are cut into
// `splits` K slices of kb_per_split blocks each, and with more than one
// slice each unit writes raw partial sums to the workspace (C rows from
// ws_row0 on, one M x N slab per slice) for the slice-reduce kernel.
// tail_tm0 = 0 cuts every tile (plain split-K, or no split with splits = 1).
struct TcParams {
  int M, N, K;
  int num_tm, num_tn, num_kb;  // num_tm counts rows of units (pairs of tile rows for PAIR)
  int splits, kb_per_split, num_units, group_m;
  int dp_units, tail_tm0;
  float alpha, beta;
  float* C;
  int64_t ldc;
  float* ws;
  int64_t ws_ld;
  int64_t ws_slice;  // elements between the partial sums of successive K slices
  int64_t ws_row0;   // the C row of workspace row 0
  int* status;
  int c_vec;  // C rows are 16-byte aligned (ldc % 4 == 0 and C aligned)
  int c_tma;  // whole tiles leave through shared memory and TMA stores (tmC is valid)
  int w_tma;  // partial tiles likewise (tmW is valid)
  int z_tma;  // EPI with GELU' and no partial tiles: tmW maps Z, whose 32 x 32 blocks the epilogue loads by TMA
  uint32_t fmt8;  // MODE 3: operand format bits of the instruction descriptor (E4M3 / E5M2)
  EpiParams epi;     // EPI kernels: bias / GELU / GELU' applied at every final store of a whole tile
  const uint8_t* sfa;  // BS: scales of the kernel's A (the weights), tiled 512-byte atoms
  const uint8_t* sfb;  // BS: scales of the kernel's B (the activations)
  int64_t sf_groups;   // BS: atoms per 128-row tile
  int sfb_res;         // BS: the activations' scale atoms held in TMEM for the whole call (their count,
                       // copied once per CTA), or 0: copied with every stage
  uint64_t wait_ns;  // limit of every bounded wait
  int fault_skip;    // test hook: CTA 0's producer issues no copies for its fault_skip-th stage
                     // (0-based; -1: none), so the MMA's wait for that stage runs out
};

// MODE: 1 = tf32 (4-byte operands), 2 = bf16 (2-byte operands), 3 = 8-bit
// floats (E4M3 or E5M2, named at run time in TcParams::fmt8; K-major only).
// BHALF: a
// stage holds one half of the B tile (the two-CTA MMA, where the other CTA
// of the pair holds the other half).
template <int MODE, int BN, bool BHALF = false, int EW_ = kTcEpiWarps>
struct TcCfg {
  static constexpr int EW = EW_;  // epilogue warps (a multiple of 4: one group per TMEM lane quarter)
  static constexpr bool BS = MODE >= 4;  // block-scaled: 4 MXFP8, 5 NVFP4 (swapped small-M form, or 128-column tiles)
  static constexpr int ES = (MODE >= 3) ? 1 : (MODE == 2) ? 2 : 4;  // operand bytes (coordinate units)
  static constexpr int BM = 128;                      // rows of the tile (UMMA M)
  static constexpr int BK = 128 / ES;                 // K units per stage: one 128-byte swizzle row
  static constexpr int UK = 32 / ES;                  // K units of one MMA instruction (32 bytes)
  static constexpr int CH = 128 / ES;                 // M/N elements of one 128-byte MN-major row
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BHALF ? BN * 64 : BN * 128;
  // BS: both operands' scale atoms for the stage's 128 bytes of K (512
  // bytes per 128 rows and 4 scale blocks: 1 atom for MXFP8, 4 for NVFP4)
  static constexpr int SF_ATOMS = (MODE == 5) ? 4 : (MODE == 4) ? 1 : 0;
  static constexpr int SF_BYTES = SF_ATOMS * 512;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + 2 * SF_BYTES;
  // Epilogue staging for TMA stores: one buffer of 32 rows x 128 bytes per
  // epilogue warp (the swapped small-M form stores directly and has none).
  static constexpr int STAGING_BYTES = (BN >= 128) ? EW * 32 * 128 : 0;
  // EPI kernels: one 128-byte slot per epilogue warp for the bias values
  // of the 32 columns it is storing (read back as broadcasts).
  static constexpr int EPI_BYTES = BS ? 0 : EW * 128;
  static constexpr int BAR_BYTES = BS ? 512 : 256;  // barriers, the TMEM address and the abort flag
  // BS, swapped small-M form: up to RES_ATOMS of the activations' scale
  // atoms held in TMEM for the whole call (below), staged through RES_BYTES
  // of shared memory (the 128-column tiles' B scales change with the tile)
  static constexpr int RES_ATOMS = (BS && BN == 16) ? 32 : 0;
  static constexpr int RES_BYTES = RES_ATOMS * 512;
  // as many as fit beside the staging when a stage holds half of B, else
  // the planned count, fewer when the staging of twelve epilogue warps
  // leaves less room
  static constexpr int STAGES_FIT =
      (232448 - STAGING_BYTES - 1024 - BAR_BYTES - RES_BYTES - EPI_BYTES) / STAGE_BYTES;
  static constexpr int STAGES_PLAN = (BN >= 192) ? 4 : (BN == 128) ? 6 : 200 * 1024 / STAGE_BYTES;
  static constexpr int STAGES = BHALF ? STAGES_FIT : (STAGES_PLAN < STAGES_FIT ? STAGES_PLAN : STAGES_FIT);
  // Two accumulators, then (BS) one ring slot of scale columns per stage
  // (4 columns per atom, A's atoms then B's); an allocation is a power of
  // two of at least 32 columns.
  static constexpr int SF_COL0 = 2 * BN;
  static constexpr int SF_COLS = 2 * SF_ATOMS * 4;
  // BS: up to RES_ATOMS of the activations' scale atoms (the same for every
  // weight tile) kept in TMEM for the whole call, after the ring, and
  // staged through RES_BYTES of shared memory after the barriers.
  static constexpr int RES_COL0 = SF_COL0 + (BS ? STAGES * SF_COLS : 0);
  static constexpr int TMEM_NEED = RES_COL0 + 4 * RES_ATOMS;
  static constexpr int TMEM_COLS = (TMEM_NEED <= 32) ? 32 : (TMEM_NEED <= 64) ? 64 : (TMEM_NEED <= 128) ? 128
                                   : (TMEM_NEED <= 256) ? 256 : 512;
  static_assert(TMEM_NEED <= 512, "TMEM columns");
  static_assert(!BS || ((BN == 16 || BN == 128) && !BHALF),
                "block-scaled: the swapped small-M form, or 128-column tiles of one CTA");
  static constexpr int CW = BN < 32 ? BN : 32;                    // accumulator columns per TMEM load
  // full/empty per stage, acc full/empty x2, drain, resident scales; BS
  // also: per stage "scale atoms copied", and the copier's drain
  static constexpr int NUM_BARS = 2 * STAGES + 6 + (BS ? STAGES + 1 : 0);
  // BS builds add a warp that copies every stage's scale atoms into TMEM,
  // so that the MMA thread issues only the MMAs
  static constexpr int THREADS = 32 * (2 + EW) + (BS ? 32 : 0);
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*align*/ + BAR_BYTES + RES_BYTES + EPI_BYTES;
  static_assert(SMEM_BYTES <= 232448, "dynamic shared memory per CTA");
  static constexpr uint32_t FORMAT = (MODE >= 3) ? 0u : (MODE == 2) ? 1u : 2u;  // 8-bit (fmt8) / bf16 / tf32
  static_assert(NUM_BARS * 8 + 16 <= BAR_BYTES, "barrier area");
  static_assert(STAGE_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "stages must keep 1024-byte swizzle atoms aligned");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "UMMA N for M = 128");
  static_assert(BN < 32 || BN % 32 == 0, "the epilogue moves 32-column chunks");
};

template <int MODE, bool PAIR>
__device__ __forceinline__ void issue_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if constexpr (PAIR) {
    if (MODE == 3)
      mma_f8f6f4_pair(d, a, b, idesc, acc);
    else if (MODE == 2)
      mma_bf16_pair(d, a, b, idesc, acc);
    else
      mma_tf32_pair(d, a, b, idesc, acc);
  } else {
    if (MODE == 3)
      mma_f8f6f4(d, a, b, idesc, acc);
    else if (MODE == 2)
      mma_bf16(d, a, b, idesc, acc);
    else
      mma_tf32(d, a, b, idesc, acc);
  }
}

// Bounded wait on a barrier of this CTA; PAIR kernels wait with cluster
// scope (the other CTA of the pair or its MMAs arrive on it).
template <bool CLUSTER>
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status, int code,
                                         uint64_t limit) {
  if constexpr (CLUSTER)
    return mbar_wait_cluster(bar, parity, abort, status, code, limit);
  else
    return mbar_wait(bar, parity, abort, status, code, limit);
}

struct Unit {
  int tm, tn, split, kb0, kb1;
  bool partial;
};

// EPI: the epilogue's inputs for columns col0 .. col0 + 4 * NQ - 1 of one
// row of C (the bias, or Z's row), all requested before any is used so
// that they cost one memory latency; `fetch` is false for a row past M,
// whose values are never stored.
template <int NQ>
__device__ __forceinline__ void epi_fetch(const EpiParams& e, int64_t row, int64_t col0, int64_t n, bool fetch,
                                          float4 (&x)[NQ]) {
#pragma unroll
  for (int q = 0; q < NQ; ++q)
    x[q] = fetch ? epilogue_fetch4(e, row, col0 + 4 * q, n) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// The elementwise epilogue of four consecutive elements, after alpha /
// beta, with the activation fixed at compile time (ACT < 0: none at all).
// Two packed pairs per quad, each element the same as epilogue_finish_t's.
template <int ACT>
__device__ __forceinline__ float4 epi_finish4(float4 v, const float4& x) {
  if constexpr (ACT >= 0) {
    uint64_t lo = f2_pack(v.x, v.y), hi = f2_pack(v.z, v.w);
    const uint64_t xl = f2_pack(x.x, x.y), xh = f2_pack(x.z, x.w);
    if constexpr (ACT == kActDGelu) {
      lo = f2_mul(lo, dgelu_x2(xl));
      hi = f2_mul(hi, dgelu_x2(xh));
    } else {
      lo = f2_add(lo, xl);
      hi = f2_add(hi, xh);
      if constexpr (ACT == kActGelu) {
        lo = gelu_x2(lo);
        hi = gelu_x2(hi);
      }
    }
    f2_unpack(lo, v.x, v.y);
    f2_unpack(hi, v.z, v.w);
  }
  return v;
}

// alpha times four accumulator words plus x (the bias), then GELU or
// nothing (ACT: kActGelu, kActNone): two packed multiply-adds, each element
// rounded once before the activation.
template <int ACT>
__device__ __forceinline__ float4 scaled_bias_act4(float a, const uint32_t* r, const float4& x) {
  const uint64_t a2 = f2_pack(a, a);
  uint64_t lo = f2_fma(a2, f2_pack(__uint_as_float(r[0]), __uint_as_float(r[1])), f2_pack(x.x, x.y));
  uint64_t hi = f2_fma(a2, f2_pack(__uint_as_float(r[2]), __uint_as_float(r[3])), f2_pack(x.z, x.w));
  if constexpr (ACT == kActGelu) {
    lo = gelu_x2(lo);
    hi = gelu_x2(hi);
  }
  float4 v;
  f2_unpack(lo, v.x, v.y);
  f2_unpack(hi, v.z, v.w);
  return v;
}

// alpha times four accumulator words, as two packed products.
__device__ __forceinline__ float4 scaled4(float a, const uint32_t* r) {
  const uint64_t a2 = f2_pack(a, a);
  float4 v;
  f2_unpack(f2_mul(a2, f2_pack(__uint_as_float(r[0]), __uint_as_float(r[1]))), v.x, v.y);
  f2_unpack(f2_mul(a2, f2_pack(__uint_as_float(r[2]), __uint_as_float(r[3]))), v.z, v.w);
  return v;
}

// Calls body(std::integral_constant<int, ACT>) with the epilogue's
// activation as a compile-time value (-1 when there is none to apply), so
// that loops over a chunk carry no per-element test of it.
template <bool EPI, typename F>
__device__ __forceinline__ void with_activation(bool on, int act, F&& body) {
  if constexpr (EPI) {
    if (on) {
      if (act == kActGelu)
        body(std::integral_constant<int, kActGelu>{});
      else if (act == kActDGelu)
        body(std::integral_constant<int, kActDGelu>{});
      else
        body(std::integral_constant<int, kActNone>{});
      return;
    }
  }
  body(std::integral_constant<int, -1>{});
}

// Tile t of a region of `rows` unit rows starting at row0, in the grouped
// raster order: group_m rows walk all columns, so units that run at the
// same time share A and B tiles in L2.
__device__ __forceinline__ void raster(int t, int row0, int rows, const TcParams& p, Unit& w) {
  const int span = p.group_m * p.num_tn;
  const int g = t / span;
  const int first_m = g * p.group_m;
  const int rem = rows - first_m;
  const int gm = rem < p.group_m ? rem : p.group_m;
  const int r = t % span;
  w.tm = row0 + first_m + r % gm;
  w.tn = r / gm;
}

__device__ __forceinline__ Unit decode_unit(int u, const TcParams& p) {
  Unit w;
  if (u < p.dp_units) {
    raster(u, 0, p.tail_tm0, p, w);
    w.split = 0;
    w.kb0 = 0;
    w.kb1 = p.num_kb;
    w.partial = false;
    return w;
  }
  const int v = u - p.dp_units;
  const int rows = p.num_tm - p.tail_tm0;
  const int tiles = rows * p.num_tn;
  raster(v % tiles, p.tail_tm0, rows, p, w);
  w.split = v / tiles;
  w.kb0 = w.split * p.kb_per_split;
  const int e = w.kb0 + p.kb_per_split;
  w.kb1 = e < p.num_kb ? e : p.num_kb;
  w.partial = p.splits > 1;
  return w;
}

// TRANS_C: the kernel computes C^T = op(B)^T op(A)^T with the operands
// swapped by the host (a small-M product whose weights fill the 128-row MMA
// side), so element (r, c) of its tile is stored at C[c * ldc + r].
// PAIR: the grid is made of two-CTA clusters that work on vertically
// adjacent tiles (same columns), and the pair issues one MMA of 256 rows
// (tcgen05 cta_group::2): each CTA loads its own 128 rows of A and its own
// half of B (BN / 2 rows) into its own shared memory, and counts the bytes
// on the even CTA's "full" barrier; one thread of the even CTA issues the
// MMAs, which read A and B from both CTAs and write each CTA's 128 rows of
// the accumulator into that CTA's TMEM, and commits to both CTAs'
// barriers; both CTAs' epilogue warps release an accumulator on the even
// CTA's barrier.  Each CTA then stages 32 KB per 256-column stage instead of
// 48.  Every copy a CTA issues lands in its own shared memory: no operand
// tile is multicast.
// EPI: whole tiles get the elementwise epilogue of p.epi (bias, GELU, GELU'
// of a kept pre-activation) in the epilogue warps, between the TMEM load
// and the store; partial tiles of a K split stay raw for the slice reduce,
// which applies it.
template <int MODE, bool A_MN, bool B_MN, int BN, bool TRANS_C, bool PAIR, bool EPI = false>
__global__ void __launch_bounds__(TcCfg<MODE, BN, PAIR, EPI ? kTcEpiWarpsEpi : kTcEpiWarps>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmW,
                   const TcParams p) {
  static_assert(!EPI || !TRANS_C, "the swapped small-M form applies no epilogue itself");
  using Cfg = TcCfg<MODE, BN, PAIR, EPI ? kTcEpiWarpsEpi : kTcEpiWarps>;
  constexpr int S = Cfg::STAGES;
  // TF32 with an MN-major A: kind::tf32 reads only K-major operands from
  // shared memory, so warps 2-5 move each stage's A tile into TMEM (row i of
  // the tile in lane i, K along the columns), where the MMA takes A from;
  // warps 6-9 are the epilogue.  A ring of NA buffers of BK columns sits
  // after the two accumulators.
  constexpr bool A_TMEM = MODE == 1 && A_MN;
  static_assert(!A_TMEM || (BN == 128 && !PAIR && !TRANS_C), "A through TMEM: 128-column tiles, one CTA");
  constexpr int NA = 4;
  constexpr int A_COL0 = 2 * BN;  // first TMEM column of the A buffers
  constexpr int TMEM_COLS = A_TMEM ? 512 : Cfg::TMEM_COLS;
  constexpr int EXTRA_BARS = A_TMEM ? 2 * NA : 0;
  static_assert((Cfg::NUM_BARS + EXTRA_BARS) * 8 + 16 <= Cfg::BAR_BYTES, "barrier area");
  static_assert(!A_TMEM || A_COL0 + NA * Cfg::BK <= TMEM_COLS, "TMEM columns");
  // MODE 3 names its operand formats at run time (the FORMAT fields are 0).
  const uint32_t IDESC = make_idesc(Cfg::FORMAT, A_MN && !A_TMEM, B_MN, PAIR ? 2 * Cfg::BM : Cfg::BM, BN) |
                         (MODE == 3 ? p.fmt8 : 0u);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + S * Cfg::STAGE_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + Cfg::STAGING_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::NUM_BARS + EXTRA_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  [[maybe_unused]] float* bias_slots =
      reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + Cfg::BAR_BYTES + Cfg::RES_BYTES);

  const uint32_t smem0 = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto accf_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto acce_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  // BS: the activations' scale atoms for the whole call land here (one
  // bulk copy, completing on res_bar) before they are copied into TMEM
  const uint32_t res_bar = bar0 + 8u * (2 * S + 5);
  [[maybe_unused]] const uint32_t res_smem = bar0 + static_cast<uint32_t>(Cfg::BAR_BYTES);
  // BS: stage s's scale atoms are in TMEM (the copier warp commits it)
  auto cpd_bar = [&](int st) { return bar0 + 8u * (2 * S + 6 + st); };
  [[maybe_unused]] const uint32_t cdrain_bar = bar0 + 8u * (3 * S + 6);
  auto afull_bar = [&](int b) { return bar0 + 8u * (Cfg::NUM_BARS + b); };        // A_TMEM: A in TMEM
  auto aempty_bar = [&](int b) { return bar0 + 8u * (Cfg::NUM_BARS + NA + b); };  // A_TMEM: buffer read

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  static_assert(!PAIR || (!TRANS_C && BN >= 128 && (!B_MN || (BN / Cfg::CH) % 2 == 0)),
                "paired CTAs each load one half of the B tile");
  // Work units: one per CTA, or one per two-CTA cluster (the pair's rank
  // picks its row of tiles).  The cluster of a pair is blockIdx.x / 2.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0u;  // PAIR: the CTA that issues the pair's MMAs
  const int unit0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int unit_step = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  auto tile_row = [&](const Unit& w) { return PAIR ? 2 * w.tm + static_cast<int>(rank) : w.tm; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      // the stage is free once its MMAs (PAIR: the one pair MMA) have read
      // it; A_TMEM: the MMAs (B) and the four warps that read A
      mbar_init(empty_bar(s), A_TMEM ? 5 : 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      // one arrival per epilogue warp (of both CTAs)
      mbar_init(acce_bar(a), A_TMEM ? 4 : PAIR ? 2 * Cfg::EW : Cfg::EW);
    }
    for (int b = 0; b < (A_TMEM ? NA : 0); ++b) {
      mbar_init(afull_bar(b), 4);
      mbar_init(aempty_bar(b), 1);
    }
    mbar_init(drain_bar, 1);
    mbar_init(res_bar, 1);
    if constexpr (Cfg::BS) {
      for (int st = 0; st < S; ++st) mbar_init(cpd_bar(st), 1);
      mbar_init(cdrain_bar, 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.c_tma) tma_prefetch_desc(&tmC);
    if (p.w_tma) tma_prefetch_desc(&tmW);
    if (p.z_tma) tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), Cfg::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // PAIR: the peer's barriers must be initialised before its copies or the
  // pair's MMA commits can signal them.
  if constexpr (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Set-up above touches no global memory; from here on the kernel reads
  // what earlier kernels in the stream wrote.
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // stages taken so far (their positions in the ring's sequence)
      if constexpr (Cfg::BS) {
        if (p.sfb_res > 0) {
          mbar_arrive_expect_tx(res_bar, static_cast<uint32_t>(p.sfb_res) * 512u);
          bulk_copy_g2s(res_smem, p.sfb, static_cast<uint32_t>(p.sfb_res) * 512u, res_bar);
        }
      }
      bool ok = true;
      // The test hook's position (CTA 0 only): its stage is taken but gets
      // no copies, so its "full" barrier never completes.
      const uint32_t skip = (blockIdx.x == 0 && p.fault_skip >= 0) ? static_cast<uint32_t>(p.fault_skip) : ~0u;
      for (int u = unit0; u < p.num_units && ok; u += unit_step) {
        const Unit w = decode_unit(u, p);
        const int tm = tile_row(w);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!bar_wait<PAIR>(empty_bar(stage), phase ^ 1u, abort_flag, p.status, kDevTimeoutEmpty, p.wait_ns)) {
            ok = false;
            break;
          }
          if (issued == skip) {
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          const uint32_t a_dst = smem0 + stage * Cfg::STAGE_BYTES;
          const uint32_t b_dst = a_dst + Cfg::A_BYTES;
          const int k0 = kb * Cfg::BK;
          if constexpr (PAIR) {
            // Both CTAs' copies are counted on the even CTA's barrier, which
            // expects the bytes of the two (a copy of the odd CTA may land
            // before that expectation: the barrier's phase cannot complete
            // until the even CTA has arrived).
            const uint32_t fb = dsmem_map(full_bar(stage), 0);
            if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * Cfg::STAGE_BYTES);
            if (A_MN) {
#pragma unroll
              for (int c = 0; c < Cfg::BM / Cfg::CH; ++c)
                tma_load_2d_pair(a_dst + c * Cfg::BK * 128, &tmA, fb, tm * Cfg::BM + c * Cfg::CH, k0);
            } else {
              tma_load_2d_pair(a_dst, &tmA, fb, k0, tm * Cfg::BM);
            }
            if (B_MN) {
              constexpr int NH = BN / Cfg::CH / 2;  // this CTA's 128-byte column chunks of B
#pragma unroll
              for (int c = 0; c < NH; ++c)
                tma_load_2d_pair(b_dst + c * Cfg::BK * 128, &tmB, fb,
                                 w.tn * BN + (static_cast<int>(rank) * NH + c) * Cfg::CH, k0);
            } else {
              tma_load_2d_pair(b_dst, &tmB, fb, k0, w.tn * BN + static_cast<int>(rank) * (BN / 2));
            }
          } else {
            const uint32_t fb = full_bar(stage);
            mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES - ((Cfg::BS && p.sfb_res > 0) ? Cfg::SF_BYTES : 0));
            if (A_MN) {
#pragma unroll
              for (int c = 0; c < Cfg::BM / Cfg::CH; ++c)
                tma_load_2d(a_dst + c * Cfg::BK * 128, &tmA, fb, tm * Cfg::BM + c * Cfg::CH, k0);
            } else {
              tma_load_2d(a_dst, &tmA, fb, k0, tm * Cfg::BM);
            }
            if (B_MN) {
#pragma unroll
              for (int c = 0; c < BN / Cfg::CH; ++c)
                tma_load_2d(b_dst + c * Cfg::BK * 128, &tmB, fb, w.tn * BN + c * Cfg::CH, k0);
            } else {
              tma_load_2d(b_dst, &tmB, fb, k0, w.tn * BN);
            }
            if constexpr (Cfg::BS) {
              // both operands' scale atoms for this stage (the swapped form's
              // B: the activations, one row tile; 128-column tiles: B's tile
              // w.tn of 128 rows)
              const uint32_t sf_dst = b_dst + Cfg::B_BYTES;
              bulk_copy_g2s(sf_dst, p.sfa + (static_cast<int64_t>(tm) * p.sf_groups + kb * Cfg::SF_ATOMS) * 512,
                            Cfg::SF_BYTES, fb);
              if (p.sfb_res == 0)
                bulk_copy_g2s(sf_dst + Cfg::SF_BYTES,
                              p.sfb + (static_cast<int64_t>(TRANS_C ? 0 : w.tn) * p.sf_groups + kb * Cfg::SF_ATOMS) * 512,
                              Cfg::SF_BYTES, fb);
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!PAIR || leader) {
        // Every copy still in flight lands before the CTA can exit.  Normally
        // the MMAs have waited for all of them already and this returns at
        // once; but when the MMA warp gave up a wait, the copies issued after
        // the stage it waited for are waited for here, whether or not this
        // loop ran to its end.  (An odd CTA's copies complete on the even
        // CTA's barriers, whose drain covers them; the pair leaves together.)
        if constexpr (Cfg::BS) {
          if (p.sfb_res > 0) drain_wait(res_bar, 0, p.status, p.wait_ns);
        }
        const uint32_t n = issued < static_cast<uint32_t>(S) ? issued : static_cast<uint32_t>(S);
        for (uint32_t i = issued - n; i < issued; ++i)
          if (i != skip) drain_wait(full_bar(i % S), (i / S) & 1u, p.status, p.wait_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // PAIR: only the even CTA of the pair issues (its MMAs cover both CTAs).
    if (lane == 0 && (!PAIR || leader)) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int ab = 0;  // A_TMEM: buffer of the next stage's A
      uint32_t a_phase = 0;
      bool ok = true;
      // block-scaled builds: stage 0's operand and scale-atom descriptors
      [[maybe_unused]] const uint64_t a_desc0 = smem_desc_sw128(smem0, 16, 1024);
      [[maybe_unused]] const uint64_t b_desc0 = smem_desc_sw128(smem0 + Cfg::A_BYTES, 16, 1024);
      [[maybe_unused]] const uint64_t sf_desc0 = smem_desc_noswizzle(smem0 + Cfg::A_BYTES + Cfg::B_BYTES, 128);
      [[maybe_unused]] const uint32_t res_col = tmem_base + static_cast<uint32_t>(Cfg::RES_COL0);
      if constexpr (Cfg::BS) {
        // The activations' scale atoms for the whole call into TMEM once:
        // atom a (stage a / SF_ATOMS, block group a % SF_ATOMS) at columns
        // res_col + 4 a.  The MMAs issued after these copies by this thread
        // see them (tcgen05 operations of one thread run in issue order).
        if (p.sfb_res > 0) {
          if (!bar_wait<false>(res_bar, 0, abort_flag, p.status, kDevTimeoutFull, p.wait_ns)) {
            ok = false;
          } else {
            tc_fence_after();
            const uint64_t rd0 = smem_desc_noswizzle(res_smem, 128);
            for (int a = 0; a < p.sfb_res; ++a) tmem_cp_32x128b_x4(res_col + 4 * a, rd0 + 32 * a);
          }
        }
      }
      for (int u = unit0; u < p.num_units && ok; u += unit_step) {
        const Unit w = decode_unit(u, p);
        if (!bar_wait<PAIR>(acce_bar(acc), acc_phase ^ 1u, abort_flag, p.status, kDevTimeoutAccEmpty, p.wait_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          // The stage's data; BS: also its scale atoms, which the copier
          // warp puts into TMEM after the data arrived (so the second wait
          // is the one that lasts)
          if (!bar_wait<PAIR>(full_bar(stage), phase, abort_flag, p.status, kDevTimeoutFull, p.wait_ns) ||
              (Cfg::BS && !bar_wait<false>(cpd_bar(stage), phase, abort_flag, p.status, kDevTimeoutFull, p.wait_ns))) {
            ok = false;
            break;
          }
          if constexpr (A_TMEM) {
            if (!bar_wait<false>(afull_bar(ab), a_phase, abort_flag, p.status, kDevTimeoutFull, p.wait_ns)) {
              ok = false;
              break;
            }
          }
          tc_fence_after();
          const uint32_t a_base = smem0 + stage * Cfg::STAGE_BYTES;
          const uint32_t b_base = a_base + Cfg::A_BYTES;
          if constexpr (Cfg::BS) {
            // Four block-scaled MMAs of 32 bytes of K, the stage's scale
            // atoms already in its TMEM ring slot (the copier warp's): MXFP8
            // picks its byte of the scale cells by ID j, NVFP4 reads atom
            // j's four bytes.
            // The descriptors are stage 0's plus the stage's byte offset in
            // their address field (bits 0-13, address >> 4; every shared
            // address here is below 256 KB, so the field cannot carry): a
            // single issuing thread rebuilding 64-bit descriptors between
            // these small instructions is what would pace them.
            const uint32_t sf_col = tmem_base + static_cast<uint32_t>(Cfg::SF_COL0 + stage * Cfg::SF_COLS);
            const uint64_t soff = static_cast<uint64_t>((stage * Cfg::STAGE_BYTES) >> 4);
            const bool res = p.sfb_res > 0;
            // B's atoms of this stage: in the resident area, or in the slot
            const uint32_t sfb_col = res ? res_col + static_cast<uint32_t>(4 * Cfg::SF_ATOMS * kb)
                                         : sf_col + static_cast<uint32_t>(4 * Cfg::SF_ATOMS);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t ad = a_desc0 + soff + 2 * j;
              const uint64_t bd = b_desc0 + soff + 2 * j;
              const uint32_t acc_in = (kb > w.kb0 || j > 0) ? 1u : 0u;
              if constexpr (MODE == 4)
                mma_mxf8f6f4_bs(d_tmem, ad, bd,
                                make_idesc_bs(0, 0, true, Cfg::BM, BN, static_cast<uint32_t>(j),
                                              static_cast<uint32_t>(j)) | p.fmt8,
                                sf_col, sfb_col, acc_in);
              else
                mma_mxf4nvf4_bs(d_tmem, ad, bd, make_idesc_bs(1, 1, false, Cfg::BM, BN, 0, 0), sf_col + 4 * j,
                                sfb_col + 4 * j, acc_in);
            }
          } else {
#pragma unroll
            for (int j = 0; j < Cfg::BK / Cfg::UK; ++j) {
              const uint64_t bd = B_MN ? smem_desc_sw128(b_base + j * Cfg::UK * 128, Cfg::BK * 128, 1024)
                                       : smem_desc_sw128(b_base + j * Cfg::UK * Cfg::ES, 16, 1024);
              if constexpr (A_TMEM) {
                mma_tf32_tmem_a(d_tmem, tmem_base + static_cast<uint32_t>(A_COL0 + ab * Cfg::BK + j * Cfg::UK), bd,
                                IDESC, (kb > w.kb0 || j > 0) ? 1u : 0u);
              } else {
                const uint64_t ad = A_MN ? smem_desc_sw128(a_base + j * Cfg::UK * 128, Cfg::BK * 128, 1024)
                                         : smem_desc_sw128(a_base + j * Cfg::UK * Cfg::ES, 16, 1024);
                issue_mma<MODE, PAIR>(d_tmem, ad, bd, IDESC, (kb > w.kb0 || j > 0) ? 1u : 0u);
              }
            }
          }
          if constexpr (A_TMEM) {
            mma_commit(aempty_bar(ab));  // the A buffer is free once these MMAs are done
            if (++ab == NA) {
              ab = 0;
              a_phase ^= 1u;
            }
          }
          if constexpr (PAIR)
            mma_commit_pair_multicast(empty_bar(stage), 0x3);  // both CTAs' halves of the stage are free
          else
            mma_commit(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          mma_commit_pair_multicast(accf_bar(acc), 0x3);  // each CTA's 128 rows are ready in its TMEM
        else
          mma_commit(accf_bar(acc));
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Every MMA this thread issued has finished once drain_bar flips.
      if constexpr (PAIR)
        mma_commit_pair(drain_bar);
      else
        mma_commit(drain_bar);
      drain_wait(drain_bar, 0, p.status, p.wait_ns);
    }
  } else if (Cfg::BS && warp == 2 + Cfg::EW) {
    // ------------------------------------------------------------ scale copier
    // BS builds: one lane walks the stages in the MMA thread's order and
    // copies each stage's scale atoms (the weights'; the activations' too
    // unless they are resident) into the stage's TMEM ring slot once its
    // data has arrived, then commits cpd_bar(stage).  The slot is free: the
    // stage was refilled only after the MMAs that read it released it.
    if constexpr (Cfg::BS) {
      if (lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        const uint64_t sf_desc0 = smem_desc_noswizzle(smem0 + Cfg::A_BYTES + Cfg::B_BYTES, 128);
        const int atoms = p.sfb_res > 0 ? Cfg::SF_ATOMS : 2 * Cfg::SF_ATOMS;
        for (int u = unit0; u < p.num_units && ok; u += unit_step) {
          const Unit w = decode_unit(u, p);
          for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!bar_wait<false>(full_bar(stage), phase, abort_flag, p.status, kDevTimeoutFull, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sf_col = tmem_base + static_cast<uint32_t>(Cfg::SF_COL0 + stage * Cfg::SF_COLS);
            const uint64_t soff = static_cast<uint64_t>((stage * Cfg::STAGE_BYTES) >> 4);
            for (int a = 0; a < atoms; ++a) tmem_cp_32x128b_x4(sf_col + 4 * a, sf_desc0 + soff + 32 * a);
            mma_commit(cpd_bar(stage));
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        // every copy this thread issued has finished once cdrain_bar flips
        mma_commit(cdrain_bar);
        drain_wait(cdrain_bar, 0, p.status, p.wait_ns);
      }
    }
  } else if (A_TMEM && warp < 6) {
    // ------------------------------------------------------------ A into TMEM
    // Warp w moves rows 32q..32q+31 (q = w % 4, the TMEM lane quarter it may
    // access) of each stage's A tile: lane l reads its row's BK values down
    // the MN-major tile -- 128-byte chunk q of the stage, K row k at k * 128
    // bytes, 16-byte unit (l / 4) ^ (k % 8), element l % 4: one conflict-free
    // access of the warp per k -- and stores them as BK columns of lane 32q + l.
    if constexpr (A_TMEM) {
      const int q = warp & 3;
      int stage = 0, ab = 0;
      uint32_t phase = 0, a_phase = 0;
      bool ok = true;
      for (int u = unit0; u < p.num_units && ok; u += unit_step) {
        const Unit w = decode_unit(u, p);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!bar_wait<false>(full_bar(stage), phase, abort_flag, p.status, kDevTimeoutFull, p.wait_ns) ||
              !bar_wait<false>(aempty_bar(ab), a_phase ^ 1u, abort_flag, p.status, kDevTimeoutEmpty, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* a_s = smem + stage * Cfg::STAGE_BYTES + q * (Cfg::BK * 128);
          uint32_t v[Cfg::BK];
#pragma unroll
          for (int k = 0; k < Cfg::BK; ++k)
            v[k] = *reinterpret_cast<const uint32_t*>(a_s + k * 128 + ((((lane >> 2) ^ (k & 7))) << 4) + (lane & 3) * 4);
          __syncwarp();
          tmem_st_32x32b_x32(tmem_base + (static_cast<uint32_t>(32 * q) << 16) +
                                 static_cast<uint32_t>(A_COL0 + ab * Cfg::BK),
                             v);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(afull_bar(ab));
            mbar_arrive(empty_bar(stage));  // this warp's reads of the stage are done
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
          if (++ab == NA) {
            ab = 0;
            a_phase ^= 1u;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // The epilogue's loop is built twice: with ZT (GELU' whose Z comes in
    // by TMA, chosen when the call allows it) and without, so that the
    // other epilogues carry none of its code.
    auto epilogue_role = [&](auto zt_c) {
      constexpr bool ZT = decltype(zt_c)::value;
      const int sub = warp & 3;          // TMEM lane quarter this warp may access
      const int group = (warp - 2) >> 2;  // which group of the tile's column chunks it stores
      int acc = 0;
      uint32_t acc_phase = 0;
      constexpr int CW = Cfg::CW;
      constexpr int NCH = BN / CW;  // column chunks of a tile
      // The EW / 4 groups of warps take consecutive runs of chunks, the
      // first NCH % groups runs one chunk longer (A_TMEM: the four epilogue
      // warps take all of them).
      constexpr int NG = A_TMEM ? 1 : Cfg::EW / 4;
      const int g = A_TMEM ? 0 : group;
      const int cc_begin = g * (NCH / NG) + (g < NCH % NG ? g : NCH % NG);
      const int cc_end = cc_begin + NCH / NG + (g < NCH % NG ? 1 : 0);
      // EPI with a bias (or no input at all): lane l holds the bias of column
      // l of the warp's next chunk, loaded one chunk ahead; at the chunk's
      // start the warp puts its 32 values into its shared-memory slot, and
      // every lane reads them back four at a time as broadcasts.
      [[maybe_unused]] const bool bias_slot = EPI && p.epi.act != kActDGelu;
      [[maybe_unused]] float* const bslot = bias_slots + (warp - 2) * 32;
      [[maybe_unused]] auto bias_of = [&](int64_t col) {
        return (p.epi.bias != nullptr && col < p.N) ? ld_nc_f32_here(p.epi.bias + col) : 0.f;
      };
      [[maybe_unused]] float bias_next = 0.f;
      // EPI with GELU' and Z readable by TMA: each chunk's 32 x 32 block of Z
      // is loaded into the warp's staging buffer, in the layout the chunk's
      // result takes there, and the result overwrites it in place; the block
      // of the warp's next chunk is pulled into L2 one chunk ahead.  The
      // warp's bias slot (unused with GELU') holds the loads' barrier (its
      // first 8 bytes), the barrier's phase (bit 0 of the next word) and
      // whether a load was left unobserved (bit 1), so that the GELU kernels
      // carry no extra registers through their loops.
      [[maybe_unused]] const uint32_t z_bar = smem_u32(bslot);
      [[maybe_unused]] volatile uint32_t* const z_word = reinterpret_cast<volatile uint32_t*>(bslot) + 2;
      if constexpr (EPI) {
        if (ZT && lane == 0) {
          mbar_init(z_bar, 1);
          fence_barrier_init();
          fence_proxy_async_smem();
          *z_word = 0u;
          if (unit0 < p.num_units) {
            const Unit w0 = decode_unit(unit0, p);
            tma_prefetch_l2_3d(&tmW, w0.tn * BN + cc_begin * CW, tile_row(w0) * Cfg::BM + sub * 32, 0);
          }
        }
        __syncwarp();
      }
      if constexpr (EPI) {
        if (bias_slot && unit0 < p.num_units)
          bias_next = bias_of(static_cast<int64_t>(decode_unit(unit0, p).tn) * BN + cc_begin * CW + lane);
      }
      for (int u = unit0; u < p.num_units; u += unit_step) {
        const Unit w = decode_unit(u, p);
        if (!bar_wait<PAIR>(accf_bar(acc), acc_phase, abort_flag, p.status, kDevTimeoutAccFull, p.wait_ns)) break;
        tc_fence_after();
        const bool partial = w.partial;
        const bool read_c = !partial && p.beta != 0.f;
        const int tm = tile_row(w);
        const int64_t row = static_cast<int64_t>(tm) * Cfg::BM + sub * 32 + lane;
        const bool row_ok = row < p.M;
        const int64_t row_base = partial ? p.ws_row0 : 0;  // C row of row 0 of the destination
        const int64_t wrow = row - row_base;
        float* base = partial ? p.ws + static_cast<int64_t>(w.split) * p.ws_slice : p.C;
        const int64_t ld = partial ? p.ws_ld : p.ldc;
        float* out = TRANS_C ? base : base + (row_ok ? wrow : 0) * ld;
        const bool vec_ok = !TRANS_C && (partial || p.c_vec);
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(sub * 32) << 16) + static_cast<uint32_t>(acc * BN);
  #pragma unroll 1
        for (int cc = cc_begin; cc < cc_end; ++cc) {
          const int64_t col0 = static_cast<int64_t>(w.tn) * BN + cc * CW;
          // EPI with GELU': Z's values for this row in the chunk's first
          // quarter, requested before the TMEM load so that both latencies
          // overlap; each further quarter is requested as a group when the
          // previous one is done (fetching more at once spilled registers).
          constexpr int NQH = (CW / 4 + 3) / 4;
          const bool epi_on = EPI && !partial;
          const bool epi_fetch_ok = row_ok && col0 < p.N;
          float4 xe[NQH];
          if constexpr (EPI) {
            if (epi_on && !bias_slot && !ZT) epi_fetch<NQH>(p.epi, row, col0, p.N, epi_fetch_ok, xe);
            if (bias_slot) {
              __syncwarp();  // every lane has read the slot's previous values
              bslot[lane] = bias_next;
              __syncwarp();
              // the next chunk of this warp: the next one of this tile, or the
              // first of its next unit's tile
              int64_t ncol = -1;
              if (cc + 1 < cc_end)
                ncol = col0 + CW + lane;
              else if (u + unit_step < p.num_units)
                ncol = static_cast<int64_t>(decode_unit(u + unit_step, p).tn) * BN + cc_begin * CW + lane;
              bias_next = ncol >= 0 ? bias_of(ncol) : 0.f;
            } else if (ZT && lane == 0) {
              // the same next chunk's block of Z into L2
              if (cc + 1 < cc_end) {
                if (col0 + CW < p.N)
                  tma_prefetch_l2_3d(&tmW, static_cast<int32_t>(col0 + CW), tm * Cfg::BM + sub * 32, 0);
              } else if (u + unit_step < p.num_units) {
                const Unit nw = decode_unit(u + unit_step, p);
                tma_prefetch_l2_3d(&tmW, nw.tn * BN + cc_begin * CW, tile_row(nw) * Cfg::BM + sub * 32, 0);
              }
            }
          }
          if constexpr (Cfg::STAGING_BYTES > 0 && CW == 32) {
            if (partial ? p.w_tma : p.c_tma) {
              // Through shared memory: this warp's 32 rows x 32 columns go to
              // one of its two 4 KB buffers in the 128-byte-swizzled layout the
              // TMA unit reads (16-byte chunk j of row t sits at chunk j ^ (t % 8)),
              // then one lane stores the box; the unit clips rows past M and
              // columns past N.
              uint8_t* buf = staging + (warp - 2) * 4096;
              if (lane == 0) bulk_wait_group_read<0>();  // the buffer's previous store has read it
              __syncwarp();
              [[maybe_unused]] const bool zt = epi_on && ZT;
              [[maybe_unused]] bool z_fail = false;
              const float a = partial ? 1.f : p.alpha;
              // EPI kernels read the chunk from TMEM in two halves of 16
              // columns (fewer live registers beside the epilogue's inputs).
              constexpr int SW = EPI ? 16 : CW;
              with_activation<EPI>(epi_on, p.epi.act, [&](auto act_c) {
                constexpr int ACT = decltype(act_c)::value;
                if constexpr (ACT == kActDGelu) {
                  if (zt && lane == 0) {
                    mbar_arrive_expect_tx(z_bar, 4096u);
                    tma_load_3d(smem_u32(buf), &tmW, z_bar, static_cast<int32_t>(col0),
                                static_cast<int32_t>(tm * Cfg::BM + sub * 32), 0);
                  }
                }
  #pragma unroll
                for (int hh = 0; hh < CW / SW; ++hh) {
                  uint32_t r[SW];
                  __syncwarp();
                  tmem_ld_32x32b<SW>(t_row + cc * CW + hh * SW, r);
                  tmem_wait_ld();
                  if constexpr (ACT == kActDGelu) {
                    if (zt && hh == 0) {
                      // the warp decides together, so that a wait that gave up
                      // takes every lane out of the loop at the same point
                      const uint32_t par = *z_word & 1u;
                      const bool ok =
                          mbar_wait(z_bar, par, abort_flag, p.status, kDevTimeoutEpiInput, p.wait_ns);
                      z_fail = !__all_sync(0xffffffffu, ok);
                      if (lane == 0) *z_word = z_fail ? (par | 2u) : (par ^ 1u);
                    }
                  }
  #pragma unroll
                  for (int qq = 0; qq < SW / 4; ++qq) {
                    const int q = hh * (SW / 4) + qq;
                    float4* const slot = reinterpret_cast<float4*>(buf + lane * 128 + ((q ^ (lane & 7)) * 16));
                    float4 v;
                    if constexpr (ACT == kActDGelu) {
                      if (zt) {
                        v = epi_finish4<ACT>(scaled4(a, r + 4 * qq), *slot);
                      } else {
                        if (q > 0 && q % NQH == 0) epi_fetch<NQH>(p.epi, row, col0 + 4 * q, p.N, epi_fetch_ok, xe);
                        v = epi_finish4<ACT>(scaled4(a, r + 4 * qq), xe[q % NQH]);
                      }
                    } else if constexpr (ACT >= 0) {
                      v = scaled_bias_act4<ACT>(a, r + 4 * qq, reinterpret_cast<const float4*>(bslot)[q]);
                    } else {
                      v = scaled4(a, r + 4 * qq);
                    }
                    *slot = v;
                  }
                }
              });
              if constexpr (EPI) {
                if (z_fail) break;  // the run is being abandoned (status set); Z's load is drained below
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(partial ? &tmW : &tmC, smem_u32(buf), static_cast<int32_t>(col0),
                             static_cast<int32_t>(tm * Cfg::BM + sub * 32 - row_base), partial ? w.split : 0);
                bulk_commit_group();
              }
              continue;
            }
          }
          // the whole chunk from TMEM, by every lane (a warp-collective load)
          uint32_t r[CW];
          __syncwarp();
          tmem_ld_32x32b<CW>(t_row + cc * CW, r);
          tmem_wait_ld();
          if (!row_ok || col0 >= p.N) {
            // nothing of this chunk is inside C for this thread
          } else if (vec_ok && col0 + CW <= p.N) {
            float4* dst = reinterpret_cast<float4*>(out + col0);
            // All of the chunk's loads of C are issued before any store, so
            // their latencies overlap (EPI kernels: one quad at a time, to
            // leave registers for the epilogue's inputs).
            constexpr int NC = EPI ? 1 : CW / 4;
            float4 c[NC];
            if (read_c && !EPI) {
  #pragma unroll
              for (int q = 0; q < NC; ++q) c[q] = dst[q];
            }
            const float a = partial ? 1.f : p.alpha;
            with_activation<EPI>(epi_on, p.epi.act, [&](auto act_c) {
              constexpr int ACT = decltype(act_c)::value;
  #pragma unroll
              for (int q = 0; q < CW / 4; ++q) {
                float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                if constexpr (ACT == kActDGelu) {
                  if (q > 0 && q % NQH == 0) epi_fetch<NQH>(p.epi, row, col0 + 4 * q, p.N, epi_fetch_ok, xe);
                  x = xe[q % NQH];
                } else if constexpr (ACT >= 0) {
                  x = reinterpret_cast<const float4*>(bslot)[q];
                }
                float4 v = scaled4(a, r + 4 * q);
                if (read_c) {
                  const float4 cq = EPI ? dst[q] : c[q % NC];
                  v.x = fmaf(p.beta, cq.x, v.x);
                  v.y = fmaf(p.beta, cq.y, v.y);
                  v.z = fmaf(p.beta, cq.z, v.z);
                  v.w = fmaf(p.beta, cq.w, v.w);
                }
                v = epi_finish4<ACT>(v, x);
                dst[q] = v;
              }
            });
          } else {
            // TRANS_C: lanes hold consecutive rows, so each access of the warp is contiguous.
            auto at = [&](int j) { return TRANS_C ? out + (col0 + j) * ld + wrow : out + col0 + j; };
            float c[CW];
            if (read_c) {
  #pragma unroll
              for (int j = 0; j < CW; ++j) c[j] = (col0 + j < p.N) ? *at(j) : 0.f;
            }
            const float a = partial ? 1.f : p.alpha;
  #pragma unroll
            for (int j = 0; j < CW; ++j) {
              if (col0 + j < p.N) {
                float v = a * __uint_as_float(r[j]);
                if (read_c) v = fmaf(p.beta, c[j], v);
                if constexpr (EPI) {
                  if (!partial) v = apply_epilogue(p.epi, v, row, col0 + j);
                }
                *at(j) = v;
              }
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(dsmem_map(acce_bar(acc), 0));  // the even CTA's MMAs reuse the accumulator
          else
            mbar_arrive(acce_bar(acc));
        }
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // A load of Z still in flight (a wait that gave up) lands before the
      // CTA exits, and so does every TMA store of this warp.
      if constexpr (EPI) {
        __syncwarp();
        if (ZT) {
          const uint32_t zs = *z_word;
          if (zs & 2u) drain_wait(z_bar, zs & 1u, p.status, p.wait_ns);
        }
      }
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    };
    if constexpr (EPI) {
      if (p.epi.act == kActDGelu && p.z_tma != 0) {
        epilogue_role(std::true_type{});
      } else {
        epilogue_role(std::false_type{});
      }
    } else {
      epilogue_role(std::false_type{});
    }
  }

  tc_fence_before();
  __syncthreads();
  // PAIR: the peer may still commit to this CTA's barriers until it is done.
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

}  // namespace dgt
