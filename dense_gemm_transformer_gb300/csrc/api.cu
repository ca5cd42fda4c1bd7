// api.cu -- the C ABI (gemm.h): handles, argument checks, the planner and the
// workspace.
//
// The planner maps a call to one kernel family with a fixed rule (no runtime
// autotuning):
//   FP32             -> the register-tiled SIMT kernel with 128 x 128 or
//                       128 x 256 tiles, one CTA per tile when the tiles fill
//                       whole waves of the resident CTAs (>= 92%), stream-K
//                       over the resident CTAs otherwise; K-contiguous
//                       operands of long GEMMs are transposed first.
//   TF32, BF16       -> the persistent tcgen05 kernel; the tile width (128 or
//                       256 columns) is the one with the least time over
//                       whole waves of one tile per SM, and K is split
//                       when there are fewer tiles than half the SMs.
//   M <= 16, A M x K -> the same kernel in its swapped form (C^T = B^T A^T):
//                       the weights stream once through the 128-row MMA side,
//                       the activations are a 16-column operand, and K is
//                       split so that the units fill whole waves of the SMs.
// An operand whose base or leading dimension breaks the TMA unit's 16-byte
// rule is first copied into the workspace with an aligned leading dimension.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>

#include "gemm.h"
#include "kernels.h"
#include "skinny.cuh"

struct gemm_handle_s {
  int device = 0;
  int sms = 0;
  int* d_status = nullptr;   // the status word, then (from word kSkCntOffset) the SIMT stream-K arrival counters
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* ws_t = nullptr;  // the transposed result of a weight-gradient-shaped TF32 product (run_checked)
  size_t ws_t_bytes = 0;
  int opt_family = GEMM_FAMILY_AUTO;
  int opt_split_k = 0;
  int opt_tile_n = 0;
  int opt_pretranspose = 0;
  int opt_pair = 0;
  int64_t opt_wait_us = 0;   // bounded-wait limit of the tcgen05 kernel (0: the default)
  int opt_fault_skip = 0;    // test hook (GEMM_OPT_FAULT_SKIP_STAGE)
  int opt_sk_fixup = 0;      // GEMM_OPT_SK_FIXUP
  int sk_active[5][dgt::kSkinnyMaxCluster + 1];  // small-M kernel per mode (TF32, BF16, FP8, MXFP8, NVFP4): resident clusters (-1: not queried)
  dgt::TmaCache* tma_cache = nullptr;             // TMA descriptors of earlier calls
  gemm_plan_t plan{};
  dgt::LaunchShape null_shape;  // main kernel of the last successful gemm_run (for gemm_launch_null)
};

namespace {

constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
constexpr int kSkCntOffset = 64;  // words: the counters start 256 bytes after the status word

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool is_fp8(int mode) { return mode >= GEMM_MODE_FP8_E4M3 && mode <= GEMM_MODE_FP8_E5M2_E4M3; }
int elem_bytes(int mode) { return is_fp8(mode) ? 1 : mode == GEMM_MODE_BF16 ? 2 : 4; }
// The 8-bit formats of A and B in an FP8 mode (0 = E4M3, 1 = E5M2), the
// codes the kind::f8f6f4 instruction descriptor takes.
uint32_t fp8_format_a(int mode) { return (mode == GEMM_MODE_FP8_E5M2 || mode == GEMM_MODE_FP8_E5M2_E4M3) ? 1u : 0u; }
uint32_t fp8_format_b(int mode) { return (mode == GEMM_MODE_FP8_E5M2 || mode == GEMM_MODE_FP8_E4M3_E5M2) ? 1u : 0u; }

gemm_status_t check_args(int mode, int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                         const void* A, int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc) {
  if (mode < GEMM_MODE_FP32 || mode > GEMM_MODE_FP8_E5M2_E4M3) return GEMM_ERR_INVALID_VALUE;
  if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return GEMM_ERR_INVALID_VALUE;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr || ldc < std::max<int64_t>(N, 1)) return GEMM_ERR_INVALID_VALUE;
  if (!aligned(C, 4)) return GEMM_ERR_MISALIGNED;
  if (K == 0 || alpha == 0.f) return GEMM_OK;  // A and B are not read
  if (A == nullptr || B == nullptr) return GEMM_ERR_INVALID_VALUE;
  if (lda < std::max<int64_t>(transA ? M : K, 1)) return GEMM_ERR_INVALID_VALUE;
  if (ldb < std::max<int64_t>(transB ? K : N, 1)) return GEMM_ERR_INVALID_VALUE;
  if (!aligned(A, elem_bytes(mode)) || !aligned(B, elem_bytes(mode))) return GEMM_ERR_MISALIGNED;
  return GEMM_OK;
}

gemm_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA; }

bool epilogue_active(const dgt::EpiParams& e) { return e.act != dgt::kActNone || e.bias != nullptr; }

// Grow the workspace to at least `bytes`.  Freeing the old block waits for
// the device, so earlier launches that still use it are finished.
gemm_status_t ensure_ws(gemm_handle_s* h, size_t bytes) {
  if (bytes <= h->ws_bytes) return GEMM_OK;
  if (h->ws) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    cudaFree(h->ws);
    h->ws = nullptr;
    h->ws_bytes = 0;
  }
  size_t want = std::max<size_t>(bytes, size_t(1) << 20);
  if (cudaMalloc(&h->ws, want) != cudaSuccess) {
    cudaGetLastError();
    h->ws = nullptr;
    return GEMM_ERR_ALLOC;
  }
  h->ws_bytes = want;
  return GEMM_OK;
}

// The same for the handle's second buffer.
gemm_status_t ensure_ws_t(gemm_handle_s* h, size_t bytes) {
  if (bytes <= h->ws_t_bytes) return GEMM_OK;
  if (h->ws_t) {
    if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
    cudaFree(h->ws_t);
    h->ws_t = nullptr;
    h->ws_t_bytes = 0;
  }
  size_t want = std::max<size_t>(bytes, size_t(1) << 20);
  if (cudaMalloc(&h->ws_t, want) != cudaSuccess) {
    cudaGetLastError();
    h->ws_t = nullptr;
    return GEMM_ERR_ALLOC;
  }
  h->ws_t_bytes = want;
  return GEMM_OK;
}

struct WsLayout {
  size_t a_off = 0, b_off = 0, p_off = 0, total = 0;
};

void set_plan(gemm_handle_s* h, int family, int tm, int tn, int tk, int splits, int stages, int grid, int kernels,
              int packed) {
  gemm_plan_t p{};
  p.family = family;
  p.tile_m = tm;
  p.tile_n = tn;
  p.tile_k = tk;
  p.split_k = splits;
  p.stages = stages;
  p.grid = grid;
  p.kernels = kernels;
  p.packed = packed;
  h->plan = p;
}

// Whole-tile schedule efficiency: the fraction of the resident CTA slots the
// tiles keep busy over their waves.
double wave_eff(int64_t tiles, int64_t slots) {
  return static_cast<double>(tiles) / static_cast<double>(ceil_div(tiles, slots) * slots);
}

gemm_status_t run_simt(gemm_handle_s* h, int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                       const float* A, int64_t lda, const float* B, int64_t ldb, float beta, float* C, int64_t ldc,
                       const dgt::EpiParams& epi, cudaStream_t s) {
  using namespace dgt;
  const int64_t kt = ceil_div(K, kSimtTileK);
  // Tile width: 128 columns, two CTAs per SM.  The 256-column kernel (one
  // CTA per SM, fewer shared-memory reads per FFMA) measured 2-3% slower on
  // every shape where it needs no padding -- M = 4096-16384, N = 1536,
  // K = 384-1536, and the 2048^3 / 4096^3 squares (1024^3 a tie): with packed
  // FMAs and the next step's fragments preloaded in both, the second
  // resident CTA hiding each tile's fill and stores is worth more.  It stays
  // available through the tile-width option.
  if (h->opt_tile_n != 0 && h->opt_tile_n != 128 && h->opt_tile_n != 256) return GEMM_ERR_NOT_SUPPORTED;
  const int tile_n = h->opt_tile_n != 0 ? h->opt_tile_n : 128;
  const int64_t tiles = ceil_div(M, kSimtTileM) * ceil_div(N, tile_n);
  const int64_t slots = (tile_n == 256 ? 1 : 2) * static_cast<int64_t>(h->sms);  // resident CTAs
  // An operand stored with K contiguous must be transposed on its way to
  // shared memory.  Transposing it once into the workspace costs 8 bytes of
  // HBM traffic per element against 2 x (N or M) FLOPs per element of the
  // GEMM: ~33 / (the other dimension) of the GEMM's time.  A K-contiguous,
  // aligned A is transposed inside the kernel instead (16-byte row copies and
  // a shared-memory transpose), which costs a few percent of the kernel at
  // any N: measured on the GPT products, the in-kernel form is 2-8% faster
  // for N = 65-384 and 4-6% slower for N = 1152-1536, so A is transposed into
  // the workspace from N >= 768.  A K-contiguous B is read with 4-byte
  // transposing copies, which load the L1/shared-memory pipe far more than
  // 16-byte copies, so it is transposed into the workspace from M >= 256.
  const int pre = h->opt_pretranspose;  // 0 planner, 1 never, 2 always
  const bool tr_a = !transA && K > 0 && (pre == 2 || (pre == 0 && N >= 768 && M >= 128 && K >= 64));
  const bool tr_b = transB && K > 0 && (pre == 2 || (pre == 0 && M >= 256 && N >= 128 && K >= 64));
  const int64_t lda_t = round_up(M, 4), ldb_t = round_up(N, 4);
  // An operand whose base or rows are not 16-byte aligned would make the
  // kernel copy both operands 4 bytes at a time; a copy with an aligned
  // leading dimension costs one read and write of it and is made instead
  // (not with pretranspose = 1, which keeps operands in place).
  auto misaligned = [](const float* q, int64_t ld) { return (reinterpret_cast<uintptr_t>(q) & 15u) != 0 || ld % 4 != 0; };
  const bool pk_a = !tr_a && K > 0 && pre != 1 && misaligned(A, lda);
  const bool pk_b = !tr_b && K > 0 && pre != 1 && misaligned(B, ldb);
  const int64_t a_rows = transA ? K : M, a_cols = transA ? M : K;  // A as stored
  const int64_t b_rows = transB ? N : K, b_cols = transB ? K : N;  // B as stored
  const int64_t lda_p = round_up(a_cols, 4), ldb_p = round_up(b_cols, 4);
  SimtArgs a{};
  a.transA = transA;
  a.transB = transB;
  a.M = M;
  a.N = N;
  a.K = K;
  a.A = A;
  a.lda = lda;
  a.B = B;
  a.ldb = ldb;
  a.C = C;
  a.ldc = ldc;
  a.alpha = alpha;
  a.beta = beta;
  a.tile_n = tile_n;
  a.ws_ld = round_up(N, 4);
  a.splits = 1;
  a.k_per_split = K;
  int grid = static_cast<int>(std::min<int64_t>(tiles, INT32_MAX));
  int kernels = 1;
  // Whole tiles when they fill whole waves of the resident CTAs (or the
  // problem is too small to share out, or K is under 16 k-tiles: then every
  // tile would be split and its partial stores and fixup cost more than the
  // idle part of the last wave -- K = 65, 384 tiles: 58 us as stream-K,
  // 32 us as two waves of whole tiles); stream-K otherwise.
  if (h->opt_split_k > 0) {
    int64_t splits = h->opt_split_k;
    const int64_t kps = round_up(ceil_div(K, splits), kSimtTileK);
    splits = ceil_div(K, kps);
    a.schedule = splits > 1 ? kSimtSplitK : kSimtTiles;
    a.splits = static_cast<int>(splits);
    a.k_per_split = kps;
    grid = static_cast<int>(tiles * splits);
  } else if (wave_eff(tiles, slots) >= 0.92 || tiles * kt < 4 * slots || kt < 16) {
    a.schedule = kSimtTiles;
  } else {
    // Whole-tile waves first, stream-K over the rest: the last partial wave
    // (or, when it would give each CTA fewer than 4 k-tiles, the last wave
    // and a half) is shared out, so only those tiles go through the fixup.
    a.schedule = kSimtStreamK;
    const int64_t g = std::min<int64_t>(slots, 510);  // at most 510 CTAs (the fixup's part list)
    int64_t dp_waves = tiles / g;
    if (dp_waves > 0 && (tiles - dp_waves * g) * kt < 4 * g) --dp_waves;
    a.dp_tiles = dp_waves * g;
    a.iters = (tiles - a.dp_tiles) * kt;
    // at least 8 k-tiles per CTA when stream-K is all there is
    a.grid = a.dp_tiles > 0 ? g : std::max<int64_t>(1, std::min<int64_t>(g, a.iters / 8));
    grid = static_cast<int>(a.grid);
    // A tile cut into about two parts (runs of at least half its k-tiles) is
    // summed by the last CTA to finish a part of it, from L2, without a
    // fixup launch: measured on the GPT products, 10 us less per call on the
    // 256-column tiles of the K = 384 products (about two parts a tile), but
    // 5-7 us more where 128-column tiles have about five parts (one CTA then
    // reads more partials than the fixup kernel's 16 CTAs per tile), so
    // those, and deep-K tiles with dozens of parts, keep the fixup kernel.
    const bool few_parts = h->opt_sk_fixup == 2 || (h->opt_sk_fixup == 0 && kt <= 2 * (a.iters / a.grid));
    a.sk_inline = (few_parts && tiles - a.dp_tiles <= kSimtInlineMaxTiles) ? 1 : 0;
    a.sk_cnt = h->d_status + kSkCntOffset;
  }
  // Workspace: [split-K slices or stream-K slots][A transposed][B transposed].
  size_t part_bytes = 0;
  if (a.schedule == kSimtSplitK) part_bytes = static_cast<size_t>(a.splits * M * a.ws_ld) * sizeof(float);
  if (a.schedule == kSimtStreamK)
    part_bytes = static_cast<size_t>(2 * a.grid * simt_streamk_slot_floats(tile_n)) * sizeof(float);
  const size_t a_off = round_up(static_cast<int64_t>(part_bytes), 256);
  const size_t a_bytes = tr_a ? static_cast<size_t>(K * lda_t) * sizeof(float)
                              : pk_a ? static_cast<size_t>(a_rows * lda_p) * sizeof(float) : 0;
  const size_t b_off = a_off + round_up(static_cast<int64_t>(a_bytes), 256);
  const size_t b_bytes = tr_b ? static_cast<size_t>(K * ldb_t) * sizeof(float)
                              : pk_b ? static_cast<size_t>(b_rows * ldb_p) * sizeof(float) : 0;
  const size_t total = b_off + b_bytes;
  if (total > 0) {
    gemm_status_t st = ensure_ws(h, total);
    if (st != GEMM_OK) return st;
  }
  char* ws = static_cast<char*>(h->ws);
  if (part_bytes > 0) a.ws = reinterpret_cast<float*>(ws);
  if (a.schedule == kSimtStreamK && !a.sk_inline) ++kernels;  // the fixup
  if (a.schedule != kSimtStreamK && ceil_div(M, kSimtTileM) > 65535) return GEMM_ERR_NOT_SUPPORTED;
  if (tr_a) {
    float* at = reinterpret_cast<float*>(ws + a_off);
    if (launch_transpose(A, lda, at, lda_t, M, K, 4, s) != cudaSuccess) return GEMM_ERR_CUDA;
    a.A = at;
    a.lda = lda_t;
    a.transA = 1;
    ++kernels;
  }
  if (tr_b) {
    float* bt = reinterpret_cast<float*>(ws + b_off);
    if (launch_transpose(B, ldb, bt, ldb_t, N, K, 4, s) != cudaSuccess) return GEMM_ERR_CUDA;
    a.B = bt;
    a.ldb = ldb_t;
    a.transB = 0;
    ++kernels;
  }
  if (pk_a) {
    float* ap = reinterpret_cast<float*>(ws + a_off);
    if (launch_pack(A, lda, ap, lda_p, a_rows, a_cols, 4, s) != cudaSuccess) return GEMM_ERR_CUDA;
    a.A = ap;
    a.lda = lda_p;
    ++kernels;
  }
  if (pk_b) {
    float* bp = reinterpret_cast<float*>(ws + b_off);
    if (launch_pack(B, ldb, bp, ldb_p, b_rows, b_cols, 4, s) != cudaSuccess) return GEMM_ERR_CUDA;
    a.B = bp;
    a.ldb = ldb_p;
    ++kernels;
  }
  if (launch_simt(a, s) != cudaSuccess) return GEMM_ERR_CUDA;
  // The epilogue: in the split-K reduction, which writes every element
  // anyway, or else in one pass over C after the GEMM.
  if (a.schedule == kSimtSplitK) {
    if (launch_splitk_reduce(M, N, a.splits, a.ws, a.ws_ld, C, ldc, alpha, beta, epi, 0, s) != cudaSuccess)
      return GEMM_ERR_CUDA;
    ++kernels;
  } else if (epilogue_active(epi)) {
    if (launch_epilogue(M, N, C, ldc, epi, s) != cudaSuccess) return GEMM_ERR_CUDA;
    ++kernels;
  }
  set_plan(h, GEMM_FAMILY_SIMT, kSimtTileM, tile_n, kSimtTileK, a.splits, tile_n == 256 ? 4 : 3, grid, kernels,
           ((tr_a || pk_a) ? 1 : 0) | ((tr_b || pk_b) ? 2 : 0));
  h->plan.schedule = a.schedule;
  h->plan.sk_fixup = a.schedule != kSimtStreamK ? 0 : a.sk_inline ? 2 : 1;
  return GEMM_OK;
}

// How one tensor-core operand reaches the kernel.  `rows x cols` is the
// operand as stored (row-major, pitch `ld`); `mn_major` says its contiguous
// dimension is M (or N) rather than K.
struct OperandPack {
  enum Kind { kNone, kCopy, kTranspose } kind = kNone;
  const void* src = nullptr;
  int64_t ld = 0, rows = 0, cols = 0, dst_ld = 0;
  bool mn_major_after = false;
  size_t bytes = 0;
};

OperandPack plan_pack(const void* src, int64_t ld, int64_t rows, int64_t cols, bool mn_major, int mode, int es,
                      bool mn_ok = false) {
  OperandPack p;
  p.src = src;
  p.ld = ld;
  p.rows = rows;
  p.cols = cols;
  p.mn_major_after = mn_major;
  if ((mode == GEMM_MODE_TF32 || mode == GEMM_MODE_FP8_E4M3) && mn_major && !mn_ok) {
    p.kind = OperandPack::kTranspose;  // stored K x MN -> MN x K
    p.dst_ld = round_up(rows, 16 / es);
    p.bytes = static_cast<size_t>(cols * p.dst_ld * es);
    p.mn_major_after = false;
  } else if (!aligned(src, 16) || (ld * es) % 16 != 0) {
    p.kind = OperandPack::kCopy;
    p.dst_ld = round_up(cols, 16 / es);
    p.bytes = static_cast<size_t>(rows * p.dst_ld * es);
  }
  return p;
}

cudaError_t run_pack(const OperandPack& p, void* dst, int es, cudaStream_t s) {
  if (p.kind == OperandPack::kTranspose) return dgt::launch_transpose(p.src, p.ld, dst, p.dst_ld, p.rows, p.cols, es, s);
  return dgt::launch_pack(p.src, p.ld, dst, p.dst_ld, p.rows, p.cols, es, s);
}

// Rates used only to weigh a wave of tiles against the extra reduction
// traffic of a K split: dense tensor rates as measured on this part, a
// kernel efficiency of 0.8 of them, HBM bandwidth and the cost of one more
// (programmatically launched) kernel.
constexpr double kBf16Flops = 1.9e15 * 0.8;
constexpr double kTf32Flops = 0.95e15 * 0.8;
constexpr double kFp8Flops = 3.8e15 * 0.8;  // twice the bf16 rate (nominal ratio)
constexpr double kHbmBytes = 6.5e12;
constexpr double kLaunchS = 1.5e-6;

// Which last rows of work units to cut into K slices, and into how many:
// units are handed out round-robin to `slots` persistent CTAs (or CTA
// pairs), whole units first; each option's time is that of the busiest CTA
// (a cut unit counts its share of K) plus the reduction of the cut rows'
// partial sums by a separate kernel.  rows == 0: no cut.  O(rows x 7).
struct TailPlan {
  int64_t rows = 0, slices = 1, kb_per = 0;
  double seconds = 0.0;  // estimated time of the chosen schedule
};

TailPlan plan_tail(int64_t unit_rows, int64_t unit_cols, int64_t kb, int64_t slots, double unit_s,
                   double c_bytes_per_row, bool read_c) {
  TailPlan best_plan;
  const int64_t U = unit_rows * unit_cols;
  double best = static_cast<double>(ceil_div(U, std::max<int64_t>(slots, 1))) * unit_s;
  best_plan.seconds = best;
  if (U <= slots || U % slots == 0 || kb < 8 || slots <= 0) return best_plan;
  for (int64_t R = 1; R < unit_rows && R * unit_cols <= 2 * slots; ++R) {
    const int64_t cut = R * unit_cols, D = U - cut;
    for (int64_t want = 2; want <= 8 && kb / want >= 4; ++want) {
      const int64_t per = ceil_div(kb, want), sl = ceil_div(kb, per);
      const double f = static_cast<double>(per) / static_cast<double>(kb);
      const int64_t T = D + cut * sl;
      // CTA c runs the units c, c + slots, ...: its counts of whole units and
      // of all units both fall as c grows, so CTA 0 is the busiest.
      const double dp0 = static_cast<double>(ceil_div(D, slots));
      const double worst = dp0 + (static_cast<double>(ceil_div(T, slots)) - dp0) * f;
      const double reduce = static_cast<double>(R) * c_bytes_per_row * (sl + 1 + (read_c ? 1 : 0)) / kHbmBytes;
      const double cost = worst * unit_s + reduce + kLaunchS;
      if (cost < 0.98 * best) {
        best = cost;
        best_plan.rows = R;
        best_plan.slices = sl;
        best_plan.kb_per = per;
        best_plan.seconds = cost;
      }
    }
  }
  return best_plan;
}

// K slices (= CTAs per cluster) for the small-M kernel: as many as one wave
// of two resident CTAs per SM holds, at least two K blocks per slice, at
// most 16, and above the portable cluster size of 8 only a size the device
// can launch.  Measured on the decode shapes (calls back to back): 280 CTAs
// for 70 tiles and 192 for 12 tiles ran fastest, 140 and 96-120 ran 25-30%
// slower, although only 7 clusters of 16 are resident at once (the next
// call's CTAs, started early, fill the SMs the second wave leaves idle).
int64_t skinny_cluster_size(gemm_handle_s* h, int mode, bool a_mn, int64_t tiles, int64_t kb) {
  int64_t cs = std::min<int64_t>(2 * h->sms / tiles, dgt::kSkinnyMaxCluster);
  cs = std::max<int64_t>(1, std::min<int64_t>(cs, kb / 2));
  while (cs > 8) {
    int& act = h->sk_active[mode - GEMM_MODE_TF32][cs];
    if (act < 0) act = dgt::skinny_max_active_clusters(mode, a_mn, static_cast<int>(cs));
    if (act > 0) break;
    --cs;
  }
  return cs;
}

gemm_status_t run_tc(gemm_handle_s* h, int mode, int transA, int transB, int64_t M, int64_t N, int64_t K,
                     float alpha, const void* A, int64_t lda, const void* B, int64_t ldb, float beta, float* C,
                     int64_t ldc, const dgt::EpiParams& epi, cudaStream_t s, bool swap, uint32_t fmt_a = 0,
                     uint32_t fmt_b = 0) {
  using namespace dgt;
  const int es = elem_bytes(mode);
  const int bk = tc_tile_k(mode);
  const int sms = h->sms;
  // The swapped form computes C^T = op(B)^T op(A)^T: the kernel sees M' = N,
  // N' = M, A' = B and B' = A, and stores its tiles transposed.
  const int64_t Mk = swap ? N : M, Nk = swap ? M : N;
  const int ta_k = swap ? !transB : transA;  // is the kernel's A stored K x M'?
  const int tb_k = swap ? !transA : transB;  // is the kernel's B stored N' x K?
  const void* Ak = swap ? B : A;
  const void* Bk = swap ? A : B;
  const int64_t ldak = swap ? ldb : lda, ldbk = swap ? lda : ldb;

  // Tile width (128, 192, 224 or 256 columns) and schedule: the least
  // estimated time over waves of work units, a unit being one tile per CTA
  // or, where a CTA pair issues one 256-row MMA, two vertically adjacent
  // tiles per pair; the last rows of units may be cut into K slices to fill
  // the final wave (plan_tail).  A tile's time is taken as proportional to the
  // shared-memory bytes of one stage, A (128 rows) + B (tile_n rows) of 128
  // bytes each: that makes a 128-column tile 3/4 as fast per column as a
  // 256-column one, as measured on square and large shapes.  Ties go to the
  // wider tile.  The B layout the kernel reads is MN-major only for BF16
  // (TF32 and FP8 operands are made K-major).
  const bool b_mn_kernel = (mode == GEMM_MODE_BF16) && tb_k == 0;
  const int64_t tm_tiles = ceil_div(Mk, 128);
  const int64_t kb = ceil_div(K, bk);
  auto pair_ok = [&](int tn) {
    return !swap && tm_tiles >= 2 && h->opt_pair != 1 && h->opt_fault_skip == 0 &&
           dgt::tc_tile_ok(mode, tn, true, b_mn_kernel);
  };
  const double peak =
      (mode == GEMM_MODE_FP8_E4M3 ? kFp8Flops : mode == GEMM_MODE_BF16 ? kBf16Flops : kTf32Flops) / sms;
  // A CTA pair issues one MMA of 256 rows (tcgen05 cta_group::2): each CTA
  // then stages and reads half of B, which measured 1.14x the speed on large
  // shapes (BF16 8192^3: 1687 -> 1929 TFLOP/s at 256 columns).  TF32 stages
  // twice the bytes per FLOP, and with 24 or more K blocks the halved B
  // measured worth more: on the N = 384 GPT products (K = 1152-1536) the
  // 256-column pairs, padding N to 512, ran 8-10% faster than 192-column
  // tiles (MLP-down forward 46.9 -> 42.4 us), which a factor of 1.3
  // reproduces; with short K the tile's fixed cost dominates and 1.14 still
  // ranks the widths as measured.
  const double pair_gain = (mode == GEMM_MODE_TF32 && kb >= 24) ? 1.3 : 1.14;
  // Estimated time of tiles of tn columns, as CTA pairs (pr) or one CTA per
  // tile.  Shapes with fewer tiles than half the SMs and 8 or more K blocks
  // are split along K so that the (tile, slice) units fill one wave (then
  // the slices' partial sums pass through the workspace); others may cut
  // their last rows of units into K slices (plan_tail).
  auto split_units = [&](int tn, bool pr) {
    const int64_t units = (pr ? ceil_div(tm_tiles, 2) : tm_tiles) * ceil_div(Nk, tn);
    return std::max<int64_t>(1, std::min<int64_t>((pr ? sms / 2 : sms) / units, kb / 4));
  };
  auto plan_for = [&](int tn, bool pr) {
    const int64_t rows = pr ? ceil_div(tm_tiles, 2) : tm_tiles;
    const int64_t cols = ceil_div(Nk, tn);
    const int64_t slots = pr ? sms / 2 : sms;
    const double unit_s = 2.0 * 128.0 * 256.0 * static_cast<double>(K) / peak *
                          (128.0 * 128.0 + 128.0 * tn) / (128.0 * 384.0) / (pr ? pair_gain : 1.0);
    const double c_row_bytes = 4.0 * static_cast<double>(Nk) * (pr ? 256.0 : 128.0);
    const bool split = !swap && h->opt_split_k == 0 && 2 * tm_tiles * cols <= sms && kb >= 8;
    if (split) {
      int64_t sl = split_units(tn, pr);
      const int64_t per = ceil_div(kb, sl);
      sl = ceil_div(kb, per);
      TailPlan t;
      t.seconds = static_cast<double>(ceil_div(rows * cols * sl, slots)) * unit_s * static_cast<double>(per) /
                      static_cast<double>(kb) +
                  4.0 * static_cast<double>(Mk) * static_cast<double>(Nk) * static_cast<double>(sl + 1 + (beta != 0.f)) /
                      kHbmBytes +
                  kLaunchS;
      return t;
    }
    if (swap || h->opt_split_k > 0) {
      TailPlan none;
      none.seconds = static_cast<double>(ceil_div(rows * cols, slots)) * unit_s;
      return none;
    }
    return plan_tail(rows, cols, kb, slots, unit_s, c_row_bytes, beta != 0.f);
  };
  int tile_n = 16;
  bool pair = false;
  if (!swap && h->opt_tile_n != 0) {
    // a forced width pairs wherever it can (unless pairs are turned off)
    if (!dgt::tc_tile_ok(mode, h->opt_tile_n, false, b_mn_kernel)) return GEMM_ERR_NOT_SUPPORTED;
    tile_n = h->opt_tile_n;
    pair = pair_ok(tile_n);
  } else if (!swap) {
    double best = 0.0;
    // A TF32 A stored with M contiguous reaches the 128-column one-CTA
    // kernel through TMEM; every other width or a pair must transpose it
    // first: 8 bytes of HBM traffic per element of A, charged to them here
    // (without it the dW products, whose A is the whole activation matrix,
    // took wider pairs and ran 1.2-2x slower).
    const bool tmem_a_possible =
        mode == GEMM_MODE_TF32 && ta_k != 0 && Nk < 1536 && h->opt_pretranspose != 2;
    const double a_transpose_s = 8.0 * static_cast<double>(Mk) * static_cast<double>(K) / kHbmBytes + kLaunchS;
    // Every width, as pairs where they can run and as single CTAs: pairs
    // halve each CTA's B traffic, but at a small odd number of tile rows
    // (M = 384: a pair row is half idle) single CTAs win (the K-split dW
    // products: 88-90 us as single CTAs against 101-108 us as pairs).
    for (int tn : {256, 224, 192, 128}) {
      if (!dgt::tc_tile_ok(mode, tn, false, b_mn_kernel)) continue;
      for (const bool pr : {true, false}) {
        if (pr && !pair_ok(tn)) continue;
        const bool a_via_tmem = tn == 128 && !pr;
        const double cost = plan_for(tn, pr).seconds + (tmem_a_possible && !a_via_tmem ? a_transpose_s : 0.0);
        if (tile_n == 16 || cost < best * 0.999) {
          best = cost;
          tile_n = tn;
          pair = pr;
        }
      }
    }
  }
  const int64_t tiles = ceil_div(Mk, 128) * ceil_div(Nk, tile_n);
  // Small M with fewer than two waves of weight tiles: the cluster kernel
  // (one tile and K slice per CTA, slices reduced within the cluster).
  // With more tiles, the persistent kernel streams them without a split.
  const bool cluster_form = swap && tiles < 2 * sms;
  int64_t splits = 1;
  if (cluster_form) {
    splits = (h->opt_split_k > 0)
                 ? std::min<int64_t>({static_cast<int64_t>(h->opt_split_k), dgt::kSkinnyMaxCluster, kb})
                 : skinny_cluster_size(h, mode, mode == GEMM_MODE_BF16 && ta_k != 0, tiles, kb);
  } else if (h->opt_split_k > 0) {
    splits = std::min<int64_t>(h->opt_split_k, kb);
  } else if (swap) {
    splits = 1;  // two or more waves of weight tiles: a K split would only add traffic
  } else if (2 * tiles <= sms && kb >= 8) {
    splits = split_units(tile_n, pair);
  }
  int64_t kb_per = ceil_div(kb, splits);
  splits = ceil_div(kb, kb_per);
  // More than a wave of units that does not end on a whole wave: the last
  // rows of units may be cut into K slices so that the final wave is full.
  const int64_t unit_rows = pair ? ceil_div(tm_tiles, 2) : tm_tiles;
  const int64_t unit_cols = ceil_div(Nk, tile_n);
  TailPlan tail;
  if (!swap && splits == 1 && h->opt_split_k == 0) {
    tail = plan_for(tile_n, pair);
    if (tail.rows > 0) {
      splits = tail.slices;
      kb_per = tail.kb_per;
    }
  }
  const int64_t tail_row0 = tail.rows > 0 ? (unit_rows - tail.rows) * (pair ? 256 : 128) : 0;  // first C row cut

  // Workspace: re-packed operands and split-K partials.  An operand is copied
  // when the TMA unit cannot read it in place (base not 16-byte aligned, or a
  // row pitch that is not a multiple of 16 bytes), and transposed into K-major
  // order when it is MN-major in TF32 or FP8 mode: kind::tf32 takes K-major
  // operands from shared memory only (an MN-major TF32 operand produced zeros
  // on this part, while BF16 reads both orders), and the FP8 build reads
  // K-major operands only.  The exception is an MN-major A with
  // 128-column tiles and no CTA pairs: that kernel moves A into TMEM, where
  // the MMA reads it row by row, so no transpose pass is needed (unless
  // pretranspose = 2 asks for one).  The warps that move A slow the MMA
  // loop by ~20% on long K, against a pass that costs 8 bytes of HBM
  // traffic per element of A for 2N FLOPs per element: measured on the TF32
  // dW products, TMEM took 20-25% off for N = 65-384, broke even at
  // N = 1152 and lost 2% at N = 1536, so it is used for N < 1536.
  const bool a_tmem = mode == GEMM_MODE_TF32 && !swap && tile_n == 128 && !pair && Nk < 1536 &&
                      h->opt_pretranspose != 2;
  OperandPack pa = plan_pack(Ak, ldak, ta_k ? K : Mk, ta_k ? Mk : K, ta_k != 0, mode, es, a_tmem);
  OperandPack pb = plan_pack(Bk, ldbk, tb_k ? Nk : K, tb_k ? K : Nk, tb_k == 0, mode, es);
  WsLayout L;
  L.a_off = 0;
  L.b_off = round_up(static_cast<int64_t>(pa.bytes), 256);
  L.p_off = L.b_off + round_up(static_cast<int64_t>(pb.bytes), 256);
  const int64_t ws_ld = round_up(N, 4);
  L.total = L.p_off +
            (splits > 1 && !cluster_form ? static_cast<size_t>(splits * (M - tail_row0) * ws_ld) * sizeof(float) : 0);
  if (L.total > 0) {
    gemm_status_t st = ensure_ws(h, L.total);
    if (st != GEMM_OK) return st;
  }
  char* ws = static_cast<char*>(h->ws);
  int kernels = 0;
  const void* Ause = Ak;
  const void* Buse = Bk;
  int64_t lda_use = ldak, ldb_use = ldbk;
  bool a_mn = ta_k != 0, b_mn = tb_k == 0;
  if (pa.kind != OperandPack::kNone) {
    if (run_pack(pa, ws + L.a_off, es, s) != cudaSuccess) return GEMM_ERR_CUDA;
    Ause = ws + L.a_off;
    lda_use = pa.dst_ld;
    a_mn = pa.mn_major_after;
    ++kernels;
  }
  if (pb.kind != OperandPack::kNone) {
    if (run_pack(pb, ws + L.b_off, es, s) != cudaSuccess) return GEMM_ERR_CUDA;
    Buse = ws + L.b_off;
    ldb_use = pb.dst_ld;
    b_mn = pb.mn_major_after;
    ++kernels;
  }
  const bool pack_a = pa.kind != OperandPack::kNone, pack_b = pb.kind != OperandPack::kNone;

  TcArgs a{};
  a.mode = mode;
  // the kernel's operands are the caller's exchanged in the swapped form
  a.fmt8 = mode == GEMM_MODE_FP8_E4M3 ? fp8_format_bits(swap ? fmt_b : fmt_a, swap ? fmt_a : fmt_b) : 0u;
  a.a_mn_major = a_mn ? 1 : 0;
  a.b_mn_major = b_mn ? 1 : 0;
  a.tile_n = tile_n;
  a.M = Mk;
  a.N = Nk;
  a.K = K;
  a.A = Ause;
  a.lda = lda_use;
  a.B = Buse;
  a.ldb = ldb_use;
  a.C = C;
  a.ldc = ldc;
  a.alpha = alpha;
  a.beta = beta;
  a.splits = static_cast<int>(splits);
  a.kb_per_split = static_cast<int>(kb_per);
  a.tma_cache = h->tma_cache;
  if (cluster_form) {
    a.status = h->d_status;
    a.grid = static_cast<int>(tiles * splits);
    if (launch_skinny(a, s) != cudaSuccess) return GEMM_ERR_CUDA;
    ++kernels;
    if (epilogue_active(epi)) {
      if (launch_epilogue(M, N, C, ldc, epi, s) != cudaSuccess) return GEMM_ERR_CUDA;
      ++kernels;
    }
    set_plan(h, GEMM_FAMILY_SKINNY, 128, 16, bk, a.splits, dgt::skinny_stages(mode), a.grid, kernels,
             (pack_b ? 1 : 0) | (pack_a ? 2 : 0));
    h->plan.cluster = a.splits;
    h->plan.schedule = a.splits > 1 ? 1 : 0;
    return GEMM_OK;
  }
  // Partial sums are kept in the caller's M x N orientation, from C row
  // tail_row0 on (0 unless only the last rows of units are cut).
  a.ws = splits > 1 ? reinterpret_cast<float*>(ws + L.p_off) : nullptr;
  a.ws_ld = ws_ld;
  a.ws_row0 = tail_row0;
  a.ws_slice = (M - tail_row0) * ws_ld;
  a.dp_units = static_cast<int>(tail.rows > 0 ? (unit_rows - tail.rows) * unit_cols : 0);
  a.tail_tm0 = static_cast<int>(tail.rows > 0 ? unit_rows - tail.rows : 0);
  a.status = h->d_status;
  // The elementwise epilogue inside the GEMM kernel's epilogue warps, where
  // it is built for the operand layouts (K-major A): whole tiles get it at
  // their store, and a split's partial sums get it in the slice reduce.
  const bool fuse = epilogue_active(epi) && (mode == GEMM_MODE_TF32 || mode == GEMM_MODE_BF16) &&
                    dgt::tc_epi_ok(mode, a_mn, b_mn);
  a.fuse_epi = fuse;
  a.epi = epi;
  a.wait_ns = static_cast<uint64_t>(h->opt_wait_us) * 1000u;
  a.fault_skip = h->opt_fault_skip;
  // CTA pairs issuing one 256-row MMA for tiles of 192 columns or more
  // with at least two rows of tiles: each CTA then stages half of B per
  // stage (256 columns: 32 KB instead of 48 KB).
  a.pair = pair ? 1 : 0;
  const int64_t units = a.dp_units + (unit_rows - a.tail_tm0) * unit_cols * splits;
  a.grid = static_cast<int>(pair ? 2 * std::min<int64_t>(units, sms / 2) : std::min<int64_t>(units, sms));
  a.group_m = a.pair ? 8 : 16;
  if (launch_tc(a, s) != cudaSuccess) return GEMM_ERR_CUDA;
  ++kernels;
  // The epilogue: fused into the GEMM kernel (and the reduction of any cut
  // rows), in the split-K reduction when it writes every element of C
  // (plain split-K), or else in one pass over C after the GEMM.
  const bool epi_in_reduce = splits > 1 && (tail_row0 == 0 || fuse);
  if (splits > 1) {
    if (launch_splitk_reduce(M - tail_row0, N, a.splits, a.ws, ws_ld, C + tail_row0 * ldc, ldc, alpha, beta,
                             epi_in_reduce ? epi : dgt::EpiParams{}, tail_row0, s) != cudaSuccess)
      return GEMM_ERR_CUDA;
    ++kernels;
  }
  if (!fuse && !epi_in_reduce && epilogue_active(epi)) {
    if (launch_epilogue(M, N, C, ldc, epi, s) != cudaSuccess) return GEMM_ERR_CUDA;
    ++kernels;
  }
  set_plan(h, swap ? GEMM_FAMILY_SKINNY : GEMM_FAMILY_TC, 128, tile_n, bk, a.splits, tc_stages(mode, tile_n, a.pair != 0, fuse),
           a.grid, kernels, (swap ? ((pack_b ? 1 : 0) | (pack_a ? 2 : 0)) : ((pack_a ? 1 : 0) | (pack_b ? 2 : 0))));
  h->plan.cluster = a.pair ? 2 : 1;
  h->plan.pair_mma = a.pair;
  h->plan.schedule = tail.rows > 0 ? 3 : (a.splits > 1 ? 1 : 0);
  h->plan.epilogue_fused = fuse ? 1 : 0;
  return GEMM_OK;
}

// The block-scaled product (gemm_run_block_scaled) after its argument
// checks, in the kernels' block-scaled builds (kernel mode 4 for MXFP8, 5
// for NVFP4).  M <= 16: the small-M kernels, swapped like every small-M
// call -- the weights B (N x K) are the 128-row MMA operand and their
// scales the kernel's A scales, the activations A (M x K) the 16-row
// operand.  M > 16: the persistent kernel on 128 x 128 tiles of one CTA,
// A and B as they are, every stage bringing both operands' scale atoms.
// Codes and scales are read in place; K and the leading dimensions travel
// in bytes.
gemm_status_t run_block_scaled(gemm_handle_s* h, int mode, int64_t M, int64_t N, int64_t K, float alpha,
                               const void* A, int64_t lda, const void* SA, const void* B, int64_t ldb,
                               const void* SB, float beta, float* C, int64_t ldc, cudaStream_t s) {
  using namespace dgt;
  const bool nvfp4 = mode == GEMM_MODE_NVFP4;
  const int kmode = nvfp4 ? 5 : 4;
  const int64_t kbytes = nvfp4 ? K / 2 : K;
  const int64_t lda_b = nvfp4 ? lda / 2 : lda, ldb_b = nvfp4 ? ldb / 2 : ldb;
  const int64_t bs = nvfp4 ? 16 : 32;  // K elements per scale
  if (M > 16) {
    const int64_t tiles = ceil_div(M, 128) * ceil_div(N, 128);
    TcArgs a{};
    a.mode = kmode;
    a.fmt8 = mode == GEMM_MODE_MXFP8_E5M2 ? fp8_format_bits(1, 1) : 0u;
    a.tile_n = 128;
    a.M = M;
    a.N = N;
    a.K = kbytes;
    a.A = A;
    a.lda = lda_b;
    a.B = B;
    a.ldb = ldb_b;
    a.C = C;
    a.ldc = ldc;
    a.alpha = alpha;
    a.beta = beta;
    a.splits = 1;
    a.kb_per_split = static_cast<int>(ceil_div(kbytes, 128));
    a.tma_cache = h->tma_cache;
    a.status = h->d_status;
    a.grid = static_cast<int>(std::min<int64_t>(tiles, h->sms));
    a.group_m = 16;
    a.wait_ns = static_cast<uint64_t>(h->opt_wait_us) * 1000u;
    a.sfa = static_cast<const uint8_t*>(SA);
    a.sfb = static_cast<const uint8_t*>(SB);
    a.sf_groups = block_scale_groups(ceil_div(K, bs));
    if (launch_tc(a, s) != cudaSuccess) return GEMM_ERR_CUDA;
    set_plan(h, GEMM_FAMILY_TC, 128, 128, static_cast<int>(nvfp4 ? 256 : 128), 1, tc_stages(kmode, 128, false),
             a.grid, 1, 0);
    return GEMM_OK;
  }
  const int64_t tiles = ceil_div(N, 128);
  const int64_t kb = ceil_div(kbytes, 128);
  // Two or more waves of weight tiles (the vocabulary projection): the
  // persistent kernel, each CTA streaming tile after tile without a split
  // (a CTA per tile would pay its set-up for a handful of stages); fewer
  // tiles: the cluster kernel with K split across the cluster.
  const bool persistent = tiles >= 2 * h->sms && h->opt_split_k == 0;
  int64_t splits = persistent ? 1
                   : (h->opt_split_k > 0)
                       ? std::min<int64_t>({static_cast<int64_t>(h->opt_split_k), kSkinnyMaxCluster, kb})
                       : skinny_cluster_size(h, kmode, false, tiles, kb);
  const int64_t kb_per = ceil_div(kb, splits);
  splits = ceil_div(kb, kb_per);
  TcArgs a{};
  a.mode = kmode;
  a.fmt8 = mode == GEMM_MODE_MXFP8_E5M2 ? fp8_format_bits(1, 1) : 0u;
  a.tile_n = 16;
  a.M = N;
  a.N = M;
  a.K = kbytes;
  a.A = B;
  a.lda = ldb_b;
  a.B = A;
  a.ldb = lda_b;
  a.C = C;
  a.ldc = ldc;
  a.alpha = alpha;
  a.beta = beta;
  a.splits = static_cast<int>(splits);
  a.kb_per_split = static_cast<int>(kb_per);
  a.tma_cache = h->tma_cache;
  a.status = h->d_status;
  a.grid = static_cast<int>(tiles * splits);
  a.sfa = static_cast<const uint8_t*>(SB);
  a.sfb = static_cast<const uint8_t*>(SA);
  a.sf_groups = block_scale_groups(ceil_div(K, bs));
  if (persistent) {
    a.grid = static_cast<int>(std::min<int64_t>(tiles, h->sms));
    a.group_m = 16;
    a.wait_ns = static_cast<uint64_t>(h->opt_wait_us) * 1000u;
    if (launch_tc(a, s) != cudaSuccess) return GEMM_ERR_CUDA;
  } else {
    if (launch_skinny(a, s) != cudaSuccess) return GEMM_ERR_CUDA;
  }
  set_plan(h, GEMM_FAMILY_SKINNY, 128, 16, static_cast<int>(nvfp4 ? 256 : 128), a.splits,
           persistent ? tc_stages(kmode, 16, false) : skinny_stages(kmode), a.grid, 1, 0);
  h->plan.cluster = persistent ? 1 : a.splits;
  h->plan.schedule = a.splits > 1 ? 1 : 0;
  return GEMM_OK;
}

// gemm_run after its argument checks.
gemm_status_t run_checked(gemm_handle_t h, int mode, int transA, int transB, int64_t M, int64_t N, int64_t K,
                          float alpha, const void* A, int64_t lda, const void* B, int64_t ldb, float beta, float* C,
                          int64_t ldc, const dgt::EpiParams& epi, cudaStream_t s) {
  if (M == 0 || N == 0) {
    set_plan(h, 0, 0, 0, 0, 0, 0, 0, 0, 0);
    return GEMM_OK;
  }
  if (K == 0 || alpha == 0.f) {
    if (dgt::launch_scale(M, N, C, ldc, beta, epi, s) != cudaSuccess) return GEMM_ERR_CUDA;
    set_plan(h, 0, 0, 0, 0, 1, 0, 0, 1, 0);
    return GEMM_OK;
  }
  const int fam = h->opt_family;
  if (mode == GEMM_MODE_FP32) {
    if (fam != GEMM_FAMILY_AUTO && fam != GEMM_FAMILY_SIMT) return GEMM_ERR_NOT_SUPPORTED;
    return run_simt(h, transA, transB, M, N, K, alpha, static_cast<const float*>(A), lda,
                    static_cast<const float*>(B), ldb, beta, C, ldc, epi, s);
  }
  // Small M: the swapped form, which streams the weights through the 128-row
  // MMA side once (activations must be stored M x K).
  const bool skinny_ok = (transA == 0) && M <= 16;
  if (fam == GEMM_FAMILY_SKINNY && !skinny_ok) return GEMM_ERR_NOT_SUPPORTED;
  if (fam == GEMM_FAMILY_SIMT) return GEMM_ERR_NOT_SUPPORTED;
  const bool swap = (fam == GEMM_FAMILY_SKINNY) || (fam == GEMM_FAMILY_AUTO && skinny_ok);
  // Every FP8 mode runs the kernels' 8-bit build (GEMM_MODE_FP8_E4M3) with
  // its operand formats named at run time.
  if (is_fp8(mode))
    return run_tc(h, GEMM_MODE_FP8_E4M3, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, epi, s, swap,
                  fp8_format_a(mode), fp8_format_b(mode));
  // Weight-gradient-shaped TF32 products, C = A^T B with A stored K x M and
  // B stored K x N and N well above M (a dW = X^T dY): kind::tf32 reads only
  // K-major operands, so one operand is moved through TMEM (the kernel's A,
  // 128-column tiles) and the other is transposed into the workspace first.
  // Computed as it stands, that transposes the wide B; computed as
  // C^T = B^T A into a second buffer, B becomes the kernel's A (through
  // TMEM) and only the narrow A is transposed, and a final transpose of the
  // M x N result (much smaller than B when K is long) puts C in place.
  if (mode == GEMM_MODE_TF32 && fam == GEMM_FAMILY_AUTO && !swap && transA == 1 && transB == 0 &&
      epi.act == dgt::kActNone && epi.bias == nullptr && beta == 0.f && N >= 2 * M && K >= 4096 &&
      h->opt_tile_n == 0 && h->opt_pair == 0 && h->opt_split_k == 0 && h->opt_pretranspose == 0 &&
      h->opt_fault_skip == 0) {
    const int64_t ldt = round_up(M, 4);
    gemm_status_t st = ensure_ws_t(h, static_cast<size_t>(N * ldt) * sizeof(float));
    if (st != GEMM_OK) return st;
    float* ct = static_cast<float*>(h->ws_t);
    h->opt_tile_n = 128;  // the kernel that takes its A through TMEM
    h->opt_pair = 1;
    st = run_tc(h, mode, 1, 0, N, M, K, alpha, B, ldb, A, lda, 0.f, ct, ldt, epi, s, false);
    h->opt_tile_n = 0;
    h->opt_pair = 0;
    if (st != GEMM_OK) return st;
    if (dgt::launch_transpose(ct, ldt, C, ldc, N, M, 4, s) != cudaSuccess) return GEMM_ERR_CUDA;
    h->plan.kernels += 1;
    return GEMM_OK;
  }
  return run_tc(h, mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, epi, s, swap);
}

}  // namespace

extern "C" {

gemm_status_t gemm_create(gemm_handle_t* out) {
  if (out == nullptr) return GEMM_ERR_INVALID_VALUE;
  *out = nullptr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GEMM_ERR_CUDA;
  // The kernels are built for sm_103a only.
  if (major != 10 || minor != 3) return GEMM_ERR_NOT_SUPPORTED;
  gemm_handle_s* h = new (std::nothrow) gemm_handle_s();
  if (h == nullptr) return GEMM_ERR_ALLOC;
  h->device = dev;
  h->sms = sms;
  for (auto& per_mode : h->sk_active)
    for (int& n : per_mode) n = -1;
  const size_t status_bytes = (kSkCntOffset + dgt::kSimtInlineMaxTiles) * sizeof(int);
  if (cudaMalloc(&h->d_status, status_bytes) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return GEMM_ERR_ALLOC;
  }
  if (cudaMemset(h->d_status, 0, status_bytes) != cudaSuccess) {
    cudaFree(h->d_status);
    delete h;
    return GEMM_ERR_CUDA;
  }
  h->tma_cache = new (std::nothrow) dgt::TmaCache();
  if (h->tma_cache == nullptr) {
    cudaFree(h->d_status);
    delete h;
    return GEMM_ERR_ALLOC;
  }
  *out = h;
  return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_handle_t h) {
  if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
  int prev = 0;
  cudaGetDevice(&prev);
  cudaSetDevice(h->device);
  gemm_status_t st = cuda_status(cudaDeviceSynchronize());
  if (h->ws) cudaFree(h->ws);
  if (h->ws_t) cudaFree(h->ws_t);
  if (h->d_status) cudaFree(h->d_status);
  delete h->tma_cache;
  cudaSetDevice(prev);
  delete h;
  return st;
}

gemm_status_t gemm_validate(int mode, int transA, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                            const void* A, int64_t lda, const void* B, int64_t ldb, const float* C, int64_t ldc) {
  return check_args(mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc);
}

gemm_status_t gemm_run(gemm_handle_t h, int mode, int transA, int transB, int64_t M, int64_t N, int64_t K,
                       float alpha, const void* A, int64_t lda, const void* B, int64_t ldb, float beta, float* C,
                       int64_t ldc, void* stream) {
  if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
  gemm_status_t st = check_args(mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc);
  if (st != GEMM_OK) return st;
  dgt::last_main_launch().valid = false;
  st = run_checked(h, mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, dgt::EpiParams{},
                   static_cast<cudaStream_t>(stream));
  if (st == GEMM_OK) h->null_shape = dgt::last_main_launch();
  return st;
}

gemm_status_t gemm_run_epilogue(gemm_handle_t h, int mode, int transA, int transB, int64_t M, int64_t N, int64_t K,
                                float alpha, const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                                float* C, int64_t ldc, const gemm_epilogue_t* ep, void* stream) {
  if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
  gemm_status_t st = check_args(mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc);
  if (st != GEMM_OK) return st;
  dgt::EpiParams epi;
  if (ep != nullptr) {
    if (ep->activation < GEMM_ACT_NONE || ep->activation > GEMM_ACT_DGELU) return GEMM_ERR_INVALID_VALUE;
    if (ep->activation == GEMM_ACT_DGELU) {
      if (ep->bias != nullptr || ep->aux == nullptr || ep->ld_aux < std::max<int64_t>(N, 1))
        return GEMM_ERR_INVALID_VALUE;
      if (!aligned(ep->aux, 4)) return GEMM_ERR_MISALIGNED;
      epi.aux = ep->aux;
      epi.ld_aux = ep->ld_aux;
    }
    if (ep->bias != nullptr && !aligned(ep->bias, 4)) return GEMM_ERR_MISALIGNED;
    epi.act = ep->activation;
    epi.bias = ep->bias;
  }
  dgt::last_main_launch().valid = false;
  st = run_checked(h, mode, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, epi,
                   static_cast<cudaStream_t>(stream));
  if (st == GEMM_OK) h->null_shape = dgt::last_main_launch();
  return st;
}

gemm_status_t gemm_launch_null(gemm_handle_t h, void* stream) {
  if (h == nullptr || !h->null_shape.valid) return GEMM_ERR_INVALID_VALUE;
  return cuda_status(dgt::launch_null(h->null_shape, static_cast<cudaStream_t>(stream)));
}


gemm_status_t gemm_set_option(gemm_handle_t h, int option, int64_t value) {
  if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
  switch (option) {
    case GEMM_OPT_FAMILY:
      if (value < GEMM_FAMILY_AUTO || value > GEMM_FAMILY_SKINNY) return GEMM_ERR_INVALID_VALUE;
      h->opt_family = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_SPLIT_K:
      if (value < 0 || value > 4096) return GEMM_ERR_INVALID_VALUE;
      h->opt_split_k = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_TILE_N:
      if (value != 0 && value != 128 && value != 192 && value != 224 && value != 256) return GEMM_ERR_INVALID_VALUE;
      h->opt_tile_n = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_PRETRANSPOSE:
      if (value < 0 || value > 2) return GEMM_ERR_INVALID_VALUE;
      h->opt_pretranspose = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_PAIR:
      if (value < 0 || value > 1) return GEMM_ERR_INVALID_VALUE;
      h->opt_pair = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_WAIT_LIMIT_US:
      if (value < 0 || value > 60000000) return GEMM_ERR_INVALID_VALUE;
      h->opt_wait_us = value;
      return GEMM_OK;
    case GEMM_OPT_FAULT_SKIP_STAGE:
      if (value < 0 || value > (int64_t(1) << 30)) return GEMM_ERR_INVALID_VALUE;
      h->opt_fault_skip = static_cast<int>(value);
      return GEMM_OK;
    case GEMM_OPT_SK_FIXUP:
      if (value < 0 || value > 2) return GEMM_ERR_INVALID_VALUE;
      h->opt_sk_fixup = static_cast<int>(value);
      return GEMM_OK;
    default:
      return GEMM_ERR_INVALID_VALUE;
  }
}

gemm_status_t gemm_get_plan(gemm_handle_t h, gemm_plan_t* out) {
  if (h == nullptr || out == nullptr) return GEMM_ERR_INVALID_VALUE;
  *out = h->plan;
  return GEMM_OK;
}

gemm_status_t gemm_run_block_scaled(gemm_handle_t h, int mode, int64_t M, int64_t N, int64_t K, float alpha,
                                    const void* A, int64_t lda, const void* SA, const void* B, int64_t ldb,
                                    const void* SB, float beta, float* C, int64_t ldc, void* stream) {
  if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
  if (mode != GEMM_MODE_MXFP8_E4M3 && mode != GEMM_MODE_MXFP8_E5M2 && mode != GEMM_MODE_NVFP4)
    return GEMM_ERR_INVALID_VALUE;
  if (M < 0 || N < 0 || K < 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return GEMM_OK;
  if (C == nullptr || ldc < std::max<int64_t>(N, 1)) return GEMM_ERR_INVALID_VALUE;
  if (!aligned(C, 4)) return GEMM_ERR_MISALIGNED;
  const bool nvfp4 = mode == GEMM_MODE_NVFP4;
  if (K > 0 && alpha != 0.f) {
    if (A == nullptr || B == nullptr || SA == nullptr || SB == nullptr) return GEMM_ERR_INVALID_VALUE;
    if (lda < K || ldb < K) return GEMM_ERR_INVALID_VALUE;
    if (nvfp4 && (K % 2 != 0 || lda % 2 != 0 || ldb % 2 != 0)) return GEMM_ERR_INVALID_VALUE;
    // the TMA unit and the bulk copies read everything in place
    const int64_t lda_b = nvfp4 ? lda / 2 : lda, ldb_b = nvfp4 ? ldb / 2 : ldb;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(SA, 16) || !aligned(SB, 16) || lda_b % 16 != 0 ||
        ldb_b % 16 != 0)
      return GEMM_ERR_MISALIGNED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dgt::last_main_launch().valid = false;
  gemm_status_t st;
  if (K == 0 || alpha == 0.f) {
    st = dgt::launch_scale(M, N, C, ldc, beta, dgt::EpiParams{}, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
    if (st == GEMM_OK) set_plan(h, 0, 0, 0, 0, 1, 0, 0, 1, 0);
  } else {
    st = run_block_scaled(h, mode, M, N, K, alpha, A, lda, SA, B, ldb, SB, beta, C, ldc, s);
  }
  if (st == GEMM_OK) h->null_shape = dgt::last_main_launch();
  return st;
}

gemm_status_t gemm_attention_forward(gemm_handle_t h, int64_t problems, int64_t T, int64_t Dh, int causal,
                                     float scale, const void* Q, const void* K, const void* V, float* O,
                                     void* stream) {
  if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
  if (problems < 0 || T < 0 || Dh < 1 || (causal != 0 && causal != 1) || !std::isfinite(scale))
    return GEMM_ERR_INVALID_VALUE;
  if (Dh != 64) return GEMM_ERR_NOT_SUPPORTED;
  if (problems == 0 || T == 0) return GEMM_OK;
  if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return GEMM_ERR_INVALID_VALUE;
  // one CTA per (problem, 128 queries) in a 1-D grid; TMA extents below 2^31
  if (T > kMaxDim || problems > kMaxDim || problems * ceil_div(T, 128) > INT32_MAX) return GEMM_ERR_INVALID_VALUE;
  if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return GEMM_ERR_MISALIGNED;
  dgt::AttnArgs a{};
  a.problems = problems;
  a.T = T;
  a.causal = causal;
  a.scale = scale;
  a.Q = Q;
  a.K = K;
  a.V = V;
  a.O = O;
  a.status = h->d_status;
  a.wait_ns = static_cast<uint64_t>(h->opt_wait_us) * 1000u;
  a.sms = h->sms;
  dgt::last_main_launch().valid = false;
  if (dgt::launch_attention(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_CUDA;
  set_plan(h, GEMM_FAMILY_ATTENTION, 128, 128, 64, 1, 2, dgt::attention_grid(problems, T, h->sms), 1, 0);
  h->null_shape = dgt::last_main_launch();
  return GEMM_OK;
}

int64_t gemm_block_scales_tiled_bytes(int64_t rows, int64_t blocks) {
  if (rows < 0 || blocks < 0 || rows > kMaxDim || blocks > kMaxDim) return -1;
  return ceil_div(rows, 128) * dgt::block_scale_groups(blocks) * 512;
}

gemm_status_t gemm_block_scales_tile(int64_t rows, int64_t blocks, const void* S, int64_t lds, void* T,
                                     void* stream) {
  if (rows < 0 || blocks < 0 || rows > kMaxDim || blocks > kMaxDim) return GEMM_ERR_INVALID_VALUE;
  if (rows == 0 || blocks == 0) return GEMM_OK;
  if (S == nullptr || T == nullptr || lds < blocks) return GEMM_ERR_INVALID_VALUE;
  if (!aligned(T, 16)) return GEMM_ERR_MISALIGNED;
  return cuda_status(dgt::launch_block_scales_tile(static_cast<const uint8_t*>(S), rows, blocks, lds,
                                                   static_cast<uint8_t*>(T), static_cast<cudaStream_t>(stream)));
}

gemm_status_t gemm_check_device(gemm_handle_t h, void* stream) {
  if (h == nullptr) return GEMM_ERR_INVALID_VALUE;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, h->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
  if (v != 0) {
    if (cudaMemset(h->d_status, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_ERR_DEVICE_TIMEOUT;
  }
  return GEMM_OK;
}

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE";
    case GEMM_ERR_NOT_SUPPORTED: return "GEMM_ERR_NOT_SUPPORTED";
    case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_ALLOC: return "GEMM_ERR_ALLOC";
    case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT";
    case GEMM_ERR_TOO_LARGE: return "GEMM_ERR_TOO_LARGE";
    default: return "GEMM_ERR_UNKNOWN";
  }
}

}  // extern "C"
