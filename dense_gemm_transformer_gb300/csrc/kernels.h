// kernels.h -- host-side launch entry points of the library's kernels (internal).
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

namespace dgt {

// Runs `set_up` (a kernel's attribute set-up) once per device: `done` holds
// one bit per device that has been set up (devices 0-63; others always run
// it).
template <typename F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, F&& set_up) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return set_up();
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t(1) << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  const cudaError_t e = set_up();
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// TMA descriptors encoded for earlier calls of a handle, keyed by every
// argument of the encoding (a descriptor holds only the base pointer, the
// sizes, the strides and the box, so an entry stays valid for equal keys).
// Direct-mapped; a handle is used from one thread at a time.
struct TmaCache {
  static constexpr int kEntries = 64;
  struct alignas(64) Entry {
    CUtensorMap map;
    int64_t key[8];
    bool valid;
  };
  Entry entry[kEntries];
};

// Every kernel of the library is launched with programmatic dependent
// launch: it may start (and run its set-up, which touches no global memory)
// while the previous kernel in the stream is finishing; each kernel executes
// griddepcontrol.wait before its first access to global memory, which
// returns once every earlier kernel in the stream has completed and its
// writes are visible, so stream order is kept.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// The elementwise epilogue of gemm_run_epilogue (activation as
// gemm_activation_t): applied to alpha * product + beta * C at the final
// store of each element, in the caller's (row, column) coordinates.
enum { kActNone = 0, kActGelu = 1, kActDGelu = 2 };
struct EpiParams {
  int act = kActNone;
  const float* bias = nullptr;  // N floats, or null
  const float* aux = nullptr;   // DGELU: the M x N pre-activation
  int64_t ld_aux = 0;
};

// The launch configuration of the main GEMM kernel most recently launched
// from this host thread (the SIMT, tcgen05 or small-M kernel of a call, not
// its transposes, re-packs or reductions).
struct LaunchShape {
  dim3 grid, block;
  size_t smem = 0;
  int cluster = 1;  // CTAs per cluster along x
  bool valid = false;
};
LaunchShape& last_main_launch();
// An empty kernel with that configuration and programmatic dependent launch:
// the launch, placement and exit cost of the configuration without its work.
cudaError_t launch_null(const LaunchShape& l, cudaStream_t stream);

// ---------------------------------------------------------------- FP32 SIMT
// C = alpha * op(A) op(B) + beta * C with FFMA, 128 x tile_n block tiles
// (tile_n 128: two CTAs per SM; 256: one), in one of three schedules:
//   kSimtTiles   one CTA per output tile (2-D grid);
//   kSimtSplitK  one CTA per (tile, K slice); slice s (k_per_split elements, a
//                multiple of 16) writes raw partial sums to ws + s * M * ws_ld
//                and launch_splitk_reduce finishes;
//   kSimtStreamK `grid` persistent CTAs share the `iters` (tile, k-tile)
//                iterations evenly; partial tiles go to 2 * grid slots of
//                128 x tile_n floats at ws, and launch_simt also launches the
//                fixup kernel that sums them in a fixed order.
enum { kSimtTiles = 0, kSimtSplitK = 1, kSimtStreamK = 2 };
struct SimtArgs {
  int transA, transB;
  int64_t M, N, K;
  const float* A;
  int64_t lda;
  const float* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
  float alpha, beta;
  int tile_n;
  int schedule;
  int splits;
  int64_t k_per_split;
  int64_t dp_tiles;  // stream-K: leading tiles processed whole, round-robin over the grid
  int64_t iters;     // stream-K: (tile, k-tile) iterations of the tiles from dp_tiles on
  int64_t grid;
  float* ws;
  int64_t ws_ld;
  // stream-K: 1 when the last CTA to store a partial of a tile sums the
  // tile's partials itself (no fixup kernel); sk_cnt then holds one arrival
  // counter per tile from dp_tiles on, zero between calls.
  int sk_inline;
  int* sk_cnt;
};
constexpr int kSimtTileM = 128, kSimtTileN = 128, kSimtTileK = 16, kSimtThreads = 256;
constexpr int kSimtInlineMaxTiles = 1024;  // arrival counters a handle keeps
int64_t simt_streamk_slot_floats(int tile_n);  // floats per stream-K partial slot
cudaError_t launch_simt(const SimtArgs& a, cudaStream_t stream);

// ---------------------------------------------------------------- tcgen05
// Persistent TMA + tcgen05 kernel: one 128 x tile_n output tile per work unit,
// an smem ring fed by a TMA producer warp, a single-thread MMA issuer with a
// double-buffered TMEM accumulator, and four epilogue warps.
struct TcArgs {
  int mode;              // 1 = tf32, 2 = bf16, 3 = 8-bit floats (formats in fmt8)
  uint32_t fmt8;         // mode 3: the A and B formats of the kernel's operands, as instruction
                         // descriptor bits (fp8_format_bits); 0 otherwise
  int a_mn_major;        // A stored with M contiguous (transA == 1)
  int b_mn_major;        // B stored with N contiguous (transB == 0)
  int tile_n;            // 128, 192, 224 or 256 (16: the swapped small-M form)
  int pair;              // tile_n >= 192: two-CTA clusters issuing one MMA of 256 rows per pair
                         // (tcgen05 cta_group::2), each CTA staging half of every B tile
  int64_t M, N, K;
  const void* A;         // base of the (possibly re-packed) operand
  int64_t lda;           // elements
  const void* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
  float alpha, beta;
  int splits;            // slices of K; > 1 writes partials to ws
  int kb_per_split;      // k blocks per slice
  int dp_units;          // whole tiles (rows of units below tail_tm0) computed before the split units
  int tail_tm0;          // first row of units (pairs of tile rows for pairs) that is cut into K slices
  int64_t ws_row0;       // C row that workspace row 0 holds (tail_tm0's first row; 0 for plain split-K)
  float* ws;
  int64_t ws_ld;
  int64_t ws_slice;      // elements between successive K slices' partial sums
  int* status;           // device status word
  int grid;              // persistent CTAs
  int group_m;           // raster group height in M tiles
  TmaCache* tma_cache;   // the handle's descriptor cache (null: encode every call)
  EpiParams epi;         // with fuse_epi: the elementwise epilogue, applied to whole tiles in the kernel
  bool fuse_epi;         // run the kernel built with the fused epilogue (tc_epi_ok)
  uint64_t wait_ns;      // limit of every bounded wait (0: the default, kWaitLimitNs)
  int fault_skip;        // test hook: n > 0 makes CTA 0's producer issue no copies for its n-th stage
                         // (one CTA per tile only); 0: none
  const uint8_t* sfa;    // block-scaled small-M modes (4, 5): the kernel's A (weights) scales, tiled
  const uint8_t* sfb;    // ... and its B (activations) scales, tiled
  int64_t sf_groups;     // 512-byte scale atoms per 128-row tile
};
// tile_n == 16 selects the swapped small-M form: the caller passes the
// operands exchanged (C^T = op(B)^T op(A)^T, M and N exchanged) and the
// kernel stores its tile transposed into the caller's C.
constexpr int kTcEpiWarps = 8;                        // epilogue warps (two per TMEM lane quarter)
constexpr int kTcEpiWarpsEpi = 12;                    // the same in the builds with the fused epilogue
// The A / B format fields (bits 7-9 / 10-12) of a kind::f8f6f4 instruction
// descriptor: 0 = E4M3, 1 = E5M2.
constexpr uint32_t fp8_format_bits(uint32_t a_fmt, uint32_t b_fmt) { return (a_fmt << 7) | (b_fmt << 10); }
int tc_tile_k(int mode);              // k elements per stage (128 bytes)
// Whether the kernel is built with the fused epilogue for these operand
// layouts (as the kernel reads them, after any transpose): TF32 or BF16
// with a K-major A, and a K-major B in TF32; tiles of 128-256 columns.
bool tc_epi_ok(int mode, bool a_mn_major, bool b_mn_major);
int tc_stages(int mode, int tile_n, bool pair, bool epi = false);  // pipeline depth (pair: one 256-row MMA per CTA pair; epi: the fused-epilogue build)
// Whether the kernel is built for this tile width, pairing and B layout
// (tile_n 128, 192, 224 or 256; pairs from 192 columns).
bool tc_tile_ok(int mode, int tile_n, bool pair, bool b_mn_major);
cudaError_t launch_tc(const TcArgs& a, cudaStream_t stream);
// The small-M kernel (tile_n 16, operands swapped as for launch_tc): one
// (tile, K slice) per CTA, `splits` K slices per cluster reduced in
// distributed shared memory (ws and group_m unused), grid = tiles
// * splits.
cudaError_t launch_skinny(const TcArgs& a, cudaStream_t stream);
cudaError_t tc_init_driver();         // resolves cuTensorMapEncodeTiled once
// The resolved cuTensorMapEncodeTiled (null until tc_init_driver succeeded).
PFN_cuTensorMapEncodeTiled_v12000 tc_encoder();

// ---------------------------------------------------------------- attention
// Fused scaled dot-product attention forward over `problems` independent
// (batch element, head) problems: Q, K, V bf16 [problems][T][64] (rows of 64
// contiguous elements, 16-byte aligned), O fp32 of the same shape.  A
// persistent grid of two CTAs per SM takes the (problem, 128 queries) items
// in turn; scores stay in tensor memory.
struct AttnArgs {
  int64_t problems, T;
  int causal;
  float scale;
  const void *Q, *K, *V;
  float* O;
  int* status;       // device status word (bounded waits)
  uint64_t wait_ns;  // 0: kWaitLimitNs
  int sms;           // the device's SMs (the persistent grid: two CTAs per SM)
};
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);
int attention_grid(int64_t problems, int64_t T, int sms);  // CTAs launch_attention starts

// ---------------------------------------------------------------- helpers
// C = epi(alpha * sum_s ws[s] + beta * C) over an M x N matrix (s
// ascending); row0 is the caller's row of the matrix's first row (for the
// epilogue's Z).
cudaError_t launch_splitk_reduce(int64_t M, int64_t N, int splits, const float* ws, int64_t ws_ld,
                                 float* C, int64_t ldc, float alpha, float beta, const EpiParams& epi, int64_t row0,
                                 cudaStream_t stream);
// C = epi(beta * C) (beta == 0 writes epi(0) without reading C).
cudaError_t launch_scale(int64_t M, int64_t N, float* C, int64_t ldc, float beta, const EpiParams& epi,
                         cudaStream_t stream);
// C = epi(C) in place over an M x N matrix: the epilogue of a call whose
// GEMM kernels have stored alpha * product + beta * C.
cudaError_t launch_epilogue(int64_t M, int64_t N, float* C, int64_t ldc, const EpiParams& epi, cudaStream_t stream);
// Block scale factors (one byte per (row, block), row-major with leading
// dimension lds bytes) into the tiled layout the block-scaled kernels read:
// for each 128-row tile, groups of 4 blocks as 512-byte atoms, row r of the
// tile and block j of the group at byte 16 * (r % 32) + 4 * (r / 32) + j;
// groups_per_tile = 4 * ceil(blocks / 16); bytes past the matrix are zero.
cudaError_t launch_block_scales_tile(const uint8_t* S, int64_t rows, int64_t blocks, int64_t lds, uint8_t* T,
                                     cudaStream_t stream);
inline int64_t block_scale_groups(int64_t blocks) { return 4 * ((blocks + 15) / 16); }

// Copy a rows x cols matrix of elem_bytes-sized elements to dst with a new
// leading dimension (elements).
cudaError_t launch_pack(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows, int64_t cols,
                        int elem_bytes, cudaStream_t stream);

// dst (cols x rows, leading dimension ld_dst) = transpose of src (rows x cols).
cudaError_t launch_transpose(const void* src, int64_t ld_src, void* dst, int64_t ld_dst, int64_t rows, int64_t cols,
                             int elem_bytes, cudaStream_t stream);

}  // namespace dgt
