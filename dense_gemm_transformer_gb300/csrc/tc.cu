// tc.cu -- tensor-map encoding and launch of the tcgen05 kernel.
//
// The TMA descriptors are encoded on the host with cuTensorMapEncodeTiled,
// obtained through the runtime's driver entry-point query so that the library
// needs no link-time dependency on the driver library.  Operand boxes are 128
// bytes wide along the contiguous dimension with the 128-byte swizzle, the
// layout the shared-memory descriptors of the kernel expect:
//   K-major operand (K contiguous):   box {BK, rows}    one box per stage
//   MN-major operand (M/N contiguous): box {CH, BK}     rows/CH boxes per stage
// Out-of-range rows and columns of a box are filled with zeros by the TMA unit.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "skinny.cuh"
#include "tc_launch.cuh"

namespace dgt {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

cudaError_t encode_2d(CUtensorMap* m, int mode, const void* ptr, int64_t inner, int64_t outer, int64_t ld,
                      uint32_t box_inner, uint32_t box_outer) {
  const int es = (mode >= 3) ? 1 : (mode == 2) ? 2 : 4;
  const CUtensorMapDataType dt = (mode >= 3)   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : (mode == 2) ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The fp32 output (C, or the split-K partial sums as S slices of M x N) as a
// 3-D map for the epilogue's TMA stores: box of 32 columns x 32 rows x 1 slice.
cudaError_t encode_out(CUtensorMap* m, float* ptr, int64_t N, int64_t M, int64_t S, int64_t ld, int64_t slice) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(S)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 4, static_cast<cuuint64_t>(slice) * 4};
  cuuint32_t box[3] = {32, 32, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// encode_2d / encode_out through the handle's cache (kind 0 / 1 in the key).
cudaError_t cached(TmaCache* cache, CUtensorMap* m, const int64_t (&key)[8], cudaError_t (*encode)(CUtensorMap*,
                                                                                            const int64_t (&)[8])) {
  if (cache == nullptr) return encode(m, key);
  uint64_t h = 1469598103934665603ull;
  for (int64_t k : key) h = (h ^ static_cast<uint64_t>(k)) * 1099511628211ull;
  TmaCache::Entry& e = cache->entry[(h >> 32) % TmaCache::kEntries];
  bool hit = e.valid;
  for (int i = 0; hit && i < 8; ++i) hit = e.key[i] == key[i];
  if (!hit) {
    const cudaError_t r = encode(&e.map, key);
    if (r != cudaSuccess) {
      e.valid = false;
      return r;
    }
    for (int i = 0; i < 8; ++i) e.key[i] = key[i];
    e.valid = true;
  }
  *m = e.map;
  return cudaSuccess;
}

cudaError_t encode_2d_key(CUtensorMap* m, const int64_t (&k)[8]) {
  return encode_2d(m, static_cast<int>(k[1]), reinterpret_cast<const void*>(k[0]), k[2], k[3], k[4],
                   static_cast<uint32_t>(k[5]), static_cast<uint32_t>(k[6]));
}

cudaError_t encode_out_key(CUtensorMap* m, const int64_t (&k)[8]) {
  return encode_out(m, reinterpret_cast<float*>(k[0]), k[2], k[3], k[4], k[5], k[6]);
}

cudaError_t encode_2d_c(TmaCache* cache, CUtensorMap* m, int mode, const void* ptr, int64_t inner, int64_t outer,
                        int64_t ld, uint32_t box_inner, uint32_t box_outer) {
  const int64_t key[8] = {static_cast<int64_t>(reinterpret_cast<uintptr_t>(ptr)), mode, inner, outer, ld,
                          box_inner, box_outer, 0};
  return cached(cache, m, key, encode_2d_key);
}

cudaError_t encode_out_c(TmaCache* cache, CUtensorMap* m, float* ptr, int64_t N, int64_t M, int64_t S, int64_t ld,
                         int64_t slice) {
  const int64_t key[8] = {static_cast<int64_t>(reinterpret_cast<uintptr_t>(ptr)), 256 + 1, N, M, S, ld, slice, 1};
  return cached(cache, m, key, encode_out_key);
}

}  // namespace

cudaError_t tc_init_driver() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) {
      g_encode_status = (e != cudaSuccess) ? e : cudaErrorNotSupported;
      return;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode_status;
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encoder() { return g_encode; }

int tc_tile_k(int mode) { return mode >= 3 ? 128 : mode == 2 ? 64 : 32; }

bool tc_epi_ok(int mode, bool a_mn_major, bool b_mn_major) {
  if (a_mn_major) return false;
  return mode == 2 || (mode == 1 && !b_mn_major);
}

namespace {
template <int EW>
int tc_stages_for(int tile_n, bool pair) {
  if (tile_n == 256 && pair) return TcCfg<2, 256, true, EW>::STAGES;
  if (tile_n == 224 && pair) return TcCfg<2, 224, true, EW>::STAGES;
  if (tile_n == 192 && pair) return TcCfg<2, 192, true, EW>::STAGES;
  if (tile_n == 256) return TcCfg<2, 256, false, EW>::STAGES;
  if (tile_n == 224) return TcCfg<2, 224, false, EW>::STAGES;
  if (tile_n == 192) return TcCfg<2, 192, false, EW>::STAGES;
  if (tile_n == 128) return TcCfg<2, 128, false, EW>::STAGES;
  return TcCfg<2, 16, false, EW>::STAGES;
}
}  // namespace

int tc_stages(int mode, int tile_n, bool pair, bool epi) {
  // a stage holds 128 bytes of K per row in every mode; the block-scaled
  // modes add their scale atoms to it; the builds with the fused epilogue
  // stage the stores of more epilogue warps
  if (mode == 4) return tile_n == 128 ? TcCfg<4, 128>::STAGES : TcCfg<4, 16>::STAGES;
  if (mode == 5) return tile_n == 128 ? TcCfg<5, 128>::STAGES : TcCfg<5, 16>::STAGES;
  return epi ? tc_stages_for<kTcEpiWarpsEpi>(tile_n, pair) : tc_stages_for<kTcEpiWarps>(tile_n, pair);
}

bool tc_tile_ok(int mode, int tile_n, bool pair, bool b_mn_major) {
  if (mode < 1 || mode > 3) return false;
  if (tile_n != 128 && tile_n != 192 && tile_n != 224 && tile_n != 256) return false;
  if (pair && tile_n == 128) return false;
  if (!b_mn_major) return true;
  if (mode != 2) return false;  // kind::tf32 and the FP8 build: K-major operands only
  const int ch = 64;            // bf16 columns in one 128-byte chunk
  return tile_n % ch == 0 && (!pair || (tile_n / ch) % 2 == 0);
}

cudaError_t launch_tc(const TcArgs& a, cudaStream_t stream) {
  if (a.mode < 1 || a.mode > 5) return cudaErrorInvalidValue;
  if (a.mode >= 4 && ((a.tile_n != 16 && a.tile_n != 128) || a.pair || a.a_mn_major || a.b_mn_major))
    return cudaErrorInvalidValue;
  cudaError_t e = tc_init_driver();
  if (e != cudaSuccess) return e;
  const int bk = tc_tile_k(a.mode);
  const int ch = 128 / ((a.mode >= 3) ? 1 : (a.mode == 2) ? 2 : 4);  // elements in a 128-byte MN-major row
  CUtensorMap ta, tb;
  e = a.a_mn_major ? encode_2d_c(a.tma_cache, &ta, a.mode, a.A, a.M, a.K, a.lda, ch, bk)
                   : encode_2d_c(a.tma_cache, &ta, a.mode, a.A, a.K, a.M, a.lda, bk, 128);
  if (e != cudaSuccess) return e;
  // Each CTA of a pair loads one half of each B tile (K-major: half the
  // rows), and the pair issues one MMA of 256 rows over both CTAs.
  const bool pair = a.tile_n >= 192 && a.pair;
  e = a.b_mn_major ? encode_2d_c(a.tma_cache, &tb, a.mode, a.B, a.N, a.K, a.ldb, ch, bk)
                   : encode_2d_c(a.tma_cache, &tb, a.mode, a.B, a.K, a.N, a.ldb, bk, pair ? a.tile_n / 2 : a.tile_n);
  if (e != cudaSuccess) return e;

  TcParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.K = static_cast<int>(a.K);
  p.num_tm = static_cast<int>((a.M + 127) / 128);
  if (pair) p.num_tm = (p.num_tm + 1) / 2;  // units are pairs of vertically adjacent tiles
  p.num_tn = static_cast<int>((a.N + a.tile_n - 1) / a.tile_n);
  p.num_kb = static_cast<int>((a.K + bk - 1) / bk);
  p.splits = a.splits;
  p.kb_per_split = a.kb_per_split;
  p.dp_units = a.dp_units;
  p.tail_tm0 = a.tail_tm0;
  p.num_units = a.dp_units + (p.num_tm - a.tail_tm0) * p.num_tn * a.splits;
  p.group_m = a.group_m;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.C = a.C;
  p.ldc = a.ldc;
  p.ws = a.ws;
  p.ws_ld = a.ws_ld;
  p.ws_slice = a.ws_slice;
  p.ws_row0 = a.ws_row0;
  p.status = a.status;
  p.fmt8 = (a.mode == 3 || a.mode == 4) ? a.fmt8 : 0u;
  p.sfa = a.sfa;
  p.sfb = a.sfb;
  p.sf_groups = a.sf_groups;
  // Block-scaled: the activations' scale atoms (SF_ATOMS per stage, the
  // same for every weight tile) are copied into TMEM once per CTA when they
  // fit its reserved columns, instead of with every stage.
  {
    const int per_kb = a.mode == 5 ? TcCfg<5, 16>::SF_ATOMS : a.mode == 4 ? TcCfg<4, 16>::SF_ATOMS : 0;
    const int64_t res = static_cast<int64_t>(p.num_kb) * per_kb;
    p.sfb_res = (a.tile_n == 16 && per_kb > 0 && a.sfb != nullptr && res <= TcCfg<5, 16>::RES_ATOMS &&
                 res <= a.sf_groups)
                    ? static_cast<int>(res)
                    : 0;
  }
  p.wait_ns = a.wait_ns > 0 ? a.wait_ns : kWaitLimitNs;
  p.epi = a.fuse_epi ? a.epi : EpiParams{};
  p.fault_skip = (a.fault_skip > 0 && !pair) ? a.fault_skip - 1 : -1;
  p.c_vec = ((reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && a.ldc % 4 == 0) ? 1 : 0;
  // Tiles leave through TMA stores when the destination allows it: not the
  // transposed small-M form, no read of C (beta == 0, or partial sums), and
  // 16-byte aligned rows.  Whole tiles go to C, partial tiles to the
  // workspace (its rows start at C row ws_row0).
  CUtensorMap tcm, twm;
  std::memset(&tcm, 0, sizeof tcm);
  std::memset(&twm, 0, sizeof twm);
  p.c_tma = 0;
  p.w_tma = 0;
  if (a.tile_n >= 128) {
    if (a.splits > 1)
      p.w_tma = (encode_out_c(a.tma_cache, &twm, a.ws, a.N, a.M - a.ws_row0, a.splits, a.ws_ld, a.ws_slice) ==
                 cudaSuccess)
                    ? 1
                    : 0;
    const bool whole = a.splits == 1 || a.dp_units > 0;
    if (whole && a.beta == 0.f && p.c_vec)
      p.c_tma = (encode_out_c(a.tma_cache, &tcm, a.C, a.N, a.M, 1, a.ldc, a.M * a.ldc) == cudaSuccess) ? 1 : 0;
  }
  // GELU' with C leaving through TMA stores and no partial tiles: Z's
  // blocks come in by TMA too, in the same boxes, through the workspace's
  // map slot (unused then), when Z's rows are 16-byte aligned.
  p.z_tma = 0;
  if (a.fuse_epi && a.epi.act == kActDGelu && p.c_tma && !p.w_tma && a.splits == 1 && a.epi.aux != nullptr &&
      (reinterpret_cast<uintptr_t>(a.epi.aux) & 15u) == 0 && a.epi.ld_aux % 4 == 0)
    p.z_tma = (encode_out_c(a.tma_cache, &twm, const_cast<float*>(a.epi.aux), a.N, a.M, 1, a.epi.ld_aux,
                            a.M * a.epi.ld_aux) == cudaSuccess)
                  ? 1
                  : 0;
  if (a.mode >= 4) return tc_launch_bs(a.mode, a.tile_n, ta, tb, tcm, twm, p, a.grid, stream);
  if (a.fuse_epi) {
    if (a.tile_n < 128 || !tc_epi_ok(a.mode, a.a_mn_major != 0, a.b_mn_major != 0)) return cudaErrorNotSupported;
    if (a.mode == 1)
      return tc_launch_tf32_epi(a.tile_n, pair, false, a.b_mn_major != 0, ta, tb, tcm, twm, p, a.grid, stream);
    if (a.tile_n == 192 || a.tile_n == 224)
      return tc_launch_bf16_epi_mid(a.tile_n, pair, false, a.b_mn_major != 0, ta, tb, tcm, twm, p, a.grid, stream);
    return tc_launch_bf16_epi(a.tile_n, pair, false, a.b_mn_major != 0, ta, tb, tcm, twm, p, a.grid, stream);
  }
  if (a.mode == 3 && (a.tile_n == 192 || a.tile_n == 224))
    return tc_launch_fp8_mid(a.tile_n, pair, a.a_mn_major != 0, a.b_mn_major != 0, ta, tb, tcm, twm, p, a.grid,
                             stream);
  if (a.mode == 3)
    return tc_launch_fp8(a.tile_n, pair, a.a_mn_major != 0, a.b_mn_major != 0, ta, tb, tcm, twm, p, a.grid, stream);
  if (a.mode == 2 && (a.tile_n == 192 || a.tile_n == 224))
    return tc_launch_bf16_mid(a.tile_n, pair, a.a_mn_major != 0, a.b_mn_major != 0, ta, tb, tcm, twm, p, a.grid,
                              stream);
  if (a.mode == 2)
    return tc_launch_bf16(a.tile_n, pair, a.a_mn_major != 0, a.b_mn_major != 0, ta, tb, tcm, twm, p, a.grid, stream);
  return tc_launch_tf32(a.tile_n, pair, a.a_mn_major != 0, a.b_mn_major != 0, ta, tb, tcm, twm, p, a.grid, stream);
}

cudaError_t launch_skinny(const TcArgs& a, cudaStream_t stream) {
  cudaError_t e = tc_init_driver();
  if (e != cudaSuccess) return e;
  const int bk = tc_tile_k(a.mode);
  const int ch = 128 / ((a.mode >= 3) ? 1 : (a.mode == 2) ? 2 : 4);
  CUtensorMap ta, tb;
  e = a.a_mn_major ? encode_2d_c(a.tma_cache, &ta, a.mode, a.A, a.M, a.K, a.lda, ch, bk)
                   : encode_2d_c(a.tma_cache, &ta, a.mode, a.A, a.K, a.M, a.lda, bk, 128);
  if (e != cudaSuccess) return e;
  if (a.b_mn_major) return cudaErrorInvalidValue;
  e = encode_2d_c(a.tma_cache, &tb, a.mode, a.B, a.K, a.N, a.ldb, bk, 16);
  if (e != cudaSuccess) return e;
  SkParams p;
  p.M = static_cast<int>(a.M);
  p.N = static_cast<int>(a.N);
  p.num_kb = static_cast<int>((a.K + bk - 1) / bk);
  p.kb_per = a.kb_per_split;
  p.cluster = a.splits;
  p.alpha = a.alpha;
  p.beta = a.beta;
  p.C = a.C;
  p.ldc = a.ldc;
  p.status = a.status;
  p.fmt8 = (a.mode == 3 || a.mode == 4) ? a.fmt8 : 0u;
  p.sfa = a.sfa;
  p.sfb = a.sfb;
  p.sf_groups = a.sf_groups;
  return skinny_launch(a.mode, a.a_mn_major != 0, ta, tb, p, a.grid, stream);
}

}  // namespace dgt
