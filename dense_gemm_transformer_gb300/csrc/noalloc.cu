// noalloc.cu -- gemm_run_small_m_noalloc: the small-M (decode-shaped) product
// of gemm_run, for callers that cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not available or not
// allowed -- a host that hands the library pre-allocated buffers and owns
// every allocation itself (an inference runtime with its own pool, a plug-in
// loaded into another process's CUDA context, a latency-critical loop that
// must not call into the allocator).  gemm_run cannot serve them: its handle
// allocates a status word at creation and a workspace on first use.
//
// This entry point runs the persistent tcgen05 kernel in its swapped
// small-M form (C^T = B^T A^T) and, when K is split, the separate slice-sum
// kernel, with every piece of scratch they need -- the device status word
// and the split-K partial sums -- in one fixed array compiled into the
// library.  (gemm_run serves the same shapes with a different kernel, the
// cluster kernel that sums its K slices in distributed shared memory; the
// two agree within the mode's tolerance, not bit for bit.)  Nothing is
// allocated: no cudaMalloc, no cudaFree, no allocating library call.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "gemm.h"
#include "kernels.h"

namespace {

// The fixed scratch: 256 bytes for the device status word, the rest for
// split-K partial sums.  Every device that loads the library holds it until
// the process exits.
constexpr size_t kScratchBytes = GEMM_NOALLOC_SCRATCH_BYTES;
constexpr size_t kStatusBytes = 256;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// The device address of g_scratch per device.  In host code `g_scratch` is
// only a host-side stand-in for the symbol, never a device pointer, so the
// address is looked up once per device with that device current.
struct DeviceScratch {
  bool ready = false;
  unsigned char* base = nullptr;
  int sms = 0;
};
constexpr int kMaxDevices = 64;
DeviceScratch g_devices[kMaxDevices];
std::mutex g_setup_mutex;

gemm_status_t scratch_for_current_device(DeviceScratch* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_NOT_SUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceScratch& d = g_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_NOT_SUPPORTED;
    void* ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
    if (e != cudaSuccess || ptr == nullptr) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    d.base = static_cast<unsigned char*>(ptr);
    d.sms = sms;
    d.ready = true;
  }
  *out = d;
  return GEMM_OK;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t x, int64_t m) { return ceil_div(x, m) * m; }

// The K-slice count: the one whose (tile, slice) units fill whole waves of
// one CTA per SM best (at most 32 slices of at least two K blocks each).
int64_t planned_splits(int64_t tiles, int64_t kb, int sms) {
  int64_t best = 1;
  double best_eff = 0.0;
  const int64_t max_s = std::max<int64_t>(1, std::min<int64_t>(32, kb / 2));
  for (int64_t s = 1; s <= max_s; ++s) {
    const int64_t per = ceil_div(kb, s);
    if (ceil_div(kb, per) != s) continue;
    const int64_t units = tiles * s;
    const double eff = static_cast<double>(units) / (ceil_div(units, sms) * sms);
    if (eff > best_eff + 0.02) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

bool tma_readable(const void* p, int64_t ld, int es) {
  return (reinterpret_cast<uintptr_t>(p) % 16) == 0 && (ld * es) % 16 == 0;
}

}  // namespace

extern "C" gemm_status_t gemm_run_small_m_noalloc(int mode, int transB, int64_t M, int64_t N, int64_t K, float alpha,
                                                  const void* A, int64_t lda, const void* B, int64_t ldb, float beta,
                                                  float* C, int64_t ldc, void* stream) {
  // The same argument checks as gemm_run (A stored M x K, transA == 0).
  gemm_status_t st = gemm_validate(mode, 0, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc);
  if (st != GEMM_OK) return st;
  if (mode != GEMM_MODE_TF32 && mode != GEMM_MODE_BF16) return GEMM_ERR_NOT_SUPPORTED;
  if (M > 16) return GEMM_ERR_TOO_LARGE;
  DeviceScratch d;
  st = scratch_for_current_device(&d);
  if (st != GEMM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0 || N == 0) return GEMM_OK;
  if (K == 0 || alpha == 0.f)
    return dgt::launch_scale(M, N, C, ldc, beta, dgt::EpiParams{}, s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;

  // Both operands must be readable in place by the TMA unit: nothing is
  // re-packed here.  kind::tf32 takes K-major operands only, so TF32 weights
  // must be stored N x K (transB == 1).
  const int es = (mode == GEMM_MODE_BF16) ? 2 : 4;
  if (!tma_readable(A, lda, es) || !tma_readable(B, ldb, es)) return GEMM_ERR_MISALIGNED;
  if (mode == GEMM_MODE_TF32 && transB == 0) return GEMM_ERR_NOT_SUPPORTED;

  // Split-K partials go to the array after the status word; fewer slices are
  // used if the planner's count would not fit.
  const int bk = dgt::tc_tile_k(mode);
  const int64_t tiles = ceil_div(N, 128);
  const int64_t kb = ceil_div(K, bk);
  const int64_t ws_ld = round_up(N, 4);
  const int64_t slice_bytes = M * ws_ld * static_cast<int64_t>(sizeof(float));
  int64_t splits = (tiles >= 2 * d.sms) ? 1 : planned_splits(tiles, kb, d.sms);
  const int64_t room = static_cast<int64_t>(kScratchBytes - kStatusBytes);
  while (splits > 1 && splits * slice_bytes > room) --splits;  // one slice needs no partial sums
  const int64_t kb_per = ceil_div(kb, splits);
  splits = ceil_div(kb, kb_per);  // never more slices than chosen above

  // The status word must start at zero on every call; partial sums are fully
  // overwritten before they are read, so they need no clearing.
  int* status = reinterpret_cast<int*>(d.base);
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return GEMM_ERR_CUDA;

  dgt::TcArgs a{};
  a.mode = mode;
  a.a_mn_major = transB ? 0 : 1;  // the weights are the kernel's 128-row operand
  a.b_mn_major = 0;               // the activations, K-major
  a.tile_n = 16;
  a.M = N;
  a.N = M;
  a.K = K;
  a.A = B;
  a.lda = ldb;
  a.B = A;
  a.ldb = lda;
  a.C = C;
  a.ldc = ldc;
  a.alpha = alpha;
  a.beta = beta;
  a.splits = static_cast<int>(splits);
  a.kb_per_split = static_cast<int>(kb_per);
  a.ws = splits > 1 ? reinterpret_cast<float*>(d.base + kStatusBytes) : nullptr;
  a.ws_ld = ws_ld;
  a.ws_slice = M * ws_ld;
  a.status = status;
  a.grid = static_cast<int>(std::min<int64_t>(tiles * splits, d.sms));
  a.group_m = 16;
  if (dgt::launch_tc(a, s) != cudaSuccess) return GEMM_ERR_CUDA;
  if (splits > 1 &&
      dgt::launch_splitk_reduce(M, N, a.splits, a.ws, ws_ld, C, ldc, alpha, beta, dgt::EpiParams{}, 0, s) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return GEMM_OK;
}

extern "C" gemm_status_t gemm_noalloc_check_device(void* stream) {
  // Like gemm_check_device, for the fixed array's status word: nothing is
  // allocated (the word is copied into a local variable and cleared in place).
  DeviceScratch d;
  gemm_status_t st = scratch_for_current_device(&d);
  if (st != GEMM_OK) return st;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return GEMM_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, d.base, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
  if (v != 0) {
    if (cudaMemset(d.base, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_ERR_DEVICE_TIMEOUT;
  }
  return GEMM_OK;
}
