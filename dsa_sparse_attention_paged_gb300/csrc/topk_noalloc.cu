// topk_noalloc.cu -- the histogram-driven top-k with its scratch memory in a
// fixed, library-owned device array, for callers that cannot allocate device
// memory themselves (see dsa_coarse_hist_topk_noalloc in include/dsa.h).
//
// The scratch is a file-scope __device__ array laid out exactly like a caller
// workspace sized for DSA_NOALLOC_MAX_ROWS rows; the regular select launcher
// runs on it unchanged, so rows of at most 131072 scores take the one-launch
// cluster select and longer rows the multi-CTA select, as with a workspace.
// Every GPU that loads the library keeps this array until the process exits.
#include <mutex>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {
namespace {

// Same byte layout as WsLayout::total(DSA_NOALLOC_MAX_ROWS): status header,
// per-row counters, candidates, histogram and fine histogram, each region
// rounded up to 256 bytes.
constexpr size_t kAlign256(size_t x) { return (x + 255) & ~(size_t)255; }
constexpr size_t kRows = DSA_NOALLOC_MAX_ROWS;
constexpr size_t kScratchBytes =
    kAlign256(kAlign256(kAlign256(kAlign256(256 + kRows * 16) + kRows * DSA_CAND_CAP * 8) +
                        kRows * DSA_NUM_BINS * 4) +
              kRows * 4096 * 4);

static __device__ __align__(256) unsigned char g_topk_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (host code cannot use the array's name as a device pointer).
void *scratch_on_current_device(dsa_status_t *err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    *err = DSA_ERR_CUDA;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {  // beyond the address table: not a CUDA failure
    *err = DSA_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_topk_scratch);
    if (e != cudaSuccess || p == nullptr) {
      record_cuda_error(e);
      *err = DSA_ERR_CUDA;
      return nullptr;
    }
    g_scratch_addr[dev] = p;
  }
  *err = DSA_OK;
  return g_scratch_addr[dev];
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" int32_t dsa_coarse_hist_topk_noalloc(const float *logits, int64_t stride,
                                                const int32_t *context_lens, int32_t next_n,
                                                int32_t len_div, int32_t R, int32_t *histogram,
                                                int32_t reset_histogram, int32_t k,
                                                int32_t *out_idx, int32_t *fallback_flags,
                                                void *stream) {
  if (R < 0 || next_n < 1 || len_div < 1 || stride < 1) return DSA_ERR_INVALID_ARG;
  if (R > DSA_NOALLOC_MAX_ROWS) return DSA_ERR_UNSUPPORTED;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (!logits || !context_lens || !out_idx) return DSA_ERR_INVALID_ARG;
  if (histogram && (reinterpret_cast<uintptr_t>(histogram) & 7) != 0) return DSA_ERR_MISALIGNED;
  if (R == 0) return DSA_OK;
  if (WsLayout::total(DSA_NOALLOC_MAX_ROWS) > kScratchBytes) return DSA_ERR_WORKSPACE;
  dsa_status_t err;
  void *ws = scratch_on_current_device(&err);
  if (!ws) return err;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left.  The kernels leave the
  // counters and histograms they use at zero when they finish, but a call
  // that never ran to the end (a wait that ran out, a launch that failed
  // after an earlier kernel of the call) would leave them dirty for every
  // later caller of the shared array.  So each call clears the status word,
  // the counters and both histograms of the rows it uses itself (three small
  // memsets, ~1.3 MB at 64 rows; the candidate buffer needs no clearing).
  char *base = static_cast<char *>(ws);
  const int64_t rows = DSA_NOALLOC_MAX_ROWS;
  cudaError_t e = cudaMemsetAsync(base, 0, WsLayout::counters_off() + (size_t)R * 16, st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(base + WsLayout::hist_off(rows), 0, (size_t)R * DSA_NUM_BINS * 4, st);
  if (e == cudaSuccess)
    e = cudaMemsetAsync(base + WsLayout::fine_off(rows), 0, (size_t)R * 4096 * 4, st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return DSA_ERR_CUDA;
  }
  TopkCall c{};
  c.logits = logits;
  c.stride = stride;
  c.context_lens = context_lens;
  c.next_n = next_n;
  c.len_div = len_div;
  c.R = R;
  c.histogram = histogram;
  c.reset_histogram = reset_histogram != 0;
  c.k = k;
  c.out_idx = out_idx;
  c.fallback_flags = fallback_flags;
  c.workspace = ws;
  c.ws_rows = DSA_NOALLOC_MAX_ROWS;
  return run_topk(c, st);
}
