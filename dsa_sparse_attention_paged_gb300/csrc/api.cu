// api.cu -- the extern "C" entry points declared in include/dsa.h: argument
// checks (all before any launch), workspace handling, tensor-map encoding and
// the small host utilities the kernels' launchers share.
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {

namespace {
thread_local int32_t g_last_cuda_error = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Workspace rows that fit in ws_bytes (the layout depends only on this, so
// every call on one workspace buffer uses the same offsets).
int64_t ws_rows_for(size_t ws_bytes) {
  if (ws_bytes < WsLayout::total(1)) return 0;
  int64_t lo = 1, hi = 1;
  while (WsLayout::total(hi * 2) <= ws_bytes && hi < (1LL << 30)) hi *= 2;
  lo = hi;
  hi = hi * 2;
  while (hi - lo > 1) {
    const int64_t mid = (lo + hi) / 2;
    if (WsLayout::total(mid) <= ws_bytes) lo = mid;
    else hi = mid;
  }
  return lo;
}

uint32_t *status_word(void *ws) {
  return reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + WsLayout::kStatusOff);
}
}  // namespace

void record_cuda_error(cudaError_t e) { g_last_cuda_error = static_cast<int32_t>(e); }

dsa_status_t check_launch() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  static std::mutex mu;
  static std::vector<std::pair<int, int>> cache;
  std::lock_guard<std::mutex> lk(mu);
  for (auto &c : cache)
    if (c.first == dev) return c.second;
  int n = 0;
  const cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return -1;
  }
  cache.emplace_back(dev, n);
  return n;
}

bool ensure_smem_attr(const void *fn, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  struct Entry {
    const void *fn;
    int dev;
    int bytes;
  };
  static std::mutex mu;
  static std::vector<Entry> done;
  std::lock_guard<std::mutex> lk(mu);
  for (auto &d : done)
    if (d.fn == fn && d.dev == dev && d.bytes >= bytes) return true;
  const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return false;
  }
  done.push_back({fn, dev, bytes});
  return true;
}

dsa_status_t make_tmap_rows128(CUtensorMap *map, const void *base, uint64_t rows,
                               uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return DSA_ERR_CUDA;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = static_cast<int32_t>(r);
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

dsa_status_t make_tmap_rows_e2m1(CUtensorMap *map, const void *base, uint64_t rows,
                                 uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return DSA_ERR_CUDA;
  const cuuint64_t dims[2] = {128, rows};  // in 4-bit elements
  const cuuint64_t strides[1] = {64};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(base),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    g_last_cuda_error = static_cast<int32_t>(r);
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

const char *dsa_status_string(int32_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_MISALIGNED: return "DSA_ERR_MISALIGNED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    default: return "DSA_ERR_UNKNOWN";
  }
}

int32_t dsa_last_cuda_error(void) { return g_last_cuda_error; }

int32_t dsa_version(void) { return 10000; }

size_t dsa_workspace_size(int32_t max_rows) {
  if (max_rows < 1) max_rows = 1;
  return WsLayout::total(max_rows);
}

int32_t dsa_workspace_init(void *workspace, size_t ws_bytes, void *stream) {
  if (!workspace) return DSA_ERR_INVALID_ARG;
  if (ws_bytes < WsLayout::kHeader) return DSA_ERR_WORKSPACE;
  const cudaError_t e =
      cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

int32_t dsa_read_device_status(const void *workspace, void *stream, uint32_t *out_host) {
  if (!workspace || !out_host) return DSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(out_host, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

static int32_t check_paged_common(const uint8_t *q, const uint8_t *kv, const float *kscale,
                                  const float *weights, const int32_t *page_table,
                                  int64_t pt_stride, const int32_t *ctx, int32_t B,
                                  int32_t next_n, int32_t H, int32_t D, int32_t ps,
                                  int32_t num_pages, const void *ws, size_t ws_bytes) {
  if (B < 0) return DSA_ERR_INVALID_ARG;
  if (next_n < 1 || next_n > 4) return DSA_ERR_UNSUPPORTED;
  if (H != 32 || D != 128) return DSA_ERR_UNSUPPORTED;
  if (ps != 64 && ps != 128) return DSA_ERR_UNSUPPORTED;
  if (num_pages < 1 || pt_stride < 1) return DSA_ERR_INVALID_ARG;
  if ((int64_t)num_pages * ps > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  if ((int64_t)B * next_n * 32 > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  if (!q || !kv || !kscale || !weights || !page_table || !ctx) return DSA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(kscale, 16) || !aligned(weights, 16))
    return DSA_ERR_MISALIGNED;
  if (!ws) return DSA_ERR_WORKSPACE;
  if (ws_bytes < WsLayout::kHeader) return DSA_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return DSA_ERR_MISALIGNED;
  return DSA_OK;
}

int32_t dsa_paged_mqa_logits(const uint8_t *q, const uint8_t *kv_pages, const float *kscale,
                             const float *weights, const int32_t *page_table,
                             int64_t page_table_stride, const int32_t *context_lens, int32_t B,
                             int32_t next_n, int32_t num_heads, int32_t head_dim,
                             int32_t page_size, int32_t num_pages, float *logits,
                             int64_t logits_stride, int32_t *histogram, float *amax,
                             int64_t amax_stride, int32_t amax_skip_if_blocks_le,
                             void *workspace, size_t ws_bytes, void *stream) {
  int32_t e = check_paged_common(q, kv_pages, kscale, weights, page_table, page_table_stride,
                                 context_lens, B, next_n, num_heads, head_dim, page_size,
                                 num_pages, workspace, ws_bytes);
  if (e != DSA_OK) return e;
  if (!logits || logits_stride < 1) return DSA_ERR_INVALID_ARG;
  if (histogram && !aligned(histogram, 8)) return DSA_ERR_MISALIGNED;
  if (amax && amax_stride < 1) return DSA_ERR_INVALID_ARG;
  if (B == 0) return DSA_OK;
  LogitsCall c{};
  c.q = q;
  c.kv = kv_pages;
  c.kscale = kscale;
  c.weights = weights;
  c.page_table = page_table;
  c.pt_stride = page_table_stride;
  c.context_lens = context_lens;
  c.B = B;
  c.next_n = next_n;
  c.page_size = page_size;
  c.num_pages = num_pages;
  c.out = logits;
  c.out_stride = logits_stride;
  c.histogram = histogram;
  c.amax = amax;
  c.amax_stride = amax_stride;
  c.amax_skip = amax_skip_if_blocks_le;
  c.sparse = false;
  c.out_fmt = DSA_OUT_F32;
  c.block_table = nullptr;
  c.kb = 0;
  c.status = status_word(workspace);
  c.wait_limit = kDefaultWaitLimit;
  return run_paged_logits(c, static_cast<cudaStream_t>(stream));
}

int32_t dsa_paged_mqa_logits_mx(const uint8_t *q, const uint8_t *k_codes, const uint8_t *k_exp,
                                const float *weights, const int32_t *page_table,
                                int64_t page_table_stride, const int32_t *context_lens, int32_t B,
                                int32_t next_n, int32_t num_heads, int32_t head_dim,
                                int32_t page_size, int32_t num_pages, float *logits,
                                int64_t logits_stride, int32_t *histogram, void *workspace,
                                size_t ws_bytes, void *stream) {
  int32_t e = check_paged_common(q, k_codes, reinterpret_cast<const float *>(k_exp), weights,
                                 page_table, page_table_stride, context_lens, B, next_n,
                                 num_heads, head_dim, page_size, num_pages, workspace, ws_bytes);
  if (e != DSA_OK) return e;
  if (!aligned(k_codes, 32)) return DSA_ERR_MISALIGNED;
  if (!logits || logits_stride < 1) return DSA_ERR_INVALID_ARG;
  if (histogram && !aligned(histogram, 8)) return DSA_ERR_MISALIGNED;
  if (B == 0) return DSA_OK;
  LogitsCall c{};
  c.q = q;
  c.kv = k_codes;
  c.kscale = reinterpret_cast<const float *>(k_exp);  // 4 bytes a token, like kscale
  c.weights = weights;
  c.page_table = page_table;
  c.pt_stride = page_table_stride;
  c.context_lens = context_lens;
  c.B = B;
  c.next_n = next_n;
  c.page_size = page_size;
  c.num_pages = num_pages;
  c.out = logits;
  c.out_stride = logits_stride;
  c.histogram = histogram;
  c.amax = nullptr;
  c.sparse = false;
  c.out_fmt = DSA_OUT_F32;
  c.status = status_word(workspace);
  c.wait_limit = kDefaultWaitLimit;
  c.mx = true;
  return run_paged_logits(c, static_cast<cudaStream_t>(stream));
}

int32_t dsa_sparse_mqa_logits(const uint8_t *q, const uint8_t *kv_pages, const float *kscale,
                              const float *weights, const int32_t *page_table,
                              int64_t page_table_stride, const int32_t *context_lens, int32_t B,
                              int32_t next_n, int32_t num_heads, int32_t head_dim,
                              int32_t page_size, int32_t num_pages, const int32_t *block_table,
                              int32_t kb, const int32_t *phys_blocks, const int32_t *valid_lens,
                              void *out, int32_t out_dtype, int64_t out_stride, void *workspace,
                              size_t ws_bytes, void *stream) {
  int32_t e = check_paged_common(q, kv_pages, kscale, weights, page_table, page_table_stride,
                                 context_lens, B, next_n, num_heads, head_dim, page_size,
                                 num_pages, workspace, ws_bytes);
  if (e != DSA_OK) return e;
  if (!block_table || !out) return DSA_ERR_INVALID_ARG;
  if ((phys_blocks == nullptr) != (valid_lens == nullptr)) return DSA_ERR_INVALID_ARG;
  if (kb < 16 || kb % 16 != 0) return DSA_ERR_UNSUPPORTED;
  if (out_dtype != DSA_OUT_F32 && out_dtype != DSA_OUT_F16 && out_dtype != DSA_OUT_BF16)
    return DSA_ERR_INVALID_ARG;
  if (out_stride < (int64_t)kb * 8) return DSA_ERR_INVALID_ARG;
  if (B == 0) return DSA_OK;
  LogitsCall c{};
  c.q = q;
  c.kv = kv_pages;
  c.kscale = kscale;
  c.weights = weights;
  c.page_table = page_table;
  c.pt_stride = page_table_stride;
  c.context_lens = context_lens;
  c.B = B;
  c.next_n = next_n;
  c.page_size = page_size;
  c.num_pages = num_pages;
  c.out = out;
  c.out_stride = out_stride;
  c.histogram = nullptr;
  c.amax = nullptr;
  c.amax_stride = 0;
  c.amax_skip = 0;
  c.sparse = true;
  c.out_fmt = out_dtype;
  c.block_table = block_table;
  c.kb = kb;
  c.phys = phys_blocks;
  c.valid_lens = valid_lens;
  c.status = status_word(workspace);
  c.wait_limit = kDefaultWaitLimit;
  return run_paged_logits(c, static_cast<cudaStream_t>(stream));
}

namespace {

// Arguments of one top-k problem, checked; fills `c` (without the workspace).
int32_t topk_args(const float *logits, int64_t stride, const int32_t *context_lens,
                  int32_t next_n, int32_t len_div, int32_t R, int32_t *histogram,
                  int32_t reset_histogram, int32_t k, int32_t *out_idx, int32_t *fallback_flags,
                  TopkCall &c) {
  if (R < 0 || next_n < 1 || len_div < 1 || stride < 1) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (!logits || !context_lens || !out_idx) return DSA_ERR_INVALID_ARG;
  if (histogram && !aligned(histogram, 8)) return DSA_ERR_MISALIGNED;
  c = TopkCall{};
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
  return DSA_OK;
}

int32_t topk_problem_args(const dsa_topk_problem &p, TopkCall &c) {
  return topk_args(p.logits, p.stride, p.context_lens, p.next_n, p.len_div, p.R, p.histogram,
                   p.reset_histogram, p.k, p.out_idx, p.fallback_flags, c);
}

}  // namespace

int32_t dsa_coarse_hist_topk(const float *logits, int64_t stride, const int32_t *context_lens,
                             int32_t next_n, int32_t len_div, int32_t R, int32_t *histogram,
                             int32_t reset_histogram, int32_t k, int32_t *out_idx,
                             int32_t *fallback_flags, void *workspace, size_t ws_bytes,
                             void *stream) {
  TopkCall c;
  const int32_t err = topk_args(logits, stride, context_lens, next_n, len_div, R, histogram,
                                reset_histogram, k, out_idx, fallback_flags, c);
  if (err != DSA_OK) return err;
  if (!workspace) return DSA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return DSA_ERR_MISALIGNED;
  const int64_t rows = ws_rows_for(ws_bytes);
  if (rows < R) return DSA_ERR_WORKSPACE;
  if (R == 0) return DSA_OK;
  c.workspace = workspace;
  c.ws_rows = (int32_t)rows;
  return run_topk(c, static_cast<cudaStream_t>(stream));
}

int32_t dsa_coarse_hist_topk_batch(const dsa_topk_problem *problems, int32_t count,
                                   void *workspace, size_t ws_bytes, void *stream) {
  if (count < 0 || (count > 0 && !problems)) return DSA_ERR_INVALID_ARG;
  if (count > DSA_TOPK_BATCH_MAX) return DSA_ERR_UNSUPPORTED;
  TopkCall calls[DSA_TOPK_BATCH_MAX];
  int n = 0;
  int64_t rows_needed = 0;
  bool blocks = false;
  for (int i = 0; i < count; ++i) {
    const dsa_topk_problem &pb = problems[i];
    if (pb.R < 0 || pb.block_k < 0) return DSA_ERR_INVALID_ARG;
    if (pb.R == 0) continue;  // nothing to check or run (pointers may be NULL)
    TopkCall c;
    const int32_t err = topk_problem_args(pb, c);
    if (err != DSA_OK) return err;
    if (pb.block_k > 0) {
      if (!pb.block_out_idx) return DSA_ERR_INVALID_ARG;
      if (pb.block_k > DSA_MAX_TOPK || pb.len_div != 1) return DSA_ERR_UNSUPPORTED;
      c.block_out = pb.block_out_idx;
      c.block_flags = pb.block_fallback_flags;
      c.block_k = pb.block_k;
      blocks = true;
      if (pb.block_page_table) {
        if (pb.block_page_size != 64 && pb.block_page_size != 128) return DSA_ERR_UNSUPPORTED;
        if (pb.block_page_table_stride < 1) return DSA_ERR_INVALID_ARG;
        c.block_pt = pb.block_page_table;
        c.block_pt_stride = pb.block_page_table_stride;
        c.block_ps = pb.block_page_size;
        c.block_phys = pb.block_phys;
        c.block_valid = pb.block_valid_lens;
      }
    } else if (pb.block_page_table) {
      return DSA_ERR_INVALID_ARG;
    }
    rows_needed += c.R;
    calls[n++] = c;
  }
  if (blocks && !topk_batchable(calls, n)) return DSA_ERR_UNSUPPORTED;
  if (!workspace) return DSA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return DSA_ERR_MISALIGNED;
  const int64_t rows = ws_rows_for(ws_bytes);
  if (rows < rows_needed) return DSA_ERR_WORKSPACE;
  if (n == 0) return DSA_OK;
  for (int i = 0; i < n; ++i) {
    calls[i].workspace = workspace;
    calls[i].ws_rows = (int32_t)rows;
  }
  return run_topk_batch(calls, n, static_cast<cudaStream_t>(stream));
}

int32_t dsa_coarse_hist_topk_batch_launches(const dsa_topk_problem *problems, int32_t count) {
  if (count < 0 || (count > 0 && !problems) || count > DSA_TOPK_BATCH_MAX)
    return -DSA_ERR_INVALID_ARG;
  TopkCall calls[DSA_TOPK_BATCH_MAX];
  int n = 0;
  for (int i = 0; i < count; ++i) {
    if (problems[i].stride < 1) return -DSA_ERR_INVALID_ARG;
    if (problems[i].R == 0) continue;
    calls[n] = TopkCall{};
    calls[n].stride = problems[i].stride;
    calls[n].histogram = problems[i].histogram;
    ++n;
  }
  if (n == 0) return 0;
  if (topk_batchable(calls, n)) return 1;
  int32_t total = 0;
  for (int i = 0; i < n; ++i)
    total += topk_launch_count(calls[i].stride, calls[i].histogram != nullptr, true);
  return total;
}

int32_t dsa_coarse_hist_topk_launches(int64_t stride, int32_t has_histogram) {
  if (stride < 1) return -DSA_ERR_INVALID_ARG;
  return topk_launch_count(stride, has_histogram != 0, true);
}

int32_t dsa_block_amax8(const float *logits, int64_t stride, const int32_t *context_lens,
                        int32_t next_n, int32_t R, int32_t skip_if_blocks_le, float *amax,
                        int64_t amax_stride, void *workspace, size_t ws_bytes, void *stream) {
  if (R < 0 || next_n < 1 || stride < 1 || amax_stride < 1) return DSA_ERR_INVALID_ARG;
  if (!logits || !context_lens || !amax) return DSA_ERR_INVALID_ARG;
  if (!aligned(logits, 16) || stride % 4 != 0) return DSA_ERR_MISALIGNED;
  if (!workspace || ws_bytes < WsLayout::kHeader) return DSA_ERR_WORKSPACE;
  if (R == 0) return DSA_OK;
  return run_block_amax8(logits, stride, context_lens, next_n, R, skip_if_blocks_le, amax,
                         amax_stride, status_word(workspace), static_cast<cudaStream_t>(stream));
}

int32_t dsa_sort_candidate_blocks(int32_t *block_ids, int32_t kb, const int32_t *context_lens,
                                  int32_t next_n, int32_t R, const int32_t *page_table,
                                  int64_t page_table_stride, int32_t page_size,
                                  int32_t *phys_blocks, int32_t *valid_lens, void *workspace,
                                  size_t ws_bytes, void *stream) {
  if (R < 0 || next_n < 1 || kb < 1) return DSA_ERR_INVALID_ARG;
  if (kb > 4096) return DSA_ERR_UNSUPPORTED;
  if (!block_ids || !context_lens || !page_table || page_table_stride < 1)
    return DSA_ERR_INVALID_ARG;
  if (page_size < 8 || page_size % 8 != 0) return DSA_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < WsLayout::kHeader) return DSA_ERR_WORKSPACE;
  if (R == 0) return DSA_OK;
  return run_sort_blocks(block_ids, kb, context_lens, next_n, R, page_table, page_table_stride,
                         page_size, phys_blocks, valid_lens, status_word(workspace),
                         static_cast<cudaStream_t>(stream));
}

int32_t dsa_pair_units(int32_t B, int32_t next_n) {
  if (B < 0 || next_n < 1) return 0;
  return B * ((next_n + 1) / 2);
}

int32_t dsa_sort_candidate_blocks_paired(int32_t *block_ids, int32_t kb,
                                         const int32_t *context_lens, int32_t next_n, int32_t B,
                                         const int32_t *page_table, int64_t page_table_stride,
                                         int32_t page_size, int32_t *phys_blocks,
                                         int32_t *valid_lens, int32_t *union_phys,
                                         int32_t *union_pos, int32_t *union_len,
                                         void *workspace, size_t ws_bytes, void *stream) {
  if (B < 0 || next_n < 1 || kb < 1) return DSA_ERR_INVALID_ARG;
  if (kb > 4096) return DSA_ERR_UNSUPPORTED;
  if (!block_ids || !context_lens || !page_table || page_table_stride < 1)
    return DSA_ERR_INVALID_ARG;
  if (!valid_lens || !union_phys || !union_pos || !union_len) return DSA_ERR_INVALID_ARG;
  if (page_size < 8 || page_size % 8 != 0) return DSA_ERR_UNSUPPORTED;
  if (!workspace || ws_bytes < WsLayout::kHeader) return DSA_ERR_WORKSPACE;
  if (B == 0) return DSA_OK;
  return run_sort_pair_blocks(block_ids, kb, context_lens, next_n, B, page_table,
                              page_table_stride, page_size, phys_blocks, valid_lens, union_phys,
                              union_pos, union_len, status_word(workspace),
                              static_cast<cudaStream_t>(stream));
}

int32_t dsa_sparse_mqa_logits_paired(const uint8_t *q, const uint8_t *kv_pages,
                                     const float *kscale, const float *weights,
                                     const int32_t *page_table, int64_t page_table_stride,
                                     const int32_t *context_lens, int32_t B, int32_t next_n,
                                     int32_t num_heads, int32_t head_dim, int32_t page_size,
                                     int32_t num_pages, int32_t kb, const int32_t *union_phys,
                                     const int32_t *union_pos, const int32_t *union_len,
                                     const int32_t *valid_lens, void *out, int32_t out_dtype,
                                     int64_t out_stride, void *workspace, size_t ws_bytes,
                                     void *stream) {
  int32_t e = check_paged_common(q, kv_pages, kscale, weights, page_table, page_table_stride,
                                 context_lens, B, next_n, num_heads, head_dim, page_size,
                                 num_pages, workspace, ws_bytes);
  if (e != DSA_OK) return e;
  if (!union_phys || !union_pos || !union_len || !valid_lens || !out) return DSA_ERR_INVALID_ARG;
  if (kb < 16 || kb % 16 != 0 || kb > 4096) return DSA_ERR_UNSUPPORTED;
  if (out_dtype != DSA_OUT_F32 && out_dtype != DSA_OUT_F16 && out_dtype != DSA_OUT_BF16)
    return DSA_ERR_INVALID_ARG;
  if (out_stride < (int64_t)kb * 8) return DSA_ERR_INVALID_ARG;
  if (B == 0) return DSA_OK;
  LogitsCall c{};
  c.q = q;
  c.kv = kv_pages;
  c.kscale = kscale;
  c.weights = weights;
  c.page_table = page_table;
  c.pt_stride = page_table_stride;
  c.context_lens = context_lens;
  c.B = B;
  c.next_n = next_n;
  c.page_size = page_size;
  c.num_pages = num_pages;
  c.out = out;
  c.out_stride = out_stride;
  c.sparse = true;
  c.out_fmt = out_dtype;
  c.kb = kb;
  c.valid_lens = valid_lens;
  c.union_phys = union_phys;
  c.union_pos = union_pos;
  c.union_len = union_len;
  c.status = status_word(workspace);
  c.wait_limit = kDefaultWaitLimit;
  return run_paged_logits(c, static_cast<cudaStream_t>(stream));
}

int32_t dsa_topk_fp16(const uint16_t *scores, int64_t stride, const int32_t *valid_lens,
                      int32_t R, int32_t k, const int32_t *block_table, int32_t kb,
                      int32_t *out_idx, void *workspace, size_t ws_bytes, void *stream) {
  if (R < 0 || stride < 2) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (!scores || !valid_lens || !out_idx) return DSA_ERR_INVALID_ARG;
  if (stride % 2 != 0 || !aligned(scores, 4)) return DSA_ERR_MISALIGNED;
  if (block_table && kb < 1) return DSA_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < WsLayout::kHeader) return DSA_ERR_WORKSPACE;
  if (R == 0) return DSA_OK;
  Fp16TopkCall c{};
  c.scores = scores;
  c.stride = stride;
  c.valid_lens = valid_lens;
  c.R = R;
  c.k = k;
  c.block_table = block_table;
  c.kb = kb;
  c.out_idx = out_idx;
  c.status = status_word(workspace);
  return run_topk_fp16(c, static_cast<cudaStream_t>(stream));
}

int32_t dsa_topk_bf16(const uint16_t *scores, int64_t stride, const int32_t *valid_lens,
                      int32_t R, int32_t k, const int32_t *block_table, int32_t kb,
                      int32_t *out_idx, void *workspace, size_t ws_bytes, void *stream) {
  if (R < 0 || stride < 2) return DSA_ERR_INVALID_ARG;
  if (k < 1 || k > DSA_MAX_TOPK) return DSA_ERR_UNSUPPORTED;
  if (!scores || !valid_lens || !out_idx) return DSA_ERR_INVALID_ARG;
  if (stride % 2 != 0 || !aligned(scores, 4)) return DSA_ERR_MISALIGNED;
  if (block_table && kb < 1) return DSA_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < WsLayout::kHeader) return DSA_ERR_WORKSPACE;
  if (R == 0) return DSA_OK;
  Fp16TopkCall c{};
  c.scores = scores;
  c.stride = stride;
  c.valid_lens = valid_lens;
  c.R = R;
  c.k = k;
  c.block_table = block_table;
  c.kb = kb;
  c.out_idx = out_idx;
  c.status = status_word(workspace);
  c.bf16 = true;
  return run_topk_fp16(c, static_cast<cudaStream_t>(stream));
}

int32_t dsa_coarse_bin_key_ranges(uint32_t *out, void *stream) {
  if (!out) return DSA_ERR_INVALID_ARG;
  return run_bin_key_ranges(out, static_cast<cudaStream_t>(stream));
}

int32_t dsa_coarse_bins_range(uint32_t start, int64_t count, int16_t *out, void *stream) {
  if (count < 0 || (count > 0 && !out)) return DSA_ERR_INVALID_ARG;
  return run_bins_range(start, count, out, static_cast<cudaStream_t>(stream));
}

int32_t dsa_fp16_order_keys(const uint16_t *in, uint16_t *out, int64_t n, void *stream) {
  if (n < 0 || n % 2 != 0) return DSA_ERR_INVALID_ARG;
  if (n > 0 && (!in || !out)) return DSA_ERR_INVALID_ARG;
  if (!aligned(in, 4) || !aligned(out, 4)) return DSA_ERR_MISALIGNED;
  return run_fp16_keys(in, out, n, static_cast<cudaStream_t>(stream));
}

int32_t dsa_bf16_order_keys(const uint16_t *in, uint16_t *out, int64_t n, void *stream) {
  if (n < 0 || n % 2 != 0) return DSA_ERR_INVALID_ARG;
  if (n > 0 && (!in || !out)) return DSA_ERR_INVALID_ARG;
  if (!aligned(in, 4) || !aligned(out, 4)) return DSA_ERR_MISALIGNED;
  return run_bf16_keys(in, out, n, static_cast<cudaStream_t>(stream));
}

int32_t dsa_decode_step(const dsa_decode_step_args *args, void *workspace, size_t ws_bytes,
                        void *stream) {
  if (!args) return DSA_ERR_INVALID_ARG;
  const dsa_decode_step_args &a = *args;
  if (a.B < 0 || a.next_n < 1 || a.kb < 1 || a.k < 1 || a.logits_stride < 1)
    return DSA_ERR_INVALID_ARG;
  if (a.B == 0) return DSA_OK;
  const int32_t R = a.B * a.next_n;
  dsa_topk_problem p{};
  p.logits = a.logits;
  p.stride = a.logits_stride;
  p.context_lens = a.context_lens;
  p.histogram = a.histogram;
  p.out_idx = a.topk_idx;
  p.block_out_idx = a.block_ids;
  p.next_n = a.next_n;
  p.len_div = 1;
  p.R = R;
  p.reset_histogram = 1;
  p.k = a.k;
  p.block_k = a.kb;
  p.block_page_table = a.page_table;
  p.block_page_table_stride = a.page_table_stride;
  p.block_page_size = a.page_size;
  p.block_phys = a.phys_blocks;
  p.block_valid_lens = a.valid_lens;
  // rows a single cluster launch takes (the select writes the table itself)
  if (dsa_coarse_hist_topk_batch_launches(&p, 1) != 1) return DSA_ERR_UNSUPPORTED;
  int32_t e = dsa_paged_mqa_logits(a.q, a.kv_pages, a.kscale, a.weights, a.page_table,
                                   a.page_table_stride, a.context_lens, a.B, a.next_n, 32, 128,
                                   a.page_size, a.num_pages, a.logits, a.logits_stride,
                                   a.histogram, nullptr, 0, a.kb, workspace, ws_bytes, stream);
  if (e != DSA_OK) return e;
  e = dsa_coarse_hist_topk_batch(&p, 1, workspace, ws_bytes, stream);
  if (e != DSA_OK) return e;
  e = dsa_sparse_mqa_logits(a.q, a.kv_pages, a.kscale, a.weights, a.page_table,
                            a.page_table_stride, a.context_lens, a.B, a.next_n, 32, 128,
                            a.page_size, a.num_pages, a.block_ids, a.kb, a.phys_blocks,
                            a.valid_lens, a.sparse_scores, DSA_OUT_F16, (int64_t)a.kb * 8,
                            workspace, ws_bytes, stream);
  if (e != DSA_OK) return e;
  return dsa_topk_fp16(a.sparse_scores, (int64_t)a.kb * 8, a.valid_lens, R, a.k, a.block_ids,
                       a.kb, a.sparse_idx, workspace, ws_bytes, stream);
}

int32_t dsa_wait_timeout_selftest(uint64_t limit_cycles, void *workspace, size_t ws_bytes,
                                  void *stream) {
  if (!workspace || ws_bytes < WsLayout::kHeader) return DSA_ERR_WORKSPACE;
  if (limit_cycles == 0 || limit_cycles > (1ULL << 40)) return DSA_ERR_INVALID_ARG;
  return run_wait_selftest(limit_cycles, status_word(workspace), static_cast<cudaStream_t>(stream));
}

}  // extern "C"
