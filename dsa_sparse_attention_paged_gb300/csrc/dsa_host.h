// dsa_host.h -- host-side helpers shared by the library's translation units
// (tensor-map encoding, launch checks, device queries, call descriptors).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "dsa.h"  // include/ is on the include path

namespace dsa {

// Default bound of every spin-wait inside a kernel, in SM clock cycles (about
// two seconds at GB300 clocks); a wait that runs out sets DSA_DEV_TIMEOUT.
constexpr long long kDefaultWaitLimit = 4000000000LL;

struct LogitsCall {
  const uint8_t *q;
  const uint8_t *kv;
  const float *kscale;
  const float *weights;
  const int32_t *page_table;
  int64_t pt_stride;
  const int32_t *context_lens;
  int32_t B, next_n, page_size, num_pages;
  void *out;
  int64_t out_stride;
  int32_t *histogram;
  float *amax;
  int64_t amax_stride;
  int32_t amax_skip;
  bool sparse;
  int32_t out_fmt;      // DSA_OUT_F32 / F16 / BF16 (sparse only)
  const int32_t *block_table;
  int32_t kb;
  const int32_t *phys = nullptr;        // sparse: physical blocks of the table, or NULL
  const int32_t *valid_lens = nullptr;  // sparse, with phys: live prefix length per row
  // sparse, paired rows: units of two rows of one request walk the union of
  // their tables (physical block, per-row position + 1, union length)
  const int32_t *union_phys = nullptr;
  const int32_t *union_pos = nullptr;
  const int32_t *union_len = nullptr;
  uint32_t *status;
  long long wait_limit;
  // MXFP4 keys: kv = E2M1 codes [slots][64] (two per byte, even dimension in
  // the low nibble), kscale = the UE8M0 exponents [slots][4] (dense only)
  bool mx = false;
};

dsa_status_t run_paged_logits(const LogitsCall &c, cudaStream_t st);
int logits_stages_for(int next_n, bool hist, bool mx = false);

struct TopkCall {
  const float *logits;
  int64_t stride;
  const int32_t *context_lens;
  int32_t next_n, len_div, R;
  int32_t *histogram;        // caller's, or NULL
  bool reset_histogram;
  int32_t k;
  int32_t *out_idx;
  int32_t *fallback_flags;
  int32_t *block_out = nullptr;    // also the top block_k block maxima per row (one launch only)
  int32_t *block_flags = nullptr;
  int32_t block_k = 0;
  // block output written as the sorted block table (with physical blocks and
  // live lengths) when block_pt is set
  const int32_t *block_pt = nullptr;
  int64_t block_pt_stride = 0;
  int32_t block_ps = 0;
  int32_t *block_phys = nullptr;
  int32_t *block_valid = nullptr;
  void *workspace;
  int32_t ws_rows;           // rows the workspace was sized for
  bool allow_cluster = true; // rows up to 131072 may take the cluster kernel
};
dsa_status_t run_topk(const TopkCall &c, cudaStream_t st);
// kernel launches run_topk makes for rows of `stride` scores
int32_t topk_launch_count(int64_t stride, bool has_histogram, bool allow_cluster);
// several independent calls sharing calls[0]'s workspace (rows laid out one
// problem after another): one launch when topk_batchable, else in sequence
bool topk_batchable(const TopkCall *calls, int count);
dsa_status_t run_topk_batch(const TopkCall *calls, int count, cudaStream_t st);

struct Fp16TopkCall {
  const uint16_t *scores;
  int64_t stride;
  const int32_t *valid_lens;
  int32_t R, k;
  const int32_t *block_table;
  int32_t kb;
  int32_t *out_idx;
  uint32_t *status;
  bool bf16 = false;  // BF16 scores instead of FP16
};
dsa_status_t run_topk_fp16(const Fp16TopkCall &c, cudaStream_t st);

dsa_status_t run_block_amax8(const float *logits, int64_t stride, const int32_t *context_lens,
                             int32_t next_n, int32_t R, int32_t skip_le, float *amax,
                             int64_t amax_stride, uint32_t *status, cudaStream_t st);

dsa_status_t run_sort_blocks(int32_t *ids, int32_t kb, const int32_t *context_lens,
                             int32_t next_n, int32_t R, const int32_t *page_table,
                             int64_t pt_stride, int32_t page_size, int32_t *phys,
                             int32_t *valid_lens, uint32_t *status, cudaStream_t st);

dsa_status_t run_sort_pair_blocks(int32_t *ids, int32_t kb, const int32_t *context_lens,
                                  int32_t next_n, int32_t B, const int32_t *page_table,
                                  int64_t pt_stride, int32_t page_size, int32_t *phys,
                                  int32_t *valid_lens, int32_t *union_phys, int32_t *union_pos,
                                  int32_t *union_len, uint32_t *status, cudaStream_t st);

dsa_status_t run_bins_range(uint32_t start, int64_t count, int16_t *out, cudaStream_t st);
dsa_status_t run_bf16_keys(const uint16_t *in, uint16_t *out, int64_t n, cudaStream_t st);
dsa_status_t run_bin_key_ranges(uint32_t *out, cudaStream_t st);
dsa_status_t run_fp16_keys(const uint16_t *in, uint16_t *out, int64_t n, cudaStream_t st);
dsa_status_t run_wait_selftest(uint64_t limit, uint32_t *status, cudaStream_t st);

void record_cuda_error(cudaError_t e);

// Launch with programmatic stream serialisation (see pdl_wait in
// dsa_device.cuh): the kernel may be scheduled while the previous kernel on
// the stream drains; it waits for it before reading or writing memory.
template <typename... KArgs, typename... Args>
dsa_status_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                        cudaStream_t st, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    (void)cudaGetLastError();
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

// --- utilities (api.cu) ---
dsa_status_t make_tmap_rows128(CUtensorMap *map, const void *base, uint64_t rows,
                               uint32_t box_rows);
// Rows of 128 E2M1 codes packed two per byte (64 bytes), copied into shared
// memory unpacked to the 128-byte rows of an 8-bit operand (each 16 codes in
// the first 8 bytes of a 16-byte chunk), 128-byte swizzle; base 32-byte aligned.
dsa_status_t make_tmap_rows_e2m1(CUtensorMap *map, const void *base, uint64_t rows,
                                 uint32_t box_rows);
int num_sms();
bool ensure_smem_attr(const void *fn, int bytes);
dsa_status_t check_launch();

}  // namespace dsa
