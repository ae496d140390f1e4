// blocks.cu -- the level-one block pipeline of the two-level candidate path
// (SGLang PR #38944, squashed commit texts):
//   amax8_varlen           block maximum of every 8 consecutive scores, the
//                          newest block forced to +inf, nothing written past
//                          the block count, short rows optionally skipped
//   sort_candidate_blocks  selected block ids (any order, -1 padded) ->
//                          ascending INT32_MAX-padded table in place, by a
//                          counting sort over a shared-memory bitmap, plus
//                          the physical blocks (pool slot / 8 through the
//                          row's page table) and the live length of the
//                          sparse row (candidate_row_lens)
//   sort_pair_blocks       the same for the two rows of a unit of the paired
//                          sparse pass, plus the ascending union of their
//                          tables (commit text on DeepGEMM's sparse schedule)
#include <algorithm>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {

namespace {

constexpr int kAmaxThreads = 256;
constexpr int kSortThreads = 512;
constexpr int kMaxBitmapWords = 8192;  // 262144 blocks = 2M tokens per row

__device__ __forceinline__ int64_t live_len(const int32_t *ctx, int next_n, int r) {
  const int64_t n = (int64_t)ctx[r / next_n] - (next_n - 1 - r % next_n);
  return n < 0 ? 0 : n;
}

__device__ __forceinline__ float key_to_f32(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key ^ 0x80000000u) : ~key);
}

// One thread per 8-score block; the maximum is taken on FP32 order keys (so
// -0 < +0 and NaN, mapped to key 0, never wins unless the block is all NaN).
__global__ void __launch_bounds__(kAmaxThreads)
    amax8_kernel(const float *logits, int64_t stride, const int32_t *ctx, int next_n,
                 int skip_le, float *amax, int64_t amax_stride, uint32_t *status) {
  pdl_wait();  // predecessor grids complete before any global access
  const int r = blockIdx.y;
  int64_t n = live_len(ctx, next_n, r);
  if (n > stride) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
    n = stride;
  }
  const int64_t nb = (n + 7) / 8;
  if (nb == 0 || (skip_le > 0 && nb <= skip_le)) return;
  const int64_t i = (int64_t)blockIdx.x * kAmaxThreads + threadIdx.x;
  if (i >= nb || i >= amax_stride) return;
  float m;
  if (i == nb - 1) {
    m = INFINITY;  // the newest block is always chosen
  } else {
    const float4 *p = reinterpret_cast<const float4 *>(logits + (int64_t)r * stride + 8 * i);
    const float4 v0 = p[0], v1 = p[1];
    const float x[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
    uint32_t best = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t kk = isnan(x[e]) ? 0u : f32_order_key(x[e]);
      best = max(best, kk);
    }
    m = best ? key_to_f32(best) : __int_as_float(0x7fc00000);
  }
  amax[(int64_t)r * amax_stride + i] = m;
}

__device__ __forceinline__ int block_excl_scan512(int v, int *ws, int *total) {
  constexpr int W = kSortThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = (lane < W) ? ws[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < W) ws[lane] = wi - w;
    if (lane == W - 1) ws[W] = wi;
  }
  __syncthreads();
  const int res = ws[warp] + incl - v;
  *total = ws[W];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kSortThreads)
    sort_blocks_kernel(int32_t *ids, int kb, const int32_t *ctx, int next_n,
                       const int32_t *page_table, int64_t pt_stride, int page_size,
                       int32_t *phys, int32_t *valid_lens, uint32_t *status) {
  pdl_wait();  // predecessor grids complete before any global access
  pdl_release_dependents();  // one CTA per row: the sparse logits set up on the idle SMs
  __shared__ uint32_t bm[kMaxBitmapWords];
  __shared__ int sm_scan[kSortThreads / 32 + 1];
  __shared__ long long sm_live[kSortThreads / 32];
  const int r = blockIdx.x;
  const int b = r / next_n;
  int64_t n = live_len(ctx, next_n, r);
  const int64_t cap = pt_stride * page_size;
  if (n > cap) {
    if (threadIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
    n = cap;
  }
  int64_t nb = (n + 7) / 8;
  if (nb > (int64_t)kMaxBitmapWords * 32) {
    if (threadIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
    nb = (int64_t)kMaxBitmapWords * 32;
  }
  int32_t *idr = ids + (int64_t)r * kb;
  // (tokens below 2^31: context lengths are int32; a power-of-two page size
  // takes shifts instead of a division per block)
  const bool pow2 = (page_size & (page_size - 1)) == 0;
  const int lg = __ffs(page_size) - 1;
  auto phys_of = [&](int64_t id) -> int32_t {
    const int tok = (int)(id * 8);
    const int pi = pow2 ? tok >> lg : tok / page_size;
    const int64_t pg = page_table[(int64_t)b * pt_stride + pi];
    return (int32_t)((pg * page_size + (tok - pi * page_size)) >> 3);
  };
  long long live = 0;
  if (nb <= kb) {
    // identity table: every block of the row, in order
    for (int i = threadIdx.x; i < kb; i += kSortThreads) {
      if (i < nb) {
        idr[i] = i;
        if (phys) phys[(int64_t)r * kb + i] = phys_of(i);
      } else {
        idr[i] = INT32_MAX;
        if (phys) phys[(int64_t)r * kb + i] = INT32_MAX;
      }
    }
    if (valid_lens && threadIdx.x == 0) valid_lens[r] = (int32_t)n;
    return;
  }
  const int W = (int)((nb + 31) / 32);
  for (int w = threadIdx.x; w < W; w += kSortThreads) bm[w] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < kb; i += kSortThreads) {
    const int32_t id = idr[i];
    if (id >= 0 && id < nb) {
      atomicOr(&bm[id >> 5], 1u << (id & 31));
    } else if (id != -1 && id != INT32_MAX) {
      set_status(status, DSA_DEV_BOUNDS);
    }
  }
  __syncthreads();
  // each thread owns a contiguous run of words; a block scan of their
  // population counts gives every set bit its ascending output slot
  const int per = (W + kSortThreads - 1) / kSortThreads;
  const int w0 = threadIdx.x * per, w1 = min(W, w0 + per);
  int c = 0;
  for (int w = w0; w < w1; ++w) c += __popc(bm[w]);
  int total;
  int pos = block_excl_scan512(c, sm_scan, &total);
  for (int w = w0; w < w1; ++w) {
    uint32_t m = bm[w];
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      const int64_t id = (int64_t)w * 32 + bit;
      if (pos < kb) idr[pos] = (int32_t)id;
      ++pos;
      const int64_t in_blk = n - id * 8;
      live += in_blk < 8 ? in_blk : 8;
    }
  }
  for (int i = total + threadIdx.x; i < kb; i += kSortThreads) idr[i] = INT32_MAX;
  if (phys) {
    // the physical blocks one table slot a thread, from the sorted ids just
    // written (visible to the whole block after the barrier), so no
    // page-table read sits in the serial bitmap walk above
    __syncthreads();
    const int nt = min(total, kb);
    for (int i = threadIdx.x; i < kb; i += kSortThreads)
      phys[(int64_t)r * kb + i] = i < nt ? phys_of(idr[i]) : INT32_MAX;
  }
  if (valid_lens) {
    long long v = live;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) sm_live[threadIdx.x >> 5] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
      long long s = 0;
      for (int i = 0; i < kSortThreads / 32; ++i) s += sm_live[i];
      valid_lens[r] = (int32_t)s;
    }
  }
}

// Row pairing of the sparse pass (SGLang PR #38944, commit text on DeepGEMM's
// sparse schedule): rows 2m and 2m+1 of a request form one unit, an odd last
// row a unit of its own.  One CTA per unit sorts both rows' tables exactly as
// sort_blocks_kernel does (ascending, INT32_MAX padded, physical blocks, live
// lengths) and emits the ascending union of the two: per entry the physical
// block and, per row, its table position + 1 (0: the row does not hold the
// block), in one pass over the two bitmaps.
__global__ void __launch_bounds__(kSortThreads)
    sort_pair_blocks_kernel(int32_t *ids, int kb, const int32_t *ctx, int next_n,
                            const int32_t *page_table, int64_t pt_stride, int page_size,
                            int wmax, int32_t *phys, int32_t *valid_lens, int32_t *uphys,
                            int32_t *upos, int32_t *ulen, uint32_t *status) {
  pdl_wait();
  pdl_release_dependents();
  extern __shared__ uint32_t bms[];  // two bitmaps of wmax words
  __shared__ int sm_scan[kSortThreads / 32 + 1];
  __shared__ long long sm_live[2][kSortThreads / 32];
  const int upr = (next_n + 1) / 2;
  const int u = blockIdx.x;
  const int b = u / upr, m = u - b * upr;
  const int r0 = b * next_n + 2 * m;
  const int nrow = (2 * m + 1 < next_n) ? 2 : 1;
  const int64_t cap = pt_stride * page_size;
  int64_t n[2] = {0, 0}, nb[2] = {0, 0};
  for (int j = 0; j < nrow; ++j) {
    n[j] = live_len(ctx, next_n, r0 + j);
    if (n[j] > cap) {
      if (threadIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
      n[j] = cap;
    }
    nb[j] = (n[j] + 7) / 8;
    if (nb[j] > (int64_t)wmax * 32) {
      if (threadIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
      nb[j] = (int64_t)wmax * 32;
    }
  }
  const int W = (int)((max(nb[0], nb[1]) + 31) / 32);
  uint32_t *bm0 = bms, *bm1 = bms + wmax;
  for (int w = threadIdx.x; w < W; w += kSortThreads) {
    // rows with at most kb blocks take every block (the identity table)
    for (int j = 0; j < 2; ++j) {
      uint32_t v = 0;
      if (j < nrow && nb[j] <= kb) {
        const int64_t lo = (int64_t)w * 32;
        v = (nb[j] >= lo + 32) ? 0xffffffffu : (nb[j] > lo ? (1u << (nb[j] - lo)) - 1u : 0u);
      }
      (j == 0 ? bm0 : bm1)[w] = v;
    }
  }
  __syncthreads();
  for (int j = 0; j < nrow; ++j) {
    if (nb[j] <= kb) continue;
    const int32_t *idr = ids + (int64_t)(r0 + j) * kb;
    uint32_t *bm = j == 0 ? bm0 : bm1;
    for (int i = threadIdx.x; i < kb; i += kSortThreads) {
      const int32_t id = idr[i];
      if (id >= 0 && id < nb[j]) {
        atomicOr(&bm[id >> 5], 1u << (id & 31));
      } else if (id != -1 && id != INT32_MAX) {
        set_status(status, DSA_DEV_BOUNDS);
      }
    }
  }
  __syncthreads();
  // (tokens below 2^31: context lengths are int32; a power-of-two page size
  // takes shifts instead of a division per block)
  const bool pow2 = (page_size & (page_size - 1)) == 0;
  const int lg = __ffs(page_size) - 1;
  auto phys_of = [&](int64_t id) -> int32_t {
    const int tok = (int)(id * 8);
    const int pi = pow2 ? tok >> lg : tok / page_size;
    const int64_t pg = page_table[(int64_t)b * pt_stride + pi];
    return (int32_t)((pg * page_size + (tok - pi * page_size)) >> 3);
  };
  const int per = (W + kSortThreads - 1) / kSortThreads;
  const int w0 = threadIdx.x * per, w1 = min(W, w0 + per);
  int ca = 0, cb = 0, cu = 0;
  for (int w = w0; w < w1; ++w) {
    ca += __popc(bm0[w]);
    cb += __popc(bm1[w]);
    cu += __popc(bm0[w] | bm1[w]);
  }
  int tot_a, tot_b, tot_u;
  int pa = block_excl_scan512(ca, sm_scan, &tot_a);
  int pb = block_excl_scan512(cb, sm_scan, &tot_b);
  int pu = block_excl_scan512(cu, sm_scan, &tot_u);
  int32_t *ida = ids + (int64_t)r0 * kb, *idb = ids + (int64_t)(r0 + 1) * kb;
  int32_t *pha = phys ? phys + (int64_t)r0 * kb : nullptr;
  int32_t *phb = phys ? phys + (int64_t)(r0 + 1) * kb : nullptr;
  int32_t *up = uphys + (int64_t)u * 2 * kb, *uq = upos + (int64_t)u * 2 * kb;
  long long live[2] = {0, 0};
  for (int w = w0; w < w1; ++w) {
    const uint32_t a = bm0[w], c = bm1[w];
    uint32_t mk = a | c;
    while (mk) {
      const int bit = __ffs(mk) - 1;
      mk &= mk - 1;
      const int64_t id = (int64_t)w * 32 + bit;
      uint32_t word = 0;
      if ((a >> bit) & 1u) {
        if (pa < kb) {
          ida[pa] = (int32_t)id;
          word |= (uint32_t)(pa + 1);
        }
        ++pa;
        const int64_t in_blk = n[0] - id * 8;
        live[0] += in_blk < 8 ? in_blk : 8;
      }
      if ((c >> bit) & 1u) {
        if (pb < kb) {
          idb[pb] = (int32_t)id;
          word |= (uint32_t)(pb + 1) << 16;
        }
        ++pb;
        const int64_t in_blk = n[1] - id * 8;
        live[1] += in_blk < 8 ? in_blk : 8;
      }
      if (pu < 2 * kb) {
        up[pu] = (int32_t)id;  // the block id for now: its physical block below
        uq[pu] = (int32_t)word;
      }
      ++pu;
    }
  }
  // the physical blocks one union slot a thread (visible to the whole block
  // after the barrier), so no page-table read sits in the serial walk above:
  // the union's own entry, and through its positions each row's
  __syncthreads();
  const int nu = min(tot_u, 2 * kb);
  for (int i = threadIdx.x; i < nu; i += kSortThreads) {
    const int32_t ph = phys_of(up[i]);
    up[i] = ph;
    const uint32_t word = (uint32_t)uq[i];
    if (pha && (word & 0xFFFFu)) pha[(word & 0xFFFFu) - 1] = ph;
    if (phb && (word >> 16)) phb[(word >> 16) - 1] = ph;
  }
  for (int j = 0; j < nrow; ++j) {
    int32_t *idr = j == 0 ? ida : idb;
    int32_t *phr = j == 0 ? pha : phb;
    for (int i = (j == 0 ? tot_a : tot_b) + threadIdx.x; i < kb; i += kSortThreads) {
      idr[i] = INT32_MAX;
      if (phr) phr[i] = INT32_MAX;
    }
  }
  for (int i = tot_u + threadIdx.x; i < 2 * kb; i += kSortThreads) {
    up[i] = INT32_MAX;
    uq[i] = 0;
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    long long v = live[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) sm_live[j][threadIdx.x >> 5] = v;
  }
  __syncthreads();
  if (threadIdx.x < nrow) {
    long long s = 0;
    for (int i = 0; i < kSortThreads / 32; ++i) s += sm_live[threadIdx.x][i];
    valid_lens[r0 + threadIdx.x] = (int32_t)s;
  }
  if (threadIdx.x == 0) ulen[u] = min(tot_u, 2 * kb);
}

}  // namespace

dsa_status_t run_block_amax8(const float *logits, int64_t stride, const int32_t *context_lens,
                             int32_t next_n, int32_t R, int32_t skip_le, float *amax,
                             int64_t amax_stride, uint32_t *status, cudaStream_t st) {
  const int64_t nbmax = (stride + 7) / 8;
  const int64_t gx = (nbmax + kAmaxThreads - 1) / kAmaxThreads;
  if (gx > 0x7fffffff || R > 65535) return DSA_ERR_UNSUPPORTED;
  return launch_pdl(amax8_kernel, dim3((unsigned)std::max<int64_t>(1, gx), (unsigned)R),
                    dim3(kAmaxThreads), 0, st, logits, stride, context_lens, next_n, skip_le, amax,
                    amax_stride, status);
}

dsa_status_t run_sort_blocks(int32_t *ids, int32_t kb, const int32_t *context_lens,
                             int32_t next_n, int32_t R, const int32_t *page_table,
                             int64_t pt_stride, int32_t page_size, int32_t *phys,
                             int32_t *valid_lens, uint32_t *status, cudaStream_t st) {
  return launch_pdl(sort_blocks_kernel, dim3(R), dim3(kSortThreads), 0, st, ids, kb, context_lens,
                    next_n, page_table, pt_stride, page_size, phys, valid_lens, status);
}

dsa_status_t run_sort_pair_blocks(int32_t *ids, int32_t kb, const int32_t *context_lens,
                                  int32_t next_n, int32_t B, const int32_t *page_table,
                                  int64_t pt_stride, int32_t page_size, int32_t *phys,
                                  int32_t *valid_lens, int32_t *union_phys, int32_t *union_pos,
                                  int32_t *union_len, uint32_t *status, cudaStream_t st) {
  const int64_t units = (int64_t)B * ((next_n + 1) / 2);
  if (units > 0x7fffffff) return DSA_ERR_UNSUPPORTED;
  // bitmap words for the longest row the page table can address
  const int64_t nbmax = (pt_stride * page_size + 7) / 8;
  const int wmax = (int)std::min<int64_t>(kMaxBitmapWords, (nbmax + 31) / 32);
  const size_t smem = (size_t)2 * wmax * 4;
  if (!ensure_smem_attr(reinterpret_cast<const void *>(sort_pair_blocks_kernel), (int)smem))
    return DSA_ERR_CUDA;
  return launch_pdl(sort_pair_blocks_kernel, dim3((unsigned)units), dim3(kSortThreads), smem, st,
                    ids, kb, context_lens, next_n, page_table, pt_stride, page_size, wmax, phys,
                    valid_lens, union_phys, union_pos, union_len, status);
}

}  // namespace dsa
