// topk.cu -- exact per-row top-k selects.
//
// FP32 select (SGLang commit 7e252c5, select.cuh, cross-referenced from
// DeepGEMM PR #94 "Motivation"): the coarse histogram the logits kernel
// produced gives each row its threshold bin T (bins above T hold fewer than k
// scores, T completes k).  One pass over the row then emits every score in a
// bin above T straight into the output and collects the scores of bin T as
// candidates; an exact radix select over the candidates (64-bit keys: value
// order key, then inverted column so ties go to the lower column) finishes
// the row.  The pass is split over several CTAs per row; the last CTA to
// finish checks the counts against the histogram and refines.  A stale
// histogram or an over-capacity bin T falls back to an exact whole-row radix
// select in that CTA instead of raising a device error.
//
// FP16 select (vLLM PR #52696 "Why"): scores arrive as packed FP16 bits; both
// halves of each 32-bit word become order keys in one 32-bit operation; a
// 10-bit coarse histogram pass finds the threshold bin and one refine pass
// over the remaining 6 bits finds the exact threshold key.
#include <algorithm>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {

namespace {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

__device__ __forceinline__ int64_t row_len(const int32_t *ctx, int next_n, int len_div, int r,
                                           int64_t stride, uint32_t *status) {
  int64_t n = (int64_t)ctx[r / next_n] - (next_n - 1 - r % next_n);
  if (n < 0) n = 0;
  n = (n + len_div - 1) / len_div;
  if (n > stride) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
    n = stride;
  }
  return n;
}

// Block-wide exclusive scan of one int per thread (kSelThreads threads).
// Returns the exclusive prefix; *total gets the block sum.  Uses `ws`
// (kSelWarps + 1 ints of shared memory); ends with a __syncthreads.
__device__ __forceinline__ int block_excl_scan(int v, int *ws, int *total) {
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
    int w = (lane < kSelWarps) ? ws[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    if (lane < kSelWarps) ws[lane] = wi - w;
    if (lane == kSelWarps - 1) ws[kSelWarps] = wi;
  }
  __syncthreads();
  const int res = ws[warp] + incl - v;
  *total = ws[kSelWarps];
  __syncthreads();
  return res;
}

// From a 256-bin digit histogram, find the digit d (searching from 255 down)
// where the count of larger digits `above` satisfies above < need <= above +
// h[d].  One warp; results to *d_out, *above_out.  If the histogram holds
// fewer than `need` entries, d = -1 and above = the total.
__device__ __forceinline__ void find_digit_desc(const int *h, int need, int *d_out,
                                                int *above_out) {
  const int lane = threadIdx.x & 31;
  // lane l owns digits 255-8l .. 248-8l (descending)
  int c[8];
  int sum = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    c[e] = h[255 - 8 * lane - e];
    sum += c[e];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  const int excl = incl - sum;
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  const unsigned m = __ballot_sync(0xffffffffu, incl >= need);
  if (m == 0) {
    if (lane == 0) {
      *d_out = -1;
      *above_out = total;
    }
    return;
  }
  const int l = __ffs(m) - 1;
  if (lane == l) {
    int acc = excl;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (acc + c[e] >= need) {
        *d_out = 255 - 8 * lane - e;
        *above_out = acc;
        break;
      }
      acc += c[e];
    }
  }
}

struct SelArgs {
  const float *logits;
  int64_t stride;
  const int32_t *ctx;
  int next_n, len_div, R;
  int32_t *hist;
  int reset_hist;
  int k;
  int32_t *out;
  int32_t *flags;
  int32_t *counters;              // [R][4]
  unsigned long long *cand;       // [R][DSA_CAND_CAP]
  uint32_t *status;
  int64_t chunk;
};

__device__ __forceinline__ unsigned long long cand_key(float x, int64_t t) {
  return ((unsigned long long)f32_order_key(x) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)t);
}

// Exact top-k of one FP32 row by MSB radix select over 32-bit order keys, run
// by the whole block.  Ties at the threshold key go to the lowest columns
// (ordered scan).  Writes all k outputs (-1 padded).
__device__ void block_radix_topk_row(const float *row, int64_t n, int k, int32_t *out,
                                     int *sm_h /*256*/, int *sm_scan /*kSelWarps+1*/,
                                     int *sm_misc /*8*/) {
  uint32_t prefix = 0, mask = 0;
  int need = k;
  bool early = false;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kSelThreads) sm_h[i] = 0;
    __syncthreads();
    for (int64_t t = threadIdx.x; t < n; t += kSelThreads) {
      const float x = row[t];
      if (isnan(x)) continue;
      const uint32_t key = f32_order_key(x);
      if ((key & mask) == prefix) atomicAdd(&sm_h[(key >> shift) & 255], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) find_digit_desc(sm_h, need, &sm_misc[0], &sm_misc[1]);
    __syncthreads();
    const int d = sm_misc[0], above = sm_misc[1];
    if (d < 0) {
      // fewer valid entries than k (only possible on the first pass): take all
      prefix = 0;
      mask = 0;
      need = 0;
      early = true;
      break;
    }
    const int hd = sm_h[d];
    need -= above;
    prefix |= (uint32_t)d << shift;
    mask |= 0xFFu << shift;
    __syncthreads();
    if (need == hd) {
      early = true;  // the whole bucket is taken: select key >= prefix
      break;
    }
  }
  // emit: key > prefix (or >= when early) in any order; ties == prefix by column
  if (threadIdx.x == 0) sm_misc[2] = 0;
  __syncthreads();
  const int n_gt_target = early ? 0 : k - need;  // number strictly above the threshold
  int eq_base = 0;
  for (int64_t base = 0; base < n; base += (int64_t)kSelThreads * 4) {
    int eqc = 0;
    bool eqf[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t t = base + threadIdx.x * 4 + e;
      eqf[e] = false;
      if (t >= n) continue;
      const float x = row[t];
      if (isnan(x)) continue;
      const uint32_t key = f32_order_key(x);
      const bool sel = early ? (key >= prefix) : (key > prefix);
      if (sel) {
        const int p = atomicAdd(&sm_misc[2], 1);
        if (p < k) out[p] = (int32_t)t;
      } else if (!early && key == prefix) {
        eqf[e] = true;
        ++eqc;
      }
    }
    int tot;
    const int ex = block_excl_scan(eqc, sm_scan, &tot);
    int rank = eq_base + ex;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (!eqf[e]) continue;
      if (rank < need) out[n_gt_target + rank] = (int32_t)(base + threadIdx.x * 4 + e);
      ++rank;
    }
    eq_base += tot;
  }
  __syncthreads();
  const int written = early ? sm_misc[2] : k;
  for (int i = written + threadIdx.x; i < k; i += kSelThreads) out[i] = -1;
  __syncthreads();
}

__global__ void __launch_bounds__(kSelThreads)
    hist_build_kernel(const float *logits, int64_t stride, const int32_t *ctx, int next_n,
                      int len_div, int64_t chunk, int32_t *hist, uint32_t *status) {
  __shared__ int h[DSA_NUM_BINS];
  const int r = blockIdx.y;
  for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kSelThreads) h[i] = 0;
  __syncthreads();
  const int64_t n = row_len(ctx, next_n, len_div, r, stride, status);
  const int64_t c0 = blockIdx.x * chunk, c1 = min(n, c0 + chunk);
  const float *row = logits + (int64_t)r * stride;
  for (int64_t t = c0 + threadIdx.x; t < c1; t += kSelThreads) {
    const int b = coarse_bin(row[t]);
    if (b >= 0) atomicAdd(&h[b], 1);
  }
  __syncthreads();
  for (int p = threadIdx.x; p < DSA_NUM_BINS / 2; p += kSelThreads) {
    const uint32_t c0v = h[2 * p], c1v = h[2 * p + 1];
    if (c0v | c1v)
      atomicAdd(reinterpret_cast<unsigned long long *>(hist + (int64_t)r * DSA_NUM_BINS + 2 * p),
                ((unsigned long long)c1v << 32) | c0v);
  }
}

__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelArgs a) {
  __shared__ int sm_h[256];
  __shared__ int sm_scan[kSelWarps + 1];
  __shared__ int sm_misc[8];
  __shared__ int sm_last;
  const int r = blockIdx.y;
  const int k = a.k;
  const int lane = threadIdx.x & 31;
  const int64_t n = row_len(a.ctx, a.next_n, a.len_div, r, a.stride, a.status);
  const float *row = a.logits + (int64_t)r * a.stride;
  const int32_t *hr = a.hist + (int64_t)r * DSA_NUM_BINS;
  int32_t *outr = a.out + (int64_t)r * k;
  int32_t *cnt = a.counters + (int64_t)r * 4;
  unsigned long long *cr = a.cand + (int64_t)r * DSA_CAND_CAP;

  // ---- threshold bin from the histogram (every CTA of the row, redundantly)
  {
    const int c0 = hr[2 * threadIdx.x], c1 = hr[2 * threadIdx.x + 1];
    if (threadIdx.x == 0) {  // sentinel: a histogram that yields no threshold is stale
      sm_misc[0] = DSA_NUM_BINS;
      sm_misc[1] = -1;
      sm_misc[2] = 0;
    }
    int tot;
    const int ex = block_excl_scan(c0 + c1, sm_scan, &tot);
    if (threadIdx.x == 0 && tot < k) {
      sm_misc[0] = DSA_NUM_BINS;  // every bin is "above": take all
      sm_misc[1] = tot;
      sm_misc[2] = 0;
    }
    if (ex < k && ex + c0 + c1 >= k) {
      if (ex + c0 >= k) {
        sm_misc[0] = 2 * threadIdx.x;
        sm_misc[1] = ex;
        sm_misc[2] = c0;
      } else {
        sm_misc[0] = 2 * threadIdx.x + 1;
        sm_misc[1] = ex + c0;
        sm_misc[2] = c1;
      }
    }
    __syncthreads();
  }
  const int T = sm_misc[0];
  const int above = sm_misc[1];
  const int histT = sm_misc[2];

  // ---- one pass over this CTA's chunk: emit bins above T, collect bin T
  const int64_t c0 = blockIdx.x * a.chunk;
  const int64_t c1 = min(n, c0 + a.chunk);
  const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
  for (int64_t base = c0; base < c1; base += (int64_t)kSelThreads * 4) {
    const int64_t t0 = base + threadIdx.x * 4;
    float x[4];
    if (vec && t0 + 3 < c1) {
      const float4 v = *reinterpret_cast<const float4 *>(row + t0);
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = (t0 + e < c1) ? row[t0 + e] : __int_as_float(0x7fffffff);
    }
    int ne = 0, nc = 0, bins[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      bins[e] = coarse_bin(x[e]);
      ne += (bins[e] >= 0 && bins[e] < T);
      nc += (bins[e] == T);
    }
    // warp-aggregated reservations: one atomic per warp and kind
    int ie = ne, ic = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a1 = __shfl_up_sync(0xffffffffu, ie, o);
      const int a2 = __shfl_up_sync(0xffffffffu, ic, o);
      if (lane >= o) {
        ie += a1;
        ic += a2;
      }
    }
    const int te = __shfl_sync(0xffffffffu, ie, 31), tc = __shfl_sync(0xffffffffu, ic, 31);
    int be = 0, bc = 0;
    if (lane == 31) {
      if (te) be = atomicAdd(&cnt[0], te);
      if (tc) bc = atomicAdd(&cnt[1], tc);
    }
    be = __shfl_sync(0xffffffffu, be, 31) + ie - ne;
    bc = __shfl_sync(0xffffffffu, bc, 31) + ic - nc;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (bins[e] < 0) continue;
      if (bins[e] < T) {
        if (be < k) outr[be] = (int32_t)(t0 + e);
        ++be;
      } else if (bins[e] == T) {
        if (bc < DSA_CAND_CAP) cr[bc] = cand_key(x[e], t0 + e);
        ++bc;
      }
    }
  }

  // ---- the last CTA of the row finishes it
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int prev = atomicAdd(&cnt[2], 1);
    sm_last = (prev == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!sm_last) return;
  __threadfence();
  const int emitted = *reinterpret_cast<volatile int *>(&cnt[0]);
  const int ncand = *reinterpret_cast<volatile int *>(&cnt[1]);
  const bool sane = (T < DSA_NUM_BINS) ? (above >= 0 && above < k && histT >= k - above)
                                        : (above >= 0 && above < k);
  const bool stale = !sane || (emitted != above) || (T < DSA_NUM_BINS && ncand != histT);
  const bool over = !stale && T < DSA_NUM_BINS && ncand > DSA_CAND_CAP;
  if (!stale && !over) {
    if (T >= DSA_NUM_BINS) {
      for (int i = emitted + threadIdx.x; i < k; i += kSelThreads) outr[i] = -1;
    } else {
      // exact top-m of the candidates (64-bit keys are unique per row)
      const int m = k - above;
      unsigned long long prefix = 0, mask = 0;
      int need = m;
      for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += kSelThreads) sm_h[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < ncand; i += kSelThreads) {
          const unsigned long long v = cr[i];
          if ((v & mask) == prefix) atomicAdd(&sm_h[(int)((v >> shift) & 255)], 1);
        }
        __syncthreads();
        if (threadIdx.x < 32) find_digit_desc(sm_h, need, &sm_misc[4], &sm_misc[5]);
        __syncthreads();
        const int d = sm_misc[4];
        if (d < 0) {  // fewer candidates than needed: take them all
          prefix = 0;
          break;
        }
        const int hd = sm_h[d];
        need -= sm_misc[5];
        prefix |= (unsigned long long)d << shift;
        mask |= 0xFFull << shift;
        __syncthreads();
        if (need == hd) break;
      }
      if (threadIdx.x == 0) sm_misc[6] = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < ncand; i += kSelThreads) {
        const unsigned long long v = cr[i];
        if (v >= prefix) {
          const int p = atomicAdd(&sm_misc[6], 1);
          if (p < m) outr[above + p] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
        }
      }
    }
    if (a.flags && threadIdx.x == 0) a.flags[r] = 0;
  } else {
    if (a.flags && threadIdx.x == 0) a.flags[r] = stale ? 1 : 2;
    __syncthreads();
    block_radix_topk_row(row, n, k, outr, sm_h, sm_scan, sm_misc);
  }
  // leave the row's counters (and, when asked, its histogram) at zero
  __syncthreads();
  if (threadIdx.x == 0) {
    cnt[0] = 0;
    cnt[1] = 0;
    cnt[2] = 0;
  }
  if (a.reset_hist) {
    int32_t *hw = a.hist + (int64_t)r * DSA_NUM_BINS;
    for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kSelThreads) hw[i] = 0;
  }
}

// ---------------------------------------------------------------- FP16 select
constexpr int kF16MaxRow = 16384;

__global__ void __launch_bounds__(kSelThreads)
    topk_fp16_kernel(const uint16_t *scores, int64_t stride, const int32_t *valid_lens, int k,
                     const int32_t *table, int kb, int32_t *out, uint32_t *status) {
  __shared__ uint32_t keys2[kF16MaxRow / 2];  // two 16-bit keys per word
  __shared__ int h[DSA_NUM_BINS];
  __shared__ int sm_scan[kSelWarps + 1];
  __shared__ int sm_misc[8];
  const int r = blockIdx.x;
  int64_t n = valid_lens[r];
  if (n < 0) n = 0;
  if (n > kF16MaxRow || n > stride) {
    if (threadIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
    n = min((int64_t)kF16MaxRow, stride);
  }
  const uint32_t *row = reinterpret_cast<const uint32_t *>(scores + (int64_t)r * stride);
  const int nw = (int)((n + 1) / 2);
  for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kSelThreads) h[i] = 0;
  __syncthreads();
  // keys, with positions >= n masked to the invalid key 0; coarse histogram
  for (int w = threadIdx.x; w < nw; w += kSelThreads) {
    uint32_t kk = f16x2_order_keys(row[w]);
    if (2 * w + 1 >= n) kk &= 0x0000FFFFu;
    keys2[w] = kk;
    const uint32_t lo = kk & 0xFFFFu, hi = kk >> 16;
    if (lo) atomicAdd(&h[lo >> 6], 1);
    if (hi) atomicAdd(&h[hi >> 6], 1);
  }
  __syncthreads();
  // threshold among 1024 coarse bins, searching from the top (bin 1023)
  {
    const int b0 = DSA_NUM_BINS - 1 - 2 * threadIdx.x;  // this thread's two bins, descending
    const int c0 = h[b0], c1 = h[b0 - 1];
    int tot;
    const int ex = block_excl_scan(c0 + c1, sm_scan, &tot);
    if (threadIdx.x == 0 && tot < k) {
      sm_misc[0] = -1;
      sm_misc[1] = tot;
    }
    if (ex < k && ex + c0 + c1 >= k) {
      if (ex + c0 >= k) {
        sm_misc[0] = b0;
        sm_misc[1] = ex;
      } else {
        sm_misc[0] = b0 - 1;
        sm_misc[1] = ex + c0;
      }
    }
    __syncthreads();
  }
  const int T10 = sm_misc[0];
  int above = sm_misc[1];
  uint32_t thr = 0;   // exact 16-bit threshold key
  int need = 0;       // entries equal to thr still to take
  bool take_all = (T10 < 0);
  if (!take_all) {
    // refine the remaining 6 bits inside bin T10
    if (threadIdx.x < 64) h[threadIdx.x] = 0;
    __syncthreads();
    for (int w = threadIdx.x; w < nw; w += kSelThreads) {
      const uint32_t kk = keys2[w];
      const uint32_t lo = kk & 0xFFFFu, hi = kk >> 16;
      if (lo && (int)(lo >> 6) == T10) atomicAdd(&h[lo & 63], 1);
      if (hi && (int)(hi >> 6) == T10) atomicAdd(&h[hi & 63], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = above;
      sm_misc[2] = 0;
      sm_misc[3] = above;
      for (int d = 63; d >= 0; --d) {
        if (acc + h[d] >= k) {
          sm_misc[2] = d;
          sm_misc[3] = acc;
          break;
        }
        acc += h[d];
      }
    }
    __syncthreads();
    thr = ((uint32_t)T10 << 6) | (uint32_t)sm_misc[2];
    above = sm_misc[3];
    need = k - above;
  }
  if (threadIdx.x == 0) sm_misc[4] = 0;
  __syncthreads();
  int32_t *outr = out + (int64_t)r * k;
  auto emit_col = [&](int p) -> int32_t {
    return table ? (int32_t)(table[(int64_t)r * kb + p / 8] * 8 + (p & 7)) : (int32_t)p;
  };
  // emission: keys above thr anywhere; keys equal to thr by position order
  int eq_base = 0;
  for (int base = 0; base < nw; base += kSelThreads * 2) {
    int eqc = 0;
    bool eqf[4];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int w = base + threadIdx.x * 2 + e;
      const uint32_t kk = (w < nw) ? keys2[w] : 0u;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t key = hh ? (kk >> 16) : (kk & 0xFFFFu);
        eqf[2 * e + hh] = false;
        if (!key) continue;
        const bool sel = take_all ? true : key > thr;
        if (sel) {
          const int p = atomicAdd(&sm_misc[4], 1);
          if (p < k) outr[p] = emit_col(2 * w + hh);
        } else if (!take_all && key == thr) {
          eqf[2 * e + hh] = true;
          ++eqc;
        }
      }
    }
    int tot;
    const int ex = block_excl_scan(eqc, sm_scan, &tot);
    int rank = eq_base + ex;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (!eqf[q]) continue;
      if (rank < need) outr[above + rank] = emit_col(2 * (base + threadIdx.x * 2 + q / 2) + (q & 1));
      ++rank;
    }
    eq_base += tot;
  }
  __syncthreads();
  const int written = take_all ? sm_misc[4] : k;
  for (int i = written + threadIdx.x; i < k; i += kSelThreads) outr[i] = -1;
}

}  // namespace

dsa_status_t run_topk(const TopkCall &c, cudaStream_t st) {
  char *ws = static_cast<char *>(c.workspace);
  uint32_t *status = reinterpret_cast<uint32_t *>(ws + WsLayout::kStatusOff);
  int32_t *counters = reinterpret_cast<int32_t *>(ws + WsLayout::counters_off());
  unsigned long long *cand = reinterpret_cast<unsigned long long *>(ws + WsLayout::cand_off(c.ws_rows));
  int32_t *ws_hist = reinterpret_cast<int32_t *>(ws + WsLayout::hist_off(c.ws_rows));
  const int sms = num_sms();
  if (sms <= 0) return DSA_ERR_CUDA;
  const int64_t total = c.stride * (int64_t)c.R;
  int64_t chunk = (total + 2LL * sms - 1) / (2LL * sms);
  chunk = std::max<int64_t>(2048, (chunk + 2047) / 2048 * 2048);
  const int64_t nchunks = std::max<int64_t>(1, (c.stride + chunk - 1) / chunk);
  if (nchunks > 65535 || c.R > 65535) return DSA_ERR_UNSUPPORTED;
  int32_t *hist = c.histogram;
  bool reset = c.reset_histogram;
  if (!hist) {
    hist = ws_hist;  // zero by contract; the select below clears it again
    reset = true;
    hist_build_kernel<<<dim3((unsigned)nchunks, (unsigned)c.R), kSelThreads, 0, st>>>(
        c.logits, c.stride, c.context_lens, c.next_n, c.len_div, chunk, hist, status);
    dsa_status_t e = check_launch();
    if (e != DSA_OK) return e;
  }
  SelArgs a;
  a.logits = c.logits;
  a.stride = c.stride;
  a.ctx = c.context_lens;
  a.next_n = c.next_n;
  a.len_div = c.len_div;
  a.R = c.R;
  a.hist = hist;
  a.reset_hist = reset ? 1 : 0;
  a.k = c.k;
  a.out = c.out_idx;
  a.flags = c.fallback_flags;
  a.counters = counters;
  a.cand = cand;
  a.status = status;
  a.chunk = chunk;
  select_kernel<<<dim3((unsigned)nchunks, (unsigned)c.R), kSelThreads, 0, st>>>(a);
  return check_launch();
}

dsa_status_t run_topk_fp16(const Fp16TopkCall &c, cudaStream_t st) {
  topk_fp16_kernel<<<c.R, kSelThreads, 0, st>>>(c.scores, c.stride, c.valid_lens, c.k,
                                                c.block_table, c.kb, c.out_idx, c.status);
  return check_launch();
}

}  // namespace dsa
