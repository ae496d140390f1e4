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
  if (len_div > 1) n = (n + len_div - 1) / len_div;
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
  int32_t *counters;              // [R][4]: emitted, candidates, done CTAs, level-1 state
  unsigned long long *cand;       // [R][DSA_CAND_CAP]
  int32_t *fine;                  // [R][kFineBins] fine histogram of an overflowing bin
  uint32_t *status;
  int64_t chunk;
};

constexpr int kFineBits = 12;
constexpr int kFineBins = 1 << kFineBits;
constexpr int kSelSmem = 32768;              // fine histogram (pass) / candidates (refine)
constexpr int kSmemCand = kSelSmem / 8;      // candidates refined from shared memory
constexpr int kPerThread = 16;               // elements per thread per pass iteration
constexpr int kIter = kSelThreads * kPerThread;

__device__ __forceinline__ unsigned long long cand_key(float x, int64_t t) {
  return ((unsigned long long)f32_order_key(x) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)t);
}

// Fine bins of a coarse bin T: an enclosing range of |x| is known in closed
// form from the bin rules (saturating: resolution spent on 223 <= |x| < 2^16;
// unit bins: [n, n+1); FP16 bins: between the neighbouring half codes); the
// range is mapped to order keys and spread over kFineBins fine bins.  The map
// is clamped, so it stays monotone (and the select exact) whatever the range.
__device__ void fine_map(int T, uint32_t *klo, int *shift) {
  const bool neg = T >= 512;
  const int m = neg ? T - 512 : 511 - T;  // magnitude code
  float alo, ahi;
  if (m >= 511) {
    alo = 223.0f;
    ahi = 65536.0f;
  } else if (m >= 304) {
    alo = (m == 304) ? 15.99f : (float)(m - 288);
    ahi = (float)(m - 287);
  } else {
    alo = (m == 0) ? 0.0f : __half2float(__ushort_as_half((unsigned short)(64 * m - 1)));
    ahi = __half2float(__ushort_as_half((unsigned short)(64 * m + 64)));
  }
  const uint32_t k1 = f32_order_key(neg ? -ahi : alo);
  const uint32_t k2 = f32_order_key(neg ? -alo : ahi);
  const uint32_t lo = min(k1, k2), hi = max(k1, k2);
  const uint64_t span = (uint64_t)(hi - lo) + 1;
  int bits = 0;
  while (bits < 33 && (1ull << bits) < span) ++bits;
  *klo = lo;
  *shift = bits > kFineBits ? bits - kFineBits : 0;
}

// Fine bin of a key inside bin T, descending like the coarse bins: fine bin 0
// holds the largest keys of the bin.
__device__ __forceinline__ int fine_bin(uint32_t key, uint32_t klo, int shift) {
  const int64_t off = (int64_t)key - (int64_t)klo;
  const int64_t f = off <= 0 ? 0 : min((int64_t)(kFineBins - 1), off >> shift);
  return (kFineBins - 1) - (int)f;
}

__device__ __forceinline__ int bitlen64(unsigned long long v) { return v ? 64 - __clzll((long long)v) : 0; }

// Threshold of the top m of the n keys keys[0..n) (key 0 = invalid), found by
// a range-adaptive MSB radix select run by the whole block: every pass spreads
// the active key range [lo, hi] over 256 digits, so bits all keys share cost
// nothing and smooth data does not pile onto one counter.  Result:
//   inclusive  -> the top m are exactly the valid keys >= thr
//   !inclusive -> they are the n_gt keys > thr plus need_eq keys == thr
// Scratch: h[256], red[2] (same type as the keys), imisc[8].
template <typename K, int NT>
__device__ void adaptive_threshold(const K *keys, int n, int m, int *h, K *red, int *imisc,
                                   K &thr, int &n_gt, int &need_eq, bool &inclusive) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    red[0] = ~(K)0;
    red[1] = 0;
    imisc[0] = 0;
  }
  __syncthreads();
  K lo = ~(K)0, hi = 0;
  int cnt = 0;
  for (int i = threadIdx.x; i < n; i += NT) {
    const K kk = keys[i];
    if (kk == 0) continue;
    lo = min(lo, kk);
    hi = max(hi, kk);
    ++cnt;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, (K)__shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, (K)__shfl_xor_sync(0xffffffffu, hi, o));
    cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  }
  if (lane == 0) {
    atomicMin(&red[0], lo);
    atomicMax(&red[1], hi);
    atomicAdd(&imisc[0], cnt);
  }
  __syncthreads();
  lo = red[0];
  hi = red[1];
  const int nvalid = imisc[0];
  __syncthreads();
  n_gt = 0;
  need_eq = 0;
  if (nvalid <= m) {  // every valid key is taken
    thr = 1;
    inclusive = true;
    return;
  }
  int need = m;
  while (true) {
    if (lo == hi) {
      thr = lo;
      need_eq = need;
      inclusive = false;
      return;
    }
    const int shift = max(0, bitlen64((unsigned long long)(hi - lo)) - 8);
    for (int i = threadIdx.x; i < 256; i += NT) h[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += NT) {
      const K kk = keys[i];
      if (kk == 0 || kk < lo || kk > hi) continue;
      atomicAdd(&h[(int)((kk - lo) >> shift)], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) find_digit_desc(h, need, &imisc[1], &imisc[2]);
    __syncthreads();
    const int d = imisc[1];
    if (d < 0) {  // cannot happen for consistent counts: take what is active
      __syncthreads();
      thr = lo;
      inclusive = true;
      return;
    }
    const int hd = h[d];
    n_gt += imisc[2];
    need -= imisc[2];
    const K nlo = lo + ((K)d << shift);
    const K width = ((K)1 << shift) - 1;  // last key of the digit is nlo + width
    const K nhi = (hi - nlo > width) ? (K)(nlo + width) : hi;  // no wrap-around
    __syncthreads();
    if (need == hd) {  // the whole digit is taken
      thr = nlo;
      inclusive = true;
      return;
    }
    if (shift == 0) {  // one key value: ties
      thr = nlo;
      need_eq = need;
      inclusive = false;
      return;
    }
    lo = nlo;
    hi = nhi;
  }
}

// Exact top-m of n unique 64-bit keys (candidates: value order key << 32 |
// inverted column), emitted as columns to out[0..m).
__device__ __noinline__ void refine_candidates(const unsigned long long *sc, int n, int m, int32_t *out,
                                  int *sm_h, int *sm_misc, unsigned long long *sm_u64) {
  unsigned long long thr;
  int n_gt, need_eq;
  bool incl;
  adaptive_threshold<unsigned long long, kSelThreads>(sc, n, m, sm_h, sm_u64, sm_misc, thr, n_gt,
                                                      need_eq, incl);
  if (threadIdx.x == 0) sm_misc[6] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += kSelThreads) {
    const unsigned long long v = sc[i];
    if (v == 0) continue;
    if (incl ? v >= thr : (v > thr || (v == thr && need_eq > 0))) {
      const int p = atomicAdd(&sm_misc[6], 1);
      if (p < m) out[p] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
    }
  }
  __syncthreads();
}

// Exact top-k of n elements by MSB radix select over their 32-bit order keys,
// run by the whole block; key_at(i) is element i's key, 0 for an element that
// never takes part.  Ties at the threshold key go to the lowest indices
// (ordered scan).  Writes all k outputs (-1 padded).
template <class KeyAt>
__device__ __noinline__ void block_radix_topk(KeyAt key_at, int64_t n, int k, int32_t *out,
                                 int *sm_h /*256*/, int *sm_scan /*kSelWarps+1*/,
                                 int *sm_misc /*8*/) {
  uint32_t prefix = 0, mask = 0;
  int need = k;
  bool early = false;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kSelThreads) sm_h[i] = 0;
    __syncthreads();
    for (int64_t t = threadIdx.x; t < n; t += kSelThreads) {
      const uint32_t key = key_at(t);
      if (key == 0) continue;
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
      const uint32_t key = key_at(t);
      if (key == 0) continue;
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

// Exact top-k of one FP32 row (NaN never taken; ties to the lower column).
__device__ void block_radix_topk_row(const float *row, int64_t n, int k, int32_t *out,
                                     int *sm_h, int *sm_scan, int *sm_misc) {
  block_radix_topk([row](int64_t t) -> uint32_t {
    const float x = row[t];
    return isnan(x) ? 0u : f32_order_key(x);
  }, n, k, out, sm_h, sm_scan, sm_misc);
}

__global__ void __launch_bounds__(kSelThreads)
    hist_build_kernel(const float *logits, int64_t stride, const int32_t *ctx, int next_n,
                      int len_div, int64_t chunk, int32_t *hist, uint32_t *status) {
  pdl_wait();  // predecessor grids complete before any global access
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

// Threshold search over a histogram held in global memory: bin T with
// cnt(bins < T) < need <= cnt(bins <= T), bins taken in increasing index
// order (index 0 = largest scores).  Every thread calls it.  Writes
// sm_misc[0..2] = (T, count above T, count in T); T = nb when the histogram
// holds fewer than `need`, and (nb, -1, 0) when no bin qualifies (a corrupt
// histogram).
template <int NB>
__device__ __noinline__ void threshold_from_hist(const int32_t *h, int need, int *sm_scan, int *sm_misc) {
  constexpr int PER = NB / kSelThreads;
  int c[PER];
  int sum = 0;
#pragma unroll
  for (int e = 0; e < PER; ++e) {
    c[e] = h[threadIdx.x * PER + e];
    sum += c[e];
  }
  if (threadIdx.x == 0) {
    sm_misc[0] = NB;
    sm_misc[1] = -1;
    sm_misc[2] = 0;
  }
  int tot;
  const int ex = block_excl_scan(sum, sm_scan, &tot);
  if (threadIdx.x == 0 && tot < need) {
    sm_misc[0] = NB;
    sm_misc[1] = tot;
    sm_misc[2] = 0;
  }
  if (ex < need && ex + sum >= need) {
    int acc = ex;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      if (acc + c[e] >= need) {
        sm_misc[0] = threadIdx.x * PER + e;
        sm_misc[1] = acc;
        sm_misc[2] = c[e];
        break;
      }
      acc += c[e];
    }
  }
  __syncthreads();
}

// One pass of the select over this CTA's chunk of the row.
//   level 0: emit coarse bins above T; collect bin T, or -- when the
//            histogram already says bin T holds more than the candidate
//            capacity -- build a fine histogram of bin T instead
//   level 1: (rows flagged by level 0 only) emit the fine bins of bin T above
//            the fine threshold S, collect fine bin S
// The last CTA of the row checks every count against the histograms, then
// refines the candidates exactly, or flags level 1, or (stale histogram /
// fine bin over capacity) runs the exact whole-row fallback.
template <int LEVEL>
__global__ void __launch_bounds__(kSelThreads) select_kernel(const SelArgs a) {
  pdl_wait();  // predecessor grids complete before any global access
  extern __shared__ unsigned long long sm_dyn[];  // fine hist (pass) / candidates (refine)
  __shared__ int sm_h[256];
  __shared__ int sm_scan[kSelWarps + 1];
  __shared__ int sm_misc[16];
  __shared__ unsigned long long sm_u64[2];
  __shared__ int sm_last;
  const int r = blockIdx.y;
  const int k = a.k;
  const int lane = threadIdx.x & 31;
  int32_t *cnt = a.counters + (int64_t)r * 4;
  if (LEVEL == 1 && *reinterpret_cast<volatile int *>(&cnt[3]) == 0) return;
  const int64_t n = row_len(a.ctx, a.next_n, a.len_div, r, a.stride, a.status);
  const float *row = a.logits + (int64_t)r * a.stride;
  int32_t *outr = a.out + (int64_t)r * k;
  unsigned long long *cr = a.cand + (int64_t)r * DSA_CAND_CAP;
  int32_t *finer = a.fine + (int64_t)r * kFineBins;
  int *fine_s = reinterpret_cast<int *>(sm_dyn);

  // ---- issue this CTA's first loads, then read the histogram while they fly
  const int64_t c0 = blockIdx.x * a.chunk;
  const int64_t c1 = min(n, c0 + a.chunk);
  const bool vec = ((reinterpret_cast<uintptr_t>(row) & 15) == 0);
  float x[kPerThread];
  auto load = [&](int64_t base) {
#pragma unroll
    for (int q = 0; q < kPerThread / 4; ++q) {
      const int64_t t0 = base + (int64_t)q * kSelThreads * 4 + threadIdx.x * 4;
      if (vec && t0 + 3 < c1) {
        const float4 v = *reinterpret_cast<const float4 *>(row + t0);
        x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          x[4 * q + e] = (t0 + e < c1) ? row[t0 + e] : __int_as_float(0x7fffffff);
      }
    }
  };
  if (c0 < c1) load(c0);

  // ---- coarse threshold bin (every CTA, redundantly)
  threshold_from_hist<DSA_NUM_BINS>(a.hist + (int64_t)r * DSA_NUM_BINS, k, sm_scan, sm_misc);
  const int T = sm_misc[0];
  const int above = sm_misc[1];
  const int histT = sm_misc[2];
  __syncthreads();
  const bool overflow0 = (T < DSA_NUM_BINS) && histT > DSA_CAND_CAP;

  uint32_t klo = 0;
  int fshift = 0, S = 0, above1 = 0, fineS = 0;
  if (overflow0 && LEVEL == 0) {
    for (int i = threadIdx.x; i < kFineBins; i += kSelThreads) fine_s[i] = 0;
  }
  if (overflow0) {
    if (threadIdx.x == 0) {
      uint32_t kl;
      int sh;
      fine_map(T, &kl, &sh);
      sm_misc[8] = (int)kl;
      sm_misc[9] = sh;
    }
    __syncthreads();
    klo = (uint32_t)sm_misc[8];
    fshift = sm_misc[9];
  }
  if (LEVEL == 1) {
    threshold_from_hist<kFineBins>(finer, k - above, sm_scan, sm_misc + 10);
    S = sm_misc[10];
    above1 = sm_misc[11];
    fineS = sm_misc[12];
    __syncthreads();
  }

  // ---- the pass
  int *cnt_e = &cnt[0];
  int *cnt_c = &cnt[1];
  for (int64_t base = c0; base < c1; base += kIter) {
    if (base != c0) load(base);
    // kind: 1 = emit, 2 = candidate, 3 = count into the fine histogram
    uint32_t kinds = 0;
    int ne = 0, nc = 0;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const int b = coarse_bin(x[e]);
      uint32_t kd = 0;
      if (b >= 0) {
        if (LEVEL == 0) {
          if (b < T) kd = 1;
          else if (b == T) kd = overflow0 ? 3 : 2;
        } else if (b == T) {
          const int f = fine_bin(f32_order_key(x[e]), klo, fshift);
          if (f < S) kd = 1;
          else if (f == S) kd = 2;
        }
      }
      kinds |= kd << (2 * e);
      ne += (kd == 1);
      nc += (kd >= 2);
    }
    const unsigned any = __ballot_sync(0xffffffffu, (ne | nc) != 0);
    if (any == 0) continue;  // warp-uniform: nothing to emit or collect here
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
      if (te) be = atomicAdd(cnt_e, te);
      if (tc) bc = atomicAdd(cnt_c, tc);
    }
    be = __shfl_sync(0xffffffffu, be, 31) + ie - ne;
    bc = __shfl_sync(0xffffffffu, bc, 31) + ic - nc;
#pragma unroll
    for (int e = 0; e < kPerThread; ++e) {
      const uint32_t kd = (kinds >> (2 * e)) & 3u;
      if (!kd) continue;
      const int64_t t = base + (int64_t)(e >> 2) * kSelThreads * 4 + threadIdx.x * 4 + (e & 3);
      if (kd == 1) {
        if (be < k) outr[be] = (int32_t)t;
        ++be;
      } else if (kd == 2) {
        if (bc < DSA_CAND_CAP) cr[bc] = cand_key(x[e], t);
        ++bc;
      } else {
        atomicAdd(&fine_s[fine_bin(f32_order_key(x[e]), klo, fshift)], 1);
        ++bc;
      }
    }
  }
  if (LEVEL == 0 && overflow0) {
    __syncthreads();
    for (int p = threadIdx.x; p < kFineBins / 2; p += kSelThreads) {
      const uint32_t f0 = fine_s[2 * p], f1 = fine_s[2 * p + 1];
      if (f0 | f1)
        atomicAdd(reinterpret_cast<unsigned long long *>(finer + 2 * p),
                  ((unsigned long long)f1 << 32) | f0);
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
  const bool sane0 = (T < DSA_NUM_BINS) ? (above >= 0 && above < k && histT >= k - above)
                                        : (above >= 0 && above < k);
  int flag = 0;           // 0 histogram path, 1 stale, 2 over capacity
  bool done = true;       // false: level 1 continues this row
  int base_out = 0, m = 0;
  if (LEVEL == 0) {
    const bool stale = !sane0 || emitted != above || (T < DSA_NUM_BINS && ncand != histT);
    if (stale) {
      flag = 1;
    } else if (overflow0) {
      done = false;       // fine histogram complete: level 1 collects bin S
    } else {
      base_out = above;
      m = (T < DSA_NUM_BINS) ? k - above : 0;
    }
  } else {
    const bool sane1 = S < kFineBins && above1 >= 0 && above1 < k - above;
    const bool stale = !sane1 || emitted != above + above1 || ncand != fineS;
    if (stale) flag = 1;
    else if (ncand > DSA_CAND_CAP) flag = 2;
    else {
      base_out = above + above1;
      m = k - base_out;
    }
  }
  if (!done) {
    if (threadIdx.x == 0) {
      cnt[1] = 0;
      cnt[2] = 0;
      cnt[3] = 1;
    }
    return;
  }
  if (flag == 0) {
    if (m > 0) {
      // small candidate sets are refined from shared memory, larger ones
      // straight from the (L2-resident) workspace buffer
      const unsigned long long *src = cr;
      if (ncand <= kSmemCand) {
        for (int i = threadIdx.x; i < ncand; i += kSelThreads) sm_dyn[i] = cr[i];
        __syncthreads();
        src = sm_dyn;
      }
      refine_candidates(src, ncand, m, outr + base_out, sm_h, sm_misc, sm_u64);
    } else {
      for (int i = emitted + threadIdx.x; i < k; i += kSelThreads) outr[i] = -1;
    }
  } else {
    __syncthreads();
    block_radix_topk_row(row, n, k, outr, sm_h, sm_scan, sm_misc);
  }
  if (a.flags && threadIdx.x == 0) a.flags[r] = flag;
  // leave the row's counters, fine histogram and (when asked) histogram at zero
  __syncthreads();
  if (threadIdx.x == 0) {
    cnt[0] = 0;
    cnt[1] = 0;
    cnt[2] = 0;
    cnt[3] = 0;
  }
  if (LEVEL == 1 || overflow0)
    for (int i = threadIdx.x; i < kFineBins; i += kSelThreads) finer[i] = 0;
  if (a.reset_hist) {
    int32_t *hw = a.hist + (int64_t)r * DSA_NUM_BINS;
    for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kSelThreads) hw[i] = 0;
  }
}

// ---------------------------------------------------------------- cluster select
// One launch selects the rows of up to kClMaxProb independent problems.
// Long rows (stride > kClChunk): one cluster of kCl CTAs per row, each CTA
// holding its share of the row as order keys in shared memory (the row is
// read from memory once):
//   1. threshold bin T from the caller's histogram (worked out while the row
//      loads), or from one the CTAs merge in the workspace (global
//      reductions, resolved in L2, one cluster barrier)
//   2. the exact key range [loT, hiT] of bin T (coarse bins descend with the
//      key, so every bin is one key range), in closed form
//   3. when bin T holds more than kClDirect scores: a fine histogram over a
//      window of bin T's key range, merged in the workspace the same way, and
//      the fine threshold bin S
//   4. every CTA classifies its scores against the emit threshold E (emit:
//      key > E; candidate: C <= key <= E), reserves output and candidate
//      ranges with one DSMEM atomic per warp on CTA 0, and writes them
//   5. CTA 0 checks the counts and ranks the candidates (or refines them, or
//      runs the exact whole-row fallback)
// With a block output the top-bk blocks of 8 scores by block maximum come out
// of the same pass without a histogram of the maxima: a block whose maximum
// is above E holds an emitted score, and every block at or below E ranks
// below every block above it, so when at least bk blocks (the newest one
// counted as +inf) lie above E, the top bk of the row are the top bk of those
// -- at most k blocks, collected in CTA 1's shared memory and selected
// exactly there.  Rows with fewer such blocks (scores crowded into few
// blocks) take the exact whole-row select over every block maximum, also on
// CTA 1.
// Short rows (stride <= kClChunk): each CTA of a cluster takes one row alone
// (the same steps inside one CTA, no cluster barrier), eight rows a cluster.
// Rows of at most kClRow / 2 scores, when one row a cluster would need more
// clusters than one wave holds: two rows a cluster, four CTAs each (each half
// has its own CTA 0 and CTA 1; both halves pass every cluster barrier).
// Every cluster-wide decision is taken from data all CTAs share, so all CTAs
// pass the same cluster barriers.  The workspace histograms are zero on entry
// and are cleared again by CTA 0 after the last barrier.
constexpr int kCl = 8;
constexpr int kClThreads = 512;
constexpr int kClVpt = 32;                       // scores per thread
constexpr int kClVec = kClVpt / 4;               // float4 groups per thread
constexpr int kClChunk = kClThreads * kClVpt;    // 16384 per CTA
constexpr int kClRow = kCl * kClChunk;           // 131072
constexpr int kClDirect = kClThreads;            // candidates kept in shared memory
constexpr int kClRank = 64;                      // items of a histogram level's bin ranked pairwise
constexpr int kClRankDirect = 256;               // score candidates ranked pairwise before any level
constexpr int kClMaxProb = 4;                    // problems per launch
constexpr int kClFine = 1024;                    // fine bins
constexpr uint32_t kFineWindow = 1u << 26;       // keys one fine histogram spans at most
static_assert(kClThreads == kSelThreads, "block scans assume kSelThreads threads");

constexpr int kClBlk = kClChunk / 8;             // block maxima per CTA
constexpr int kClBPer = kClBlk / kClThreads;     // block maxima per thread
constexpr int kBSel = DSA_MAX_TOPK;              // block candidates kept (blocks above E)
constexpr int kClGroups = 4;                     // bulk-copy groups of a CTA's scores
constexpr int kClGroupVec = kClVec / kClGroups;  // float4 slots per thread in a group

struct ClSmem {
  uint4 keys[kClVec * kClThreads];      // keys[q * kClThreads + tid] = slots 4q..4q+3 of tid
  int hist[DSA_NUM_BINS];               // local coarse / fine histogram, then the row's
  unsigned long long cand[kClDirect];   // the row's first candidates (CTA 0 / local CTA)
  uint32_t bkey[kClBlk];                // block maxima keys of this CTA's positions
  unsigned long long bsel[kBSel];       // block candidates (CTA 1 / local CTA)
  int fmerge[kClFine];                  // CTA 0: the cluster's fine histogram of bin T
  unsigned long long ctr;               // CTA 0: emitted | candidates << 32
  int bctr;                             // CTA 1: block candidates (or emitted blocks)
  unsigned long long bar[1 + kClGroups];  // bulk copies landed: histogram row, score groups
};
static_assert(sizeof(uint4) * kClVec * kClThreads >= sizeof(unsigned long long) * DSA_CAND_CAP,
              "the refine reuses the key buffer for the candidates");
static_assert(sizeof(uint4) * kClVec * kClThreads >= sizeof(uint32_t) * (kClRow / 8),
              "the whole-row block select keeps every block maximum in the key buffer");
static_assert(kClBlk >= DSA_MAX_TOPK, "the block-key buffer holds the chosen block ids");

struct ClProb {
  const float *logits;
  int64_t stride;
  const int32_t *ctx;
  int next_n, len_div, R;
  int32_t *hist;  // caller's histogram, or NULL
  int reset_hist;
  int k;
  int32_t *out;
  int32_t *flags;
  int32_t *bout;  // block output [R][bk], or NULL (bk = 0)
  int32_t *bflags;
  int bk;
  int ws_row0;    // first workspace row of this problem
  int local;      // 1: rows of at most kClChunk, one CTA per row; 2: rows of at
                  // most kClRow / 2, two rows per cluster (four CTAs each); 0:
                  // one row per cluster
  int vec;        // rows 16-byte aligned: vector loads
  // block output as the sorted block table, or bpt = NULL
  const int32_t *bpt;
  int64_t bpt_stride;
  int bps;
  int32_t *bphys;
  int32_t *bvalid;
};

struct ClArgs {
  ClProb p[kClMaxProb];
  int cl_begin[kClMaxProb + 1];  // first cluster (blockIdx.y) of each problem
  int nprob;
  unsigned long long *cand;  // [workspace rows][DSA_CAND_CAP]
  int32_t *ws_hist;          // [workspace rows][DSA_NUM_BINS], zero on entry
  int32_t *ws_fine;          // [workspace rows][kFineBins], zero on entry
  uint32_t *status;
};

constexpr uint32_t kKeyNegInf = 0x007FFFFFu;  // order key of -inf (lowest non-NaN)
constexpr uint32_t kKeyPosInf = 0xFF800000u;  // order key of +inf (highest non-NaN)

__device__ __forceinline__ int coarse_bin_of_key(uint32_t key) {
  const uint32_t bits = (key & 0x80000000u) ? (key ^ 0x80000000u) : ~key;
  return coarse_bin(__uint_as_float(bits));
}

// Smallest magnitude with coarse magnitude code >= m (1 <= m <= 511), from
// the bin rules: 223 for the saturating code; m - 288 for the unit bins
// (codes 305..510); for codes 1..304 the midpoint between the FP16 values
// 64m - 1 and 64m, which round-to-nearest-even sends up to the even 64m.  The
// midpoint of two FP16 values is exact in FP32.
__device__ __forceinline__ float code_lo_mag(int m) {
  if (m == 511) return 223.0f;
  if (m >= 305) return (float)(m - 288);
  const float h1 = __half2float(__ushort_as_half((unsigned short)(64 * m - 1)));
  const float h2 = __half2float(__ushort_as_half((unsigned short)(64 * m)));
  return 0.5f * (h1 + h2);
}

// Exact order-key range [loT, hiT] of coarse bin T (bins descend with the
// value, so every bin is one key range); empty (loT > hiT) for T past the
// last bin.  Bin T < 512 holds x in [A(m), A(m+1)) with m = 511 - T (x >= 223
// for m = 511, x >= +0 for m = 0); bin T >= 512 holds x in (-A(m+1), -A(m)]
// with m = T - 512 (-0 for m = 0, down to -inf for m = 511).
__device__ __forceinline__ void bin_key_range(int T, uint32_t &loT, uint32_t &hiT) {
  if (T >= DSA_NUM_BINS) {
    loT = kKeyNegInf;
    hiT = kKeyNegInf - 1;
    return;
  }
  const bool pos = T < 512;
  const int m = pos ? 511 - T : T - 512;
  const float a0 = m == 0 ? 0.0f : code_lo_mag(m);
  if (pos) {
    loT = f32_order_key(a0);
    hiT = m == 511 ? kKeyPosInf : f32_order_key(code_lo_mag(m + 1)) - 1;
  } else {
    hiT = f32_order_key(-a0);
    loT = m == 511 ? kKeyNegInf : f32_order_key(-code_lo_mag(m + 1)) + 1;
  }
}

// Fine map of bin T: its key range [loT, hiT] spread over kClFine descending
// fine bins -- or, for the four bins wider than kFineWindow keys (|x| >= 223
// and |x| below the smallest FP16 step, each sign), the range [dmin, dmax] the
// row's scores in the bin actually take (dmax = 0: not known, the end of the
// bin nearer to magnitude 1 is used).  Keys outside the map clamp to the end
// bins, so the map stays monotone and the select exact.
__device__ __forceinline__ void cl_fine_window(int T, uint32_t loT, uint32_t hiT, uint32_t dmin,
                                               uint32_t dmax, uint32_t &flo, int &fshift) {
  uint32_t span1 = hiT - loT;
  flo = loT;
  if (span1 >= kFineWindow) {
    if (dmax != 0 && dmin <= dmax) {
      flo = dmin;
      span1 = dmax - dmin;
    } else {
      span1 = kFineWindow - 1;
      const bool pos = T < 512;
      const int mag = pos ? 511 - T : T - 512;
      const bool window_low = (mag == 511) ? pos : !pos;
      if (!window_low) flo = hiT - span1;
    }
  }
  fshift = 0;
  while ((span1 >> fshift) >= (uint32_t)kClFine) ++fshift;
}

__device__ __forceinline__ int cl_fine_idx(uint32_t kk, uint32_t flo, int fshift) {
  const uint32_t off = kk > flo ? kk - flo : 0u;
  return (kClFine - 1) - (int)min((uint32_t)(kClFine - 1), off >> fshift);
}

// The CTA's local histogram (nb bins) is added into the row's workspace copy.
__device__ __forceinline__ void cl_flush(const int *local, int32_t *row_ws, int nb) {
  for (int i = threadIdx.x; i < nb; i += kClThreads) {
    const int v = local[i];
    if (v) atomicAdd(&row_ws[i], v);
  }
}

// The row's merged histogram is read back from L2 (no L1: other SMs wrote it).
__device__ __forceinline__ void cl_fetch(int *local, const int32_t *row_ws, int nb) {
  const int4 *src = reinterpret_cast<const int4 *>(row_ws);
  int4 *dst = reinterpret_cast<int4 *>(local);
  for (int i = threadIdx.x; i < nb / 4; i += kClThreads) dst[i] = __ldcg(src + i);
}

// Position of slot (q, j) of this thread: c0 + 4 (q kClThreads + tid) + j.
__device__ __forceinline__ int64_t cl_pos(int64_t c0, int q, int j) {
  return c0 + 4 * ((int64_t)q * kClThreads + threadIdx.x) + j;
}

// Loads of the CTA's positions [c0, c1) into registers (NaN past c1); read
// once, so the lines are marked evict-first.  Positions of a cluster row are
// below 2^31.
__device__ __forceinline__ void cl_issue_loads(const float *row, int64_t c0, int64_t c1, int vq,
                                               bool vec, float4 (&v)[kClVec]) {
  const float nanv = __int_as_float(0x7fffffff);
  const uint64_t pol = policy_evict_first();
  const int t0 = (int)c0 + 4 * (int)threadIdx.x, e1 = (int)c1;
#pragma unroll
  for (int q = 0; q < kClVec; ++q) {
    float4 x = make_float4(nanv, nanv, nanv, nanv);
    const int t = t0 + 4 * q * kClThreads;
    if (q < vq) {
      if (vec && t + 3 < e1) {
        x = ld_f4_hint(row + t, pol);
      } else {
        if (t < e1) x.x = __ldg(row + t);
        if (t + 1 < e1) x.y = __ldg(row + t + 1);
        if (t + 2 < e1) x.z = __ldg(row + t + 2);
        if (t + 3 < e1) x.w = __ldg(row + t + 3);
      }
    }
    v[q] = x;
  }
}

// Order key, 0 for NaN (branch-free).
__device__ __forceinline__ uint32_t key_or_zero(float x) {
  const uint32_t u = __float_as_uint(x);
  const uint32_t k = u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
  return isnan(x) ? 0u : k;
}

// Key range [C, E] of fine bin S of bin T under cl_fine_idx's clamped map
// (fine bins descend): the keys of the bin are exactly C <= key <= E, and the
// keys of the fine bins above it (and of the coarse bins above T) are > E.
__device__ __forceinline__ void fine_bin_keys(uint32_t loT, uint32_t hiT, uint32_t flo, int fshift,
                                              int S, uint32_t &C, uint32_t &E) {
  const int g = (kClFine - 1) - S;  // ascending offset index
  int64_t c = (g == 0) ? (int64_t)loT : (int64_t)flo + ((int64_t)g << fshift);
  int64_t e = (g == kClFine - 1) ? (int64_t)hiT : (int64_t)flo + ((int64_t)(g + 1) << fshift) - 1;
  c = max(c, (int64_t)loT);
  e = min(e, (int64_t)hiT);
  C = (uint32_t)c;
  E = (uint32_t)e;
}

// One slot's kind: 1 = emit (key > E), 2 = candidate (C <= key <= E), else 0.
// Key 0 (NaN, padding) is never either: E >= key(-inf) - 1 > 0, C > 0.
__device__ __forceinline__ uint32_t cl_kind(uint32_t k, uint32_t C, uint32_t E) {
  return (uint32_t)(k > E) | ((uint32_t)(k >= C && k <= E) << 1);
}

// Two bits per slot e = 4q + j.
__device__ __forceinline__ unsigned long long cl_classify(const uint4 *keys, int vq, uint32_t C,
                                                          uint32_t E) {
  unsigned long long kinds = 0;
#pragma unroll
  for (int q = 0; q < kClVec; ++q) {
    if (q < vq) {
      const uint4 k4 = keys[q * kClThreads + threadIdx.x];
      const uint32_t w = cl_kind(k4.x, C, E) | (cl_kind(k4.y, C, E) << 2) |
                         (cl_kind(k4.z, C, E) << 4) | (cl_kind(k4.w, C, E) << 6);
      kinds |= (unsigned long long)w << (8 * q);
    }
  }
  return kinds;
}

// Writes this thread's emits (output slots pe, pe+1, ...) and candidates
// (candidate slots pc, pc+1, ...: the first kClDirect in the shared buffer of
// CTA 0 or of this CTA, the rest in the workspace).
__device__ __forceinline__ void cl_write(unsigned long long kinds, const uint4 *keys, int64_t c0,
                                         int pe, int pc, int k, int cap, int32_t *outr,
                                         bool remote, uint32_t cand_remote,
                                         unsigned long long *cand_local, unsigned long long *cr) {
  while (kinds) {
    const int e = (__ffsll((long long)kinds) - 1) >> 1;
    const uint32_t kd = (uint32_t)(kinds >> (2 * e)) & 3u;
    kinds &= ~(3ull << (2 * e));
    const int q = e >> 2, j = e & 3;
    const int64_t t = cl_pos(c0, q, j);
    if (kd == 1) {
      if (pe < k) outr[pe] = (int32_t)t;
      ++pe;
    } else {
      const uint32_t kk = reinterpret_cast<const uint32_t *>(&keys[q * kClThreads + threadIdx.x])[j];
      const unsigned long long v = ((unsigned long long)kk << 32) |
                                   (unsigned long long)(0xFFFFFFFFu - (uint32_t)t);
      if (pc < kClDirect) {
        if (remote) dsmem_st64(cand_remote + 8u * (uint32_t)pc, v);
        else cand_local[pc] = v;
      } else if (pc < cap) {
        cr[pc] = v;
      }
      ++pc;
    }
  }
}

// Rank of v among the n unique items a[0..n): the number of larger items
// (every thread of a rank pass reads the same items: broadcast loads).
__device__ __forceinline__ int rank_of(const unsigned long long *a, int n, unsigned long long v) {
  int rk = 0;
  for (int j = 0; j < n; ++j) rk += a[j] > v;
  return rk;
}

// Exact top-m of the n unique items it[0..n) (order key << 32 | ~id, so
// equal keys rank by lower id), written as ids to out[0..m) in any order;
// every item's key lies in [lo, hi] and n >= m.  Level by level a 1024-bin
// histogram of the keys still in play -- the coarse score bins at the first
// level when `coarse`, else an even split of [lo, hi] -- gives the threshold
// bin: items above it are emitted, the bin's items stay in play with [lo, hi]
// narrowed to the bin.  A threshold bin of at most kClRank items (or the one
// left after the third level) is ranked pairwise.  Run by the whole block;
// scratch: h[1024], two item buffers of n (not aliasing `it`).
__device__ __noinline__ void local_hist_select(const unsigned long long *it, int n, int m,
                                               int32_t *out, bool coarse, uint32_t lo, uint32_t hi,
                                               int *h, unsigned long long *bufA,
                                               unsigned long long *bufB, int *sm_scan,
                                               int *sm_misc) {
  const unsigned long long *src = it;
  int ns = n, base = 0, need = m;
  for (int level = 0;; ++level) {
    int shift = 0;
    if (!coarse)
      while (((hi - lo) >> shift) >= (uint32_t)kClFine) ++shift;
    for (int i = threadIdx.x; i < kClFine; i += kClThreads) h[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < ns; i += kClThreads) {
      const uint32_t k32 = (uint32_t)(src[i] >> 32);
      if (k32 >= lo && k32 <= hi)
        atomicAdd(&h[coarse ? coarse_bin_of_key(k32) : cl_fine_idx(k32, lo, shift)], 1);
    }
    __syncthreads();
    threshold_from_hist<kClFine>(h, need, sm_scan, sm_misc);
    const int T = sm_misc[0];
    uint32_t C, E;
    if (T >= kClFine) {  // fewer than `need` in play (inconsistent input): take them all
      C = lo;
      E = hi;
    } else if (coarse) {
      bin_key_range(T, C, E);
      C = max(C, lo);
      E = min(E, hi);
    } else {
      fine_bin_keys(lo, hi, lo, shift, T, C, E);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      sm_misc[4] = 0;
      sm_misc[5] = 0;
    }
    __syncthreads();
    // emit the items above the threshold bin, gather those in it
    unsigned long long *dst = (level & 1) ? bufB : bufA;
    for (int i = threadIdx.x; i < ns; i += kClThreads) {
      const unsigned long long v = src[i];
      const uint32_t k32 = (uint32_t)(v >> 32);
      if (k32 > E && k32 <= hi) {
        const int p = base + atomicAdd(&sm_misc[4], 1);
        if (p < m) out[p] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
      } else if (k32 >= C && k32 <= E) {
        dst[atomicAdd(&sm_misc[5], 1)] = v;
      }
    }
    __syncthreads();
    const int emitted = sm_misc[4], inbin = sm_misc[5];
    base += emitted;
    need -= emitted;
    __syncthreads();
    if (T >= kClFine) need = min(need, inbin);
    if (need <= 0) break;
    if (inbin <= kClRank || level == 2 || T >= kClFine || C == E) {
      // unique keys: each item's rank is the number of larger items
      for (int i = threadIdx.x; i < inbin; i += kClThreads) {
        const unsigned long long v = dst[i];
        const int rk = rank_of(dst, inbin, v);
        if (rk < need) out[base + rk] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
      }
      __syncthreads();
      break;
    }
    src = dst;
    ns = inbin;
    lo = C;
    hi = E;
    coarse = false;
  }
}

// The m-th largest (1 <= m <= n) of the n unique items it[0..n) whose keys
// lie in [lo, hi] (items outside the range are ignored; at least m lie in
// it).  Level by level a 1024-bin histogram over an even split of [lo, hi]
// gives the bin holding the m-th item, and the range narrows to that bin; a
// bin of at most kClRank items, one key wide, or left after the third level
// is ranked pairwise.  Run by the whole block; every thread gets the item.
// Scratch: h[1024], two item buffers of n (not aliasing `it`).
__device__ __noinline__ unsigned long long local_hist_kth(const unsigned long long *it, int n,
                                                          int m, uint32_t lo, uint32_t hi, int *h,
                                                          unsigned long long *bufA,
                                                          unsigned long long *bufB, int *sm_scan,
                                                          int *sm_misc,
                                                          unsigned long long *sm_res) {
  const unsigned long long *src = it;
  int ns = n, need = m;
  if (threadIdx.x == 0) *sm_res = 0;
  for (int level = 0;; ++level) {
    int shift = 0;
    while (((hi - lo) >> shift) >= (uint32_t)kClFine) ++shift;
    for (int i = threadIdx.x; i < kClFine; i += kClThreads) h[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < ns; i += kClThreads) {
      const uint32_t k32 = (uint32_t)(src[i] >> 32);
      if (k32 >= lo && k32 <= hi) atomicAdd(&h[cl_fine_idx(k32, lo, shift)], 1);
    }
    __syncthreads();
    threshold_from_hist<kClFine>(h, need, sm_scan, sm_misc);
    const int T = sm_misc[0];
    const int above = sm_misc[1];
    if (T >= kClFine) return 0ull;  // fewer than m in play: not a valid input
    uint32_t C, E;
    fine_bin_keys(lo, hi, lo, shift, T, C, E);
    need -= above;
    if (threadIdx.x == 0) sm_misc[5] = 0;
    __syncthreads();
    unsigned long long *dst = (level & 1) ? bufB : bufA;
    for (int i = threadIdx.x; i < ns; i += kClThreads) {
      const unsigned long long v = src[i];
      const uint32_t k32 = (uint32_t)(v >> 32);
      if (k32 >= C && k32 <= E) dst[atomicAdd(&sm_misc[5], 1)] = v;
    }
    __syncthreads();
    const int inbin = sm_misc[5];
    if (inbin <= kClRank || level == 2 || C == E) {
      // unique items: the one with exactly need - 1 larger items in the bin
      for (int i = threadIdx.x; i < inbin; i += kClThreads) {
        const unsigned long long v = dst[i];
        const int rk = rank_of(dst, inbin, v);
        if (rk == need - 1) *sm_res = v;
      }
      __syncthreads();
      return *sm_res;
    }
    src = dst;
    ns = inbin;
    lo = C;
    hi = E;
  }
}

// Last step of the score select, run by one CTA once every emit and
// candidate of the row is in place: check the counts, then rank or refine
// the candidates, or run the exact whole-row fallback.  Returns the fallback
// flag (0 histogram path, 1 stale histogram, 2 over capacity).
// The candidates' keys lie in [C, E] (bin T, or its fine bin S).
__device__ __noinline__ int cl_finish(const float *row, int64_t n, int k, int32_t *outr,
                                      bool take_all, int T, int above, int histT, bool fine,
                                      int S, int above1, int fineS, int emitted, int ncand,
                                      int cap, uint32_t C, uint32_t E,
                                      const unsigned long long *cand,
                                      const unsigned long long *cr, unsigned long long *scratch,
                                      int *hist, int *sm_h, int *sm_scan, int *sm_misc,
                                      unsigned long long *sm_u64) {
  const bool sane = (T < DSA_NUM_BINS) ? (above >= 0 && above < k && histT >= k - above)
                                       : (above >= 0 && above < k);
  int flag = 0, base_out = 0, m = 0;
  if (take_all) {
    m = 0;  // every non-NaN score is emitted; the rest is padding
  } else if (!sane) {
    flag = 1;
  } else if (!fine) {
    if (emitted != above || (T < DSA_NUM_BINS && ncand != histT)) flag = 1;
    base_out = above;
    m = (T < DSA_NUM_BINS) ? k - above : 0;
  } else {
    const bool sane1 = S < kClFine && above1 >= 0 && above1 < k - above;
    // emitted = above + above1 < k and ncand = fineS >= k - emitted make the
    // result exact whatever the histogram said about bin T's total
    if (!sane1 || emitted != above + above1 || ncand != fineS) flag = 1;
    else if (ncand > cap) flag = 2;
    base_out = above + above1;
    m = k - base_out;
  }
  if (flag == 0) {
    if (m <= 0) {
      for (int i = emitted + threadIdx.x; i < k; i += kClThreads) outr[i] = -1;
    } else if (ncand <= kClRankDirect) {
      // candidate keys are unique (the column is part of the key): each
      // thread ranks one against all the others (quadratic, but one pass:
      // cheaper than the two or three histogram levels that several hundred
      // candidates would take from scratch)
      if (threadIdx.x < ncand) {
        const unsigned long long v = cand[threadIdx.x];
        const int rk = rank_of(cand, ncand, v);
        if (rk < m) outr[base_out + rk] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
      }
    } else if (ncand <= kClDirect) {
      local_hist_select(cand, ncand, m, outr + base_out, false, C, E, hist, scratch,
                        scratch + kClDirect, sm_scan, sm_misc);
    } else {
      for (int i = threadIdx.x; i < ncand; i += kClThreads)
        scratch[i] = i < kClDirect ? cand[i] : __ldcg(cr + i);
      __syncthreads();
      if (3 * ncand <= DSA_CAND_CAP)
        local_hist_select(scratch, ncand, m, outr + base_out, false, C, E, hist, scratch + ncand,
                          scratch + 2 * ncand, sm_scan, sm_misc);
      else
        refine_candidates(scratch, ncand, m, outr + base_out, sm_h, sm_misc, sm_u64);
    }
  } else {
    __syncthreads();
    block_radix_topk_row(row, n, k, outr, sm_h, sm_scan, sm_misc);
  }
  return flag;
}

// Order key of the maximum of a block of 8 scores: NaN scores do not count,
// a block with no other score has key 0 (never selected).
__device__ __forceinline__ uint32_t max_key8(float4 a, float4 b) {
  return max(max(max(key_or_zero(a.x), key_or_zero(a.y)), max(key_or_zero(a.z), key_or_zero(a.w))),
             max(max(key_or_zero(b.x), key_or_zero(b.y)), max(key_or_zero(b.z), key_or_zero(b.w))));
}

// The selected block ids of a row (ids[0..bk), any order, -1 padding) become
// the sorted block table out[0..bk) -- ascending, INT32_MAX padded -- with the
// physical block of each (pool slot / 8 through the request's page-table row)
// and the row's live length (the chosen blocks hold a prefix of the live
// positions: the newest, partial block is the largest id), by a counting
// sort over a bitmap of the row's nbk blocks ([SG38944]
// sort_candidate_blocks).  A row of at most bk blocks takes the identity
// table 0 .. nbk-1, whatever was selected.  Every thread calls it; bm holds
// nbk bits.  `ids` is shared memory: once the bitmap holds them it takes the
// sorted ids, whose physical blocks are then looked up one a thread (the
// bitmap walk itself is serial within a thread's words, so no page-table
// read sits in it).
__device__ __noinline__ void cl_sort_table(int32_t *ids, int32_t *out, int bk, int64_t n,
                                           int64_t nbk,
                                           const int32_t *pt_row, int ps, int32_t *phys,
                                           int32_t *valid, uint32_t *bm, int *sm_scan,
                                           long long *sm_live) {
  const bool pow2 = (ps & (ps - 1)) == 0;
  const int lg = __ffs(ps) - 1;
  auto phys_of = [&](int64_t id) -> int32_t {
    const int tok = (int)id * 8;  // blocks of a cluster row: below 2^14
    const int pi = pow2 ? tok >> lg : tok / ps;
    const int64_t pg = __ldg(&pt_row[pi]);
    return (int32_t)((pg * ps + (tok - pi * ps)) >> 3);
  };
  if (nbk <= bk) {
    for (int i = threadIdx.x; i < bk; i += kClThreads) {
      out[i] = i < nbk ? i : INT32_MAX;
      if (phys) phys[i] = i < nbk ? phys_of(i) : INT32_MAX;
    }
    if (valid && threadIdx.x == 0) *valid = (int32_t)n;
    __syncthreads();
    return;
  }
  const int W = (int)((nbk + 31) / 32);
  for (int w = threadIdx.x; w < W; w += kClThreads) bm[w] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < bk; i += kClThreads) {
    const int32_t id = ids[i];
    if (id >= 0 && id < nbk) atomicOr(&bm[id >> 5], 1u << (id & 31));
  }
  __syncthreads();
  const int per = (W + kClThreads - 1) / kClThreads;
  const int w0 = threadIdx.x * per, w1 = min(W, w0 + per);
  int c = 0;
  for (int w = w0; w < w1; ++w) c += __popc(bm[w]);
  int total;
  int pos = block_excl_scan(c, sm_scan, &total);  // its barriers order the reads of ids above
  long long live = 0;
  for (int w = w0; w < w1; ++w) {
    uint32_t m = bm[w];
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      const int64_t id = (int64_t)w * 32 + bit;
      if (pos < bk) {
        out[pos] = (int32_t)id;
        ids[pos] = (int32_t)id;
      }
      ++pos;
      const int64_t in_blk = n - id * 8;
      live += in_blk < 8 ? in_blk : 8;
    }
  }
  if (phys) {
    __syncthreads();  // the sorted ids are in place
    const int nt = min(total, bk);
    for (int i = threadIdx.x; i < bk; i += kClThreads) phys[i] = i < nt ? phys_of(ids[i]) : INT32_MAX;
  }
  for (int i = total + threadIdx.x; i < bk; i += kClThreads) out[i] = INT32_MAX;
  if (valid) {
    live = __reduce_add_sync(0xffffffffu, (unsigned)live);
    if ((threadIdx.x & 31) == 0) sm_live[threadIdx.x >> 5] = live;
    __syncthreads();
    if (threadIdx.x == 0) {
      long long s2 = 0;
      for (int i = 0; i < kClThreads / 32; ++i) s2 += sm_live[i];
      *valid = (int32_t)s2;
    }
  }
  __syncthreads();
}

// Last step of the block select, run by one CTA: nbc block candidates (every
// block whose maximum is above the score select's E, as (key << 32 | ~block))
// are in bsel.  With at least bk of them the top bk are among them: the
// blocks at +inf (the newest one at least) are taken first, the others by
// local_hist_select over the key range they span.  Otherwise every block
// maximum of the row is recomputed into the key buffer `tab` and the exact
// whole-row select runs over them.  Returns the fallback flag (2: more
// candidates than bsel holds).
__device__ __noinline__ int cl_block_finish(const float *row, int64_t n, bool vec, int bk,
                                            int32_t *boutr, bool btake, int nbc,
                                            const unsigned long long *bsel, uint32_t *tab,
                                            int *hist, int *sm_h, int *sm_scan, int *sm_misc) {
  const int64_t nbk = (n + 7) / 8;
  if (btake) {  // every block with a valid maximum was emitted directly
    for (int i = nbc + threadIdx.x; i < bk; i += kClThreads) boutr[i] = -1;
    return 0;
  }
  if (nbc >= bk && nbc <= kBSel) {
    // key range of the finite maxima; the blocks at +inf are counted
    if (threadIdx.x == 0) {
      sm_misc[4] = -1;  // min (as unsigned)
      sm_misc[5] = 0;   // max
      sm_misc[6] = 0;           // blocks at +inf
    }
    __syncthreads();
    uint32_t lo = 0xFFFFFFFFu, hi = 0;
    int ninf = 0;
    for (int i = threadIdx.x; i < nbc; i += kClThreads) {
      const uint32_t k32 = (uint32_t)(bsel[i] >> 32);
      if (k32 >= kKeyPosInf) {
        ++ninf;
      } else {
        lo = min(lo, k32);
        hi = max(hi, k32);
      }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    ninf = __reduce_add_sync(0xffffffffu, ninf);
    if ((threadIdx.x & 31) == 0) {
      atomicMin(reinterpret_cast<unsigned int *>(&sm_misc[4]), lo);
      atomicMax(reinterpret_cast<unsigned int *>(&sm_misc[5]), hi);
      atomicAdd(&sm_misc[6], ninf);
    }
    __syncthreads();
    lo = (uint32_t)sm_misc[4];
    hi = (uint32_t)sm_misc[5];
    ninf = sm_misc[6];
    __syncthreads();
    if (ninf < bk) {
      // the blocks at +inf, in any order, then the rest
      if (threadIdx.x == 0) sm_misc[7] = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < nbc; i += kClThreads) {
        const unsigned long long v = bsel[i];
        if ((uint32_t)(v >> 32) >= kKeyPosInf)
          boutr[atomicAdd(&sm_misc[7], 1)] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
      }
      __syncthreads();
      unsigned long long *buf = reinterpret_cast<unsigned long long *>(tab);
      local_hist_select(bsel, nbc, bk - ninf, boutr + ninf, false, lo, hi, hist, buf,
                        buf + kBSel, sm_scan, sm_misc);
      return 0;
    }
  }
  for (int64_t b = threadIdx.x; b < nbk; b += kClThreads) {
    uint32_t mk;
    if (b == nbk - 1) {
      mk = kKeyPosInf;  // the newest block is always chosen
    } else if (vec) {   // a whole block of live scores, 32-byte aligned
      mk = max_key8(__ldcg(reinterpret_cast<const float4 *>(row + 8 * b)),
                    __ldcg(reinterpret_cast<const float4 *>(row + 8 * b + 4)));
    } else {
      mk = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) mk = max(mk, key_or_zero(__ldcg(row + 8 * b + j)));
    }
    tab[b] = mk;
  }
  __syncthreads();
  block_radix_topk([tab](int64_t b) { return tab[b]; }, nbk, bk, boutr, sm_h, sm_scan, sm_misc);
  return nbc > kBSel ? 2 : 0;
}

// Block-candidate histogram of a cluster row whose block output is the sorted
// table: bins of 2^kBShift keys (1/512 of a binade) above the score select's
// E, descending, the last 2 binades' worth clamped into bin 0 with +inf.
constexpr int kBShift = 14;
// Warp groups of a cluster row: 8 CTAs x 16 warps, 128 blocks (4 a thread) each.
constexpr int kWGroups = kCl * kSelWarps;

// CTA 1 of a cluster row whose block output is the sorted block table.  When
// the row has more than bk blocks and bk to kBSel block candidates (every
// block whose maximum key is above the score select's E: the top bk blocks
// are among them), the table is the bk blocks whose item (key << 32 | ~block)
// is at least V, the bk-th largest candidate item.  The candidates' histogram
// bh (built by every CTA as it stored them) gives V's bin; the candidates
// above that bin are counted, the bin's own are ranked (pairwise, or by
// local_hist_kth when many), and V is the item of rank bk - above.  Every
// CTA's blocks are one contiguous range of the row and each of its warps
// covers 128 consecutive blocks, so this CTA counts the chosen blocks of each
// warp group, and stores V and the warp groups' exclusive offsets into every
// CTA's shared memory (tab_addr: V; woff_addr: kSelWarps offsets), with the
// row's live length.  V = 0 everywhere: this CTA builds the table alone.
__device__ __forceinline__ void cl_block_publish(int64_t n, int bk, bool btake, int nbc,
                                              const unsigned long long *bsel, const int *bh,
                                              uint32_t base, int nloc, int ncl, uint32_t rbase,
                                              unsigned long long *buf, int *hist, int *sm_h,
                                              int *sm_scan, int *sm_misc,
                                              unsigned long long *sm_res, uint32_t tab_addr,
                                              uint32_t woff_addr, int32_t *valid,
                                              int32_t *bflag) {
  unsigned long long vstar = 0;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // warp group of block b: its CTA c = b / nloc (b < kCl * nloc = 8 nloc, so
  // c by three compares, not a division), then its 128-block run in the CTA
  auto wgroup = [&](int64_t b64) {
    const int b = (int)b64;
    int c = b >= 4 * nloc ? 4 : 0;  // kCl = 8: three halving steps
    c += b >= (c + 2) * nloc ? 2 : 0;
    c += b >= (c + 1) * nloc ? 1 : 0;
    return c * kSelWarps + ((b - c * nloc) >> 7);
  };
  auto live_of = [&](int64_t b) { const int64_t t = n - 8 * b; return t < 8 ? (int)t : 8; };
  if (!btake && nbc >= bk && nbc <= kBSel) {
    for (int i = threadIdx.x; i <= kWGroups; i += kClThreads) sm_h[i] = 0;  // + live length
    if (threadIdx.x == 0) {
      sm_misc[5] = 0;
      *sm_res = 0;
    }
    threshold_from_hist<kClFine>(bh, bk, sm_scan, sm_misc);
    const int Tb = sm_misc[0];
    const int need = bk - sm_misc[1];  // 1 .. the bin's count
    if (Tb < kClFine) {
      int live = 0;
      // the items of a warp mostly come from one warp group: one shared
      // atomic per distinct group
      for (int i0 = 0; i0 < nbc; i0 += kClThreads) {
        const int i = i0 + (int)threadIdx.x;
        const unsigned long long v = i < nbc ? bsel[i] : 0ull;
        const int bin = i < nbc ? cl_fine_idx((uint32_t)(v >> 32), base, kBShift) : kClFine;
        const int64_t b = (int64_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
        const bool up = bin < Tb;
        const unsigned act = __ballot_sync(0xffffffffu, up);
        if (up) {
          const int wg = wgroup(b);
          const unsigned peers = __match_any_sync(act, wg);
          if (lane == __ffs(peers) - 1) atomicAdd(&sm_h[wg], __popc(peers));
          live += live_of(b);
        } else if (bin == Tb) {
          buf[atomicAdd(&sm_misc[5], 1)] = v;
        }
      }
      __syncthreads();
      const int ni = sm_misc[5];
      if (ni <= kClRank) {
        if ((int)threadIdx.x < ni) {
          const unsigned long long v = buf[threadIdx.x];
          const int rk = rank_of(buf, ni, v);
          if (rk < need) {
            const int64_t b = (int64_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
            atomicAdd(&sm_h[wgroup(b)], 1);
            live += live_of(b);
          }
          if (rk == need - 1) *sm_res = v;
        }
        __syncthreads();
      } else {
        const uint32_t g = (uint32_t)((kClFine - 1) - Tb);
        const uint32_t lo = base + (g << kBShift);
        const uint32_t hi = Tb == 0 ? 0xFFFFFFFFu : lo + (1u << kBShift) - 1u;
        const unsigned long long vk = local_hist_kth(buf, ni, need, lo, hi, hist, buf + kBSel,
                                                     buf + 2 * kBSel, sm_scan, sm_misc, sm_res);
        for (int i = threadIdx.x; i < ni; i += kClThreads) {
          const unsigned long long v = buf[i];
          if (vk && v >= vk) {
            const int64_t b = (int64_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
            atomicAdd(&sm_h[wgroup(b)], 1);
            live += live_of(b);
          }
        }
      }
      live = (int)__reduce_add_sync(0xffffffffu, (unsigned)live);
      if (lane == 0 && live) atomicAdd(&sm_h[kWGroups], live);
      __syncthreads();
      vstar = *sm_res;
      // exclusive offsets of the warp groups in block order (warp 0, four a lane)
      if (vstar && warp == 0) {
        int c[kWGroups / 32], sum = 0;
#pragma unroll
        for (int j = 0; j < kWGroups / 32; ++j) {
          c[j] = sm_h[lane * (kWGroups / 32) + j];
          sum += c[j];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int x = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += x;
        }
        int off = incl - sum;
#pragma unroll
        for (int j = 0; j < kWGroups / 32; ++j) {
          sm_h[lane * (kWGroups / 32) + j] = off;
          off += c[j];
        }
      }
      __syncthreads();
    }
  }
  if (vstar) {
    if ((int)threadIdx.x < ncl * kSelWarps)  // the row's CTAs (rbase .. rbase + ncl - 1)
      dsmem_st32(dsmem_map(woff_addr + 4u * (threadIdx.x % kSelWarps),
                           rbase + threadIdx.x / kSelWarps),
                 sm_h[threadIdx.x]);
    if (threadIdx.x == 0) {
      if (valid) *valid = sm_h[kWGroups];
      if (bflag) *bflag = 0;
    }
  }
  if ((int)threadIdx.x < ncl) dsmem_st64(dsmem_map(tab_addr, rbase + threadIdx.x), vstar);
}

// This CTA's slice of the sorted block table: of its blocks b0 + 4t .. b0 +
// 4t + 3 (thread t; keys in bkey) those whose item is at least V, ascending,
// from the warp's table offset woff[warp], with their physical blocks (pool
// slot / 8 through the request's page-table row; pg0 is the page of the
// thread's first block when page_size is a multiple of 32, so all four of its
// blocks lie in that page).  No block barrier: warp scans only.
__device__ __forceinline__ void cl_table_slice(const uint32_t *bkey, int nloc, int64_t b0,
                                               unsigned long long vstar, const int *woff,
                                               int32_t *out, int32_t *phys, const int32_t *pt_row,
                                               int ps, int32_t pg0) {
  const int lane = threadIdx.x & 31;
  uint4 k4 = make_uint4(0u, 0u, 0u, 0u);
  if (4 * (int)threadIdx.x < nloc) k4 = reinterpret_cast<const uint4 *>(bkey)[threadIdx.x];
  const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
  const int64_t bb = b0 + 4 * (int64_t)threadIdx.x;
  uint32_t sel = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const unsigned long long item = ((unsigned long long)kv[j] << 32) |
                                    (unsigned long long)(0xFFFFFFFFu - (uint32_t)(bb + j));
    sel |= (uint32_t)(kv[j] != 0u && item >= vstar) << j;
  }
  const int c = __popc(sel);
  int incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  int pos = woff[threadIdx.x >> 5] + incl - c;
  const bool pow2 = (ps & (ps - 1)) == 0;  // page sizes are powers of two in practice
  const int lg = __ffs(ps) - 1;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (!((sel >> j) & 1u)) continue;
    const int b = (int)(bb + j);  // blocks of a cluster row: below 2^14
    out[pos] = b;
    if (phys) {
      const int tok = b * 8;
      const int pi = pow2 ? tok >> lg : tok / ps;  // page of the block, slot within it
      const int in_pg = tok - pi * ps;
      const int64_t pg = (ps % 32 == 0) ? (int64_t)pg0 : (int64_t)__ldg(&pt_row[pi]);
      phys[pos] = (int32_t)((pg * ps + in_pg) >> 3);
    }
    ++pos;
  }
}

// Bounded wait for phase 0 of `bar` (a CTA's bulk copies).  A wait that runs
// out records DSA_DEV_TIMEOUT and waits once more, bounded again: the copies
// must land before the CTA reads or leaves its shared memory.
__device__ __forceinline__ void cl_wait_copies(uint32_t bar, uint32_t *status) {
  if (mbar_try_wait(bar, 0)) return;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, 0)) {
    if (clock64() - t0 > kDefaultWaitLimit) {
      set_status(status, DSA_DEV_TIMEOUT);
      mbar_wait_drain(bar, 0, kDefaultWaitLimit);
      return;
    }
  }
}

__device__ __forceinline__ unsigned long long dsmem_atomic_add64(uint32_t addr, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.shared::cluster.add.u64 %0, [%1], %2;" : "=l"(old) : "r"(addr), "l"(v)
               : "memory");
  return old;
}

// The sorted block table of a cluster row, written by the whole cluster when
// its fast case holds: CTA 1 publishes the threshold item V and the warp
// groups' offsets (cl_block_publish), and after a cluster barrier each CTA
// writes its slice.  Returns false (V = 0) when CTA 1 must build the table
// alone.  Every CTA of the cluster calls it; `base` is the score select's
// E + 1, the bottom of the block-candidate histogram (CTA 1's sm.fmerge).
__device__ __noinline__ bool cl_table_cluster(const ClProb &p, int r, int64_t n, uint32_t rsub,
                                              uint32_t rbase, int ncl, int nloc, uint32_t base,
                                              ClSmem &sm, int *sm_h, int *sm_scan, int *sm_misc,
                                              unsigned long long *sm_u64) {
  __shared__ unsigned long long sm_tab;  // V
  __shared__ int sm_woff[kSelWarps];     // this CTA's warps' first table positions
  const int bk = p.bk;
  const int64_t bs0 = (int64_t)rsub * nloc;  // nloc: blocks a CTA
  const int32_t *pt_row = p.bpt + (int64_t)(r / p.next_n) * p.bpt_stride;
  if (rsub == 1)
    cl_block_publish(n, bk, (n + 7) / 8 <= bk, sm.bctr, sm.bsel, sm.fmerge, base, nloc, ncl,
                     rbase, reinterpret_cast<unsigned long long *>(sm.keys), sm.hist, sm_h, sm_scan,
                     sm_misc, sm_u64, smem_u32(&sm_tab), smem_u32(&sm_woff[0]),
                     p.bvalid ? p.bvalid + r : nullptr, p.bflags ? p.bflags + r : nullptr);
  int32_t pg0 = 0;  // the page of this thread's first block, read ahead of the barrier
  const int64_t bt = bs0 + 4 * (int64_t)threadIdx.x;
  if (p.bphys && p.bps % 32 == 0 && 4 * (int)threadIdx.x < nloc && bt * 8 < n)
    pg0 = __ldg(&pt_row[(int)(bt * 8) / p.bps]);
  cluster_sync();  // every CTA's V and offsets are in place
  const unsigned long long vstar = sm_tab;
  if (!vstar) return false;
  cl_table_slice(sm.bkey, nloc, bs0, vstar, sm_woff, p.bout + (int64_t)r * bk,
                 p.bphys ? p.bphys + (int64_t)r * bk : nullptr, pt_row, p.bps, pg0);
  return true;
}

// The block select and table of one row by this CTA alone: the top bk
// blocks by cl_block_finish, then (with a table to write) the counting sort
// of cl_sort_table over the chosen ids, which go to the block-key buffer
// (free after the last cluster barrier).
__device__ __noinline__ void cl_block_general(const ClProb &p, int r, int64_t n, ClSmem &sm,
                                              int *sm_h, int *sm_scan, int *sm_misc) {
  const int bk = p.bk;
  const int64_t nbk = (n + 7) / 8;
  int32_t *boutr = p.bout + (int64_t)r * bk;
  int32_t *ids = p.bpt ? reinterpret_cast<int32_t *>(sm.bkey) : boutr;
  const int flag = cl_block_finish(p.logits + (int64_t)r * p.stride, n, p.vec != 0, bk, ids,
                                   nbk <= bk, sm.bctr, sm.bsel,
                                   reinterpret_cast<uint32_t *>(sm.keys), sm.hist, sm_h, sm_scan,
                                   sm_misc);
  if (p.bflags && threadIdx.x == 0) p.bflags[r] = flag;
  if (p.bpt) {
    __syncthreads();  // the block ids are in place
    __shared__ long long sm_live[kClThreads / 32];
    cl_sort_table(ids, boutr, bk, n, nbk, p.bpt + (int64_t)(r / p.next_n) * p.bpt_stride, p.bps,
                  p.bphys ? p.bphys + (int64_t)r * bk : nullptr,
                  p.bvalid ? p.bvalid + r : nullptr, reinterpret_cast<uint32_t *>(sm.hist),
                  sm_scan, sm_live);
  }
}

__global__ void __launch_bounds__(kClThreads, 2)
    cluster_select_kernel(const __grid_constant__ ClArgs a) {
  extern __shared__ __align__(16) unsigned char cl_raw[];
  ClSmem &sm = *reinterpret_cast<ClSmem *>(cl_raw);
  __shared__ int sm_h[256];
  __shared__ int sm_scan[kSelWarps + 1];
  __shared__ int sm_misc[32];  // [0..2] T, [8..10] S
  __shared__ unsigned long long sm_u64[2];
  const uint32_t rank = cluster_ctarank();
  const int lane = threadIdx.x & 31;
  const int y = blockIdx.y;
  int pi = 0;
  while (pi + 1 < a.nprob && y >= a.cl_begin[pi + 1]) ++pi;
  const ClProb &p = a.p[pi];
  const bool local = p.local == 1;
  // two rows a cluster: CTAs 0-3 take one, 4-7 the other; every CTA still
  // passes every cluster barrier, so the rows' barrier sequences are the same
  const bool pairm = p.local == 2;
  const uint32_t rsub = pairm ? (rank & 3u) : rank;  // CTA of the row
  const uint32_t rbase = pairm ? (rank & 4u) : 0u;   // the row's first CTA
  const int ncl = pairm ? kCl / 2 : kCl;             // CTAs of the row
  const int r = local ? (y - a.cl_begin[pi]) * kCl + (int)rank
                      : pairm ? (y - a.cl_begin[pi]) * 2 + (int)(rank >> 2) : y - a.cl_begin[pi];
  if (local && r >= p.R) return;  // a local CTA passes no cluster barrier
  const int k = p.k;
  const float *row = p.logits + (int64_t)r * p.stride;
  int32_t *outr = p.out + (int64_t)r * k;
  const int64_t wr = (int64_t)p.ws_row0 + r;
  unsigned long long *cr = a.cand + wr * DSA_CAND_CAP;
  int32_t *wh = a.ws_hist + wr * DSA_NUM_BINS;
  const int32_t *hrow = p.hist ? p.hist + (int64_t)r * DSA_NUM_BINS : nullptr;
  const bool blk = p.bk > 0;  // block select alongside the score select
  const int bk = p.bk;
  // this CTA's positions: [c0, c0 + chunk) of the row's stride, in groups of
  // 2048 (one float4 per thread); cut by the stride, so the copies can start
  // before the row's live length is read
  const int64_t chunk = ((local ? p.stride : (p.stride + ncl - 1) / ncl) + 2047) / 2048 * 2048;
  const int64_t c0 = local ? 0 : (int64_t)rsub * chunk;
  const int vq = (int)(chunk / 2048);  // <= kClVec
  const int64_t b0 = c0 / 8;           // this CTA's first block
  // 16-byte aligned rows come into shared memory by bulk copies (the key
  // buffer takes the CTA's scores as they lie, then they become keys in
  // place); the caller's histogram row likewise when it is 16-byte aligned
  const bool bulk = p.vec != 0;
  const bool hbulk = hrow && ((reinterpret_cast<uintptr_t>(hrow) & 15) == 0);
  const int64_t cend = min(p.stride, c0 + chunk);
  const int64_t rbytes = (bulk && cend > c0) ? (cend - c0) * 4 : 0;  // multiple of 16
  // the scores come in kClGroups groups (group g: the float4 slots q of
  // kClGroupVec * g .. of every thread, 16 KB of consecutive scores), each on
  // its own barrier, so keys are made from one group while the next lands
  const uint32_t bar_h = smem_u32(&sm.bar[0]);
  auto bar_g = [&](int g) { return smem_u32(&sm.bar[1 + g]); };
  constexpr int64_t kGroupBytes = (int64_t)kClGroupVec * kClThreads * 16;

  // ---- set-up that reads no global memory, ahead of the predecessor's end
  if (threadIdx.x == 0) {
    sm.ctr = 0;
    sm.bctr = 0;
    for (int i = 0; i <= kClGroups; ++i) mbar_init(smem_u32(&sm.bar[i]), 1);
    fence_mbar_init();
  }
  if (!hrow)
    for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kClThreads) sm.hist[i] = 0;
  // this CTA's fine histogram of bin T lives in the candidate buffer until the
  // fine merge (CTA 0's candidates arrive only after that merge's barrier)
  int *const fh = reinterpret_cast<int *>(sm.cand);
  for (int i = threadIdx.x; i < kClFine; i += kClThreads) {
    sm.fmerge[i] = 0;
    fh[i] = 0;
  }
  __syncthreads();
  // cluster barrier A: every CTA's counters and merge buffer are zeroed; it is
  // waited for just before the first remote access
  if (!local) cluster_arrive();
  bool pending = !local;
  auto wait_pending = [&]() {
    if (pending) {
      cluster_wait();
      pending = false;
    }
  };

  pdl_wait();  // predecessor grids complete before any global access
  if ((bulk || hbulk) && threadIdx.x < 32) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_h, hbulk ? DSA_NUM_BINS * 4 : 0);
      if (hbulk) bulk_load(smem_u32(sm.hist), hrow, DSA_NUM_BINS * 4, bar_h);
    }
    if (lane <= kClGroups && lane > 0) {
      const int64_t gb = rbytes - (lane - 1) * kGroupBytes;
      mbar_arrive_expect_tx(bar_g(lane - 1), (uint32_t)(gb <= 0 ? 0 : min(gb, kGroupBytes)));
    }
    __syncwarp();
    const uint64_t pol = policy_evict_first();
    const uint32_t kdst = smem_u32(sm.keys);
    const char *src = reinterpret_cast<const char *>(row + c0);
    for (int64_t off = (int64_t)lane * 4096; off < rbytes; off += 32 * 4096)
      bulk_load_hint(kdst + (uint32_t)off, src + off, (uint32_t)min((int64_t)4096, rbytes - off),
                     bar_g((int)(off / kGroupBytes)), pol);
  }
  const int64_t n = row_len(p.ctx, p.next_n, p.len_div, r, p.stride, a.status);
  const int64_t c1 = min(n, c0 + chunk);
  const int64_t nrow = c1 > c0 ? c1 - c0 : 0;  // this CTA's live scores
  const int64_t nbk = (n + 7) / 8;             // blocks of the row
  const bool btake = nbk <= bk;                // every block is taken
  const bool take_all = n <= k;
  // T known without the row's own histogram (two rows a cluster: a row of k
  // or fewer scores builds it too, so both rows pass the same barriers)
  const bool early = hrow || (take_all && !pairm);
  float4 v[kClVec];
  if (!bulk) cl_issue_loads(row, c0, c1, vq, false, v);

  // ---- 1. threshold bin T from the caller's histogram, while the row loads
  // (rows of at most k scores take every non-NaN score: T past the last bin)
  int T = DSA_NUM_BINS, above = 0, histT = 0;
  if (hbulk) cl_wait_copies(bar_h, a.status);  // every copy lands before the CTA moves on
  if (early && !take_all) {
    threshold_from_hist<DSA_NUM_BINS>(hbulk ? sm.hist : hrow, k, sm_scan, sm_misc);
    T = sm_misc[0];
    above = sm_misc[1];
    histT = sm_misc[2];
  }
  // keys into shared memory, and the block maxima (a block of 8 scores is
  // two neighbouring threads' slots; the newest block counts as +inf)
  const float nanv = __int_as_float(0x7fffffff);
  auto convert = [&](int q, float4 x) {
    const int i = q * kClThreads + threadIdx.x;
    const uint4 kk = make_uint4(key_or_zero(x.x), key_or_zero(x.y), key_or_zero(x.z),
                                key_or_zero(x.w));
    sm.keys[i] = kk;
    if (blk) {
      uint32_t mk = max(max(kk.x, kk.y), max(kk.z, kk.w));
      mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, 1));
      const int lb = q * (kClThreads / 2) + (threadIdx.x >> 1);
      const int64_t b = b0 + lb;
      if (q >= vq || b >= nbk) mk = 0;          // slots past this CTA's positions or the row
      else if (b == nbk - 1) mk = kKeyPosInf;   // the newest block is always chosen
      if ((threadIdx.x & 1) == 0) sm.bkey[lb] = mk;
    }
  };
  if (bulk) {
#pragma unroll
    for (int q = 0; q < kClVec; ++q) {
      if (q % kClGroupVec == 0) cl_wait_copies(bar_g(q / kClGroupVec), a.status);
      const int i = q * kClThreads + threadIdx.x;
      const int64_t t = 4 * (int64_t)i;  // chunk offset of the slot's first score
      float4 x = make_float4(nanv, nanv, nanv, nanv);
      if (q < vq && t < nrow) {
        x = reinterpret_cast<const float4 *>(sm.keys)[i];
        if (t + 4 > nrow) {  // the row ends inside this slot
          if (t + 1 >= nrow) x.y = nanv;
          if (t + 2 >= nrow) x.z = nanv;
          x.w = nanv;
        }
      }
      convert(q, x);
    }
  } else {
#pragma unroll
    for (int q = 0; q < kClVec; ++q) convert(q, v[q]);
  }
  __syncthreads();
  uint32_t loT = 0, hiT = 0;  // loT > hiT: bin T empty (T past the last bin)
  bool fine = false;
  uint32_t flo = 0;
  int fshift = 0;
  // this CTA's fine histogram of bin T into fh (still zero): an even split of
  // the bin's key range, or for the four bins wider than kFineWindow keys a
  // window of that many keys at the end nearer to magnitude 1 (keys outside
  // clamp to the end bins)
  auto fine_local = [&]() {
    cl_fine_window(T, loT, hiT, 0u, 0u, flo, fshift);
    for (int q = 0; q < vq; ++q) {
      const uint4 k4 = sm.keys[q * kClThreads + threadIdx.x];
      const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (kv[j] >= loT && kv[j] <= hiT) atomicAdd(&fh[cl_fine_idx(kv[j], flo, fshift)], 1);
    }
    __syncthreads();
  };
  if (early) {
    bin_key_range(T, loT, hiT);
    fine = (T < DSA_NUM_BINS) && histT > kClDirect;
    if (fine) fine_local();
  } else {
    // ---- 2. the row's own coarse histogram (no histogram given): local,
    // then merged in the workspace behind one cluster barrier
    for (int q = 0; q < vq; ++q) {
      const uint4 k4 = sm.keys[q * kClThreads + threadIdx.x];
      const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (kv[j]) atomicAdd(&sm.hist[coarse_bin_of_key(kv[j])], 1);
    }
    __syncthreads();
    if (!local) {
      cl_flush(sm.hist, wh, DSA_NUM_BINS);
      wait_pending();
      cluster_sync();
      cl_fetch(sm.hist, wh, DSA_NUM_BINS);
      __syncthreads();
    }
    threshold_from_hist<DSA_NUM_BINS>(sm.hist, k, sm_scan, sm_misc);
    T = sm_misc[0];
    above = sm_misc[1];
    histT = sm_misc[2];
    if (take_all) {  // every non-NaN score is taken: T past the last bin
      T = DSA_NUM_BINS;
      above = histT = 0;
    }
    bin_key_range(T, loT, hiT);
    fine = (T < DSA_NUM_BINS) && histT > kClDirect;
    if (fine) fine_local();
  }

  // ---- 3. the fine threshold bin S of bin T: the CTAs' fine histograms are
  // added into CTA 0's merge buffer and read back from there
  int S = 0, above1 = 0, fineS = 0;
  uint32_t C = loT, E = hiT;
  if (fine || pairm) {  // two rows a cluster: both rows pass this barrier
    if (!local) {
      wait_pending();
      const uint32_t fm0 = dsmem_map(smem_u32(&sm.fmerge[0]), rbase);
      if (fine)
        for (int i = threadIdx.x; i < kClFine; i += kClThreads) {
          const int c = fh[i];
          if (c) dsmem_red_add(fm0 + 4u * (uint32_t)i, c);
        }
      cluster_sync();
      if (fine)
        for (int i = threadIdx.x; i < kClFine / 4; i += kClThreads)
          reinterpret_cast<int4 *>(sm.hist)[i] = dsmem_ld4(fm0 + 16u * (uint32_t)i);
      __syncthreads();
    }
    if (fine) {
      threshold_from_hist<kClFine>(local ? fh : sm.hist, k - above, sm_scan, sm_misc + 8);
      S = sm_misc[8];
      above1 = sm_misc[9];
      fineS = sm_misc[10];
      fine_bin_keys(loT, hiT, flo, fshift, S, C, E);
    }
  }

  // ---- 4. classify, reserve output and candidate ranges (scores on CTA 0,
  // blocks on CTA 1) with one atomic per warp, write.  Scores: emit when
  // key > E, candidate when C <= key <= E.  Blocks: with bk or fewer blocks in
  // the row every block with a valid maximum is emitted; otherwise every
  // block whose maximum is above E is a candidate.
  const unsigned long long kinds = cl_classify(sm.keys, vq, C, E);
  const int ne = __popcll(kinds & 0x5555555555555555ull);
  const int nc = __popcll(kinds & 0xAAAAAAAAAAAAAAAAull);
  const uint32_t EB = btake ? kKeyNegInf - 1 : E;
  uint32_t bmask = 0;
  if (blk) {
#pragma unroll
    for (int e = 0; e < kClBPer; ++e)
      bmask |= (uint32_t)(sm.bkey[threadIdx.x + e * kClThreads] > EB) << e;
  }
  const int nb = __popc(bmask);
  // warp-inclusive scans of the three counts (ne, nc <= 32; nb <= kClBPer)
  int ie = ne, ic = nc, ib = nb;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x1 = __shfl_up_sync(0xffffffffu, ie, o);
    const int x2 = __shfl_up_sync(0xffffffffu, ic, o);
    const int x3 = __shfl_up_sync(0xffffffffu, ib, o);
    if (lane >= o) {
      ie += x1;
      ic += x2;
      ib += x3;
    }
  }
  wait_pending();  // every CTA's counters are zeroed before the first remote atomic
  int we = 0, wc = 0, wb = 0;  // this warp's bases
  if (lane == 31) {
    const unsigned long long add = (unsigned long long)ie | ((unsigned long long)ic << 32);
    if (add) {
      const unsigned long long old =
          local ? atomicAdd(&sm.ctr, add)
                : dsmem_atomic_add64(dsmem_map(smem_u32(&sm.ctr), rbase), add);
      we = (int)(old & 0xFFFFFFFFull);
      wc = (int)(old >> 32);
    }
    if (ib)
      wb = local ? atomicAdd(&sm.bctr, ib)
                 : dsmem_atomic_add(dsmem_map(smem_u32(&sm.bctr), rbase + 1u), ib);
  }
  we = __shfl_sync(0xffffffffu, we, 31) + ie - ne;
  wc = __shfl_sync(0xffffffffu, wc, 31) + ic - nc;
  wb = __shfl_sync(0xffffffffu, wb, 31) + ib - nb;
  const uint32_t cand0 = local ? 0u : dsmem_map(smem_u32(&sm.cand[0]), rbase);
  if (kinds)
    cl_write(kinds, sm.keys, c0, we, wc, k, DSA_CAND_CAP, outr, !local, cand0, sm.cand, cr);
  int32_t *boutr = blk ? p.bout + (int64_t)r * bk : nullptr;
  if (bmask) {
    const uint32_t bsel1 = local ? 0u : dsmem_map(smem_u32(&sm.bsel[0]), rbase + 1u);
    // a sorted table written by the cluster: the candidates' histogram on CTA 1
    const uint32_t bh1 =
        (p.bpt && !local && !btake) ? dsmem_map(smem_u32(&sm.fmerge[0]), rbase + 1u) : 0u;
    int pb = wb;
#pragma unroll
    for (int e = 0; e < kClBPer; ++e) {
      if (!((bmask >> e) & 1u)) continue;
      const int idx = threadIdx.x + e * kClThreads;
      const int64_t b = b0 + idx;
      if (btake) {
        if (pb < bk) boutr[pb] = (int32_t)b;
      } else if (pb < kBSel) {
        const unsigned long long cv = ((unsigned long long)sm.bkey[idx] << 32) |
                                      (unsigned long long)(0xFFFFFFFFu - (uint32_t)b);
        if (local) sm.bsel[pb] = cv;
        else dsmem_st64(bsel1 + 8u * (uint32_t)pb, cv);
        if (bh1) dsmem_red_add(bh1 + 4u * (uint32_t)cl_fine_idx(sm.bkey[idx], E + 1u, kBShift), 1);
      }
      ++pb;
    }
  }
  if (!local) cluster_sync();  // all emits and candidates are in place
  else __syncthreads();

  // ---- 5. check, rank or refine, or fall back: the score select on CTA 0
  // (the local CTA), the block select on CTA 1 (the local CTA, after).  The
  // next kernel (the sparse logits over the block table) may set itself up
  // on the SMs the other CTAs leave; it waits for this grid before reading.
  pdl_release_dependents();
  unsigned long long *scratch = reinterpret_cast<unsigned long long *>(sm.keys);
  if (local || rsub == 0) {
    const int emitted = (int)(sm.ctr & 0xFFFFFFFFull);
    const int ncand = (int)(sm.ctr >> 32);
    const int flag = cl_finish(row, n, k, outr, take_all, T, above, histT, fine, S, above1, fineS,
                               emitted, ncand, DSA_CAND_CAP, C, E, sm.cand, cr, scratch, sm.hist,
                               sm_h, sm_scan, sm_misc, sm_u64);
    if (p.flags && threadIdx.x == 0) p.flags[r] = flag;
    // restore the zero workspace histogram; clear the caller's on request
    if (!local && !early)
      for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kClThreads) wh[i] = 0;
    if (p.reset_hist && p.hist) {
      int32_t *hw = p.hist + (int64_t)r * DSA_NUM_BINS;
      for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kClThreads) hw[i] = 0;
    }
  }
  // ---- 6. the sorted block table: CTA 1 works out the chosen blocks'
  // threshold item and every CTA's slice offset, then each CTA writes its
  // slice; in the general case (V = 0) CTA 1 selects and sorts alone
  const bool dtab = blk && p.bpt && !local;
  if (dtab && cl_table_cluster(p, r, n, rsub, rbase, ncl, (int)(chunk / 8), E + 1u, sm, sm_h,
                               sm_scan, sm_misc, sm_u64))
    return;
  if (blk && (local || rsub == 1)) {
    __syncthreads();  // the local CTA: the score select's finish is done with the scratch
    cl_block_general(p, r, n, sm, sm_h, sm_scan, sm_misc);
  }
}

// ---------------------------------------------------------------- short rows
// Rows of at most kSmemRow scores with no histogram given (the block maxima
// of the two-level path): one CTA per row holds the row as FP32 order keys in
// shared memory and runs the range-adaptive radix select there -- no global
// counters, no second launch.
constexpr int kSmemRow = 16384;
constexpr int kRowThreads = 1024;
constexpr int kRowWarps = kRowThreads / 32;

__device__ __forceinline__ int block_excl_scan_1024(int v, int *ws, int *total) {
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
    const int w = ws[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    ws[lane] = wi - w;
    if (lane == 31) ws[kRowWarps] = wi;
  }
  __syncthreads();
  const int res = ws[warp] + incl - v;
  *total = ws[kRowWarps];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kRowThreads)
    row_topk_kernel(const float *logits, int64_t stride, const int32_t *ctx, int next_n,
                    int len_div, int k, int32_t *out, uint32_t *status) {
  pdl_wait();  // predecessor grids complete before any global access
  extern __shared__ uint32_t keys[];  // [kSmemRow]
  __shared__ int h[256];
  __shared__ int sm_scan[kRowWarps + 1];
  __shared__ int sm_misc[8];
  __shared__ uint32_t sm_red[2];
  const int r = blockIdx.x;
  int64_t n = row_len(ctx, next_n, len_div, r, stride, status);
  if (n > kSmemRow) {
    if (threadIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
    n = kSmemRow;
  }
  const float *row = logits + (int64_t)r * stride;
  int32_t *outr = out + (int64_t)r * k;
  // order keys; NaN and positions past the row become key 0 (never chosen).
  // Thread tid owns positions e * kRowThreads + tid: all loads in flight at
  // once, and conflict-free shared-memory access in the radix passes.
  constexpr int PER = kSmemRow / kRowThreads;
  const int nn = (int)n;
  {
    float xv[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const int t = e * kRowThreads + threadIdx.x;
      xv[e] = (t < nn) ? row[t] : __int_as_float(0x7fffffff);
    }
#pragma unroll
    for (int e = 0; e < PER; ++e)
      keys[e * kRowThreads + threadIdx.x] = isnan(xv[e]) ? 0u : f32_order_key(xv[e]);
  }
  __syncthreads();
  // threshold of the top k (key 0 is only ever NaN or padding: -inf has key
  // 0x007FFFFF)
  uint32_t thr;
  int n_gt, need_eq;
  bool incl;
  adaptive_threshold<uint32_t, kRowThreads>(keys, kSmemRow, k, h, sm_red, sm_misc, thr, n_gt,
                                            need_eq, incl);
  // emit: above the threshold in any order, ties by position (ordered scan)
  if (threadIdx.x == 0) sm_misc[3] = 0;
  __syncthreads();
#pragma unroll 4
  for (int e = 0; e < PER; ++e) {
    const int t = e * kRowThreads + threadIdx.x;
    const uint32_t kk = keys[t];
    if (kk == 0) continue;
    if (incl ? kk >= thr : kk > thr) {
      const int p = atomicAdd(&sm_misc[3], 1);
      if (p < k) outr[p] = t;
    }
  }
  // ties at the threshold key, lowest positions first: here each thread
  // takes a contiguous run of positions so a block scan orders them
  const bool ties = !incl && need_eq > 0;
  const int t0 = threadIdx.x * PER;
  int eqc = 0;
  if (ties) {
    for (int e = 0; e < PER; ++e) eqc += (keys[t0 + e] == thr);
  }
  int tot;
  int rank = block_excl_scan_1024(eqc, sm_scan, &tot);
  if (ties && eqc) {
    for (int e = 0; e < PER; ++e) {
      if (keys[t0 + e] != thr) continue;
      if (rank < need_eq) outr[n_gt + rank] = t0 + e;
      ++rank;
    }
  }
  __syncthreads();
  const int written = incl ? sm_misc[3] : k;
  for (int i = written + threadIdx.x; i < k; i += kRowThreads) outr[i] = -1;
}

// ---------------------------------------------------------------- FP16 select
// [VL52696] "Why": top-k over packed 16-bit scores.  Each thread owns a
// contiguous run of words (two scores each) in registers: one pass builds the
// 10-bit coarse histogram of the order keys, a block scan finds the threshold
// bin, a second pass over the run refines the remaining 6 bits inside it (a
// warp finds the digit), and one block scan of packed counts gives every
// thread its output slots -- the keys above the threshold anywhere, the keys
// equal to it in position order (ties to the lower position).

// WPT: words a thread holds (rows of up to 2 * WPT * kSelThreads scores)
template <bool BF16, int WPT>
__global__ void __launch_bounds__(kSelThreads, 1)
    topk_fp16_kernel(const uint16_t *scores, int64_t stride, const int32_t *valid_lens, int k,
                     const int32_t *table, int kb, int32_t *out, uint32_t *status) {
  pdl_wait();  // predecessor grids complete before any global access
  __shared__ int h[DSA_NUM_BINS];
  __shared__ int sm_scan[kSelWarps + 1];
  __shared__ int sm_misc[8];
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31;
  int64_t n = valid_lens[r];
  if (n < 0) n = 0;
  constexpr int kMaxRow = 2 * WPT * kSelThreads;
  if (n > kMaxRow || n > stride) {
    if (threadIdx.x == 0) set_status(status, DSA_DEV_BOUNDS);
    n = min((int64_t)kMaxRow, stride);
  }
  const uint32_t *row = reinterpret_cast<const uint32_t *>(scores + (int64_t)r * stride);
  const int nw = (int)((n + 1) / 2);
  // this thread's words [w0, w0 + wpt), wpt a multiple of 4 (16-byte loads)
  const int wpt = ((nw + kSelThreads - 1) / kSelThreads + 3) & ~3;
  const int w0 = threadIdx.x * wpt;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kSelThreads) h[i] = 0;
  // this thread's positions [2 w0, 2 w0 + 2 wpt) are whole blocks of 8 (wpt a
  // multiple of 4): their table entries, read once here instead of once per
  // emitted position
  int32_t tab[WPT / 4];
#pragma unroll
  for (int q = 0; q < WPT / 4; ++q) {
    const int b = (2 * w0) / 8 + q;
    tab[q] = (table && 4 * q < wpt && b < kb) ? __ldg(&table[(int64_t)r * kb + b]) : 0;
  }
  uint32_t kv[WPT];  // order keys, two per word; 0 = no score
#pragma unroll
  for (int q = 0; q < WPT / 4; ++q) {
    const int w = w0 + 4 * q;
    uint32_t x[4] = {0u, 0u, 0u, 0u};
    if (4 * q < wpt) {
      if (vec && w + 3 < nw) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row + w));
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (w + e < nw) x[e] = __ldg(row + w + e);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t kk = (4 * q < wpt && w + e < nw)
                        ? (BF16 ? bf16x2_order_keys(x[e]) : f16x2_order_keys(x[e])) : 0u;
      if (2 * (w + e) + 1 >= n) kk &= 0x0000FFFFu;  // the odd position past the row
      kv[4 * q + e] = kk;
    }
  }
  __syncthreads();  // h zeroed
#pragma unroll
  for (int e = 0; e < WPT; ++e) {
    const uint32_t lo = kv[e] & 0xFFFFu, hi = kv[e] >> 16;
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
  const bool take_all = (T10 < 0);
  uint32_t thr = 0;  // exact 16-bit threshold key
  if (!take_all) {
    // the remaining 6 bits inside bin T10
    if (threadIdx.x < 64) h[threadIdx.x] = 0;
    __syncthreads();
#pragma unroll
    for (int e = 0; e < WPT; ++e) {
      const uint32_t lo = kv[e] & 0xFFFFu, hi = kv[e] >> 16;
      if (lo && (int)(lo >> 6) == T10) atomicAdd(&h[lo & 63], 1);
      if (hi && (int)(hi >> 6) == T10) atomicAdd(&h[hi & 63], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // lane l holds digits 63-2l and 62-2l (descending)
      const int d0 = 63 - 2 * lane;
      const int a0 = h[d0], a1 = h[d0 - 1];
      int incl = a0 + a1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const int ex = incl - a0 - a1;
      const unsigned m = __ballot_sync(0xffffffffu, above + incl >= k);
      const int l = m ? __ffs(m) - 1 : 31;
      if (lane == l) {
        const bool first = above + ex + a0 >= k;
        sm_misc[2] = first ? d0 : d0 - 1;
        sm_misc[3] = above + (first ? ex : ex + a0);
      }
    }
    __syncthreads();
    thr = ((uint32_t)T10 << 6) | (uint32_t)sm_misc[2];
    above = sm_misc[3];
  }
  const int need = take_all ? 0 : k - above;
  // one scan of (keys above thr, keys equal to thr) per thread, in position order
  int nsel = 0, neq = 0;
#pragma unroll
  for (int e = 0; e < WPT; ++e) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t key = hh ? (kv[e] >> 16) : (kv[e] & 0xFFFFu);
      if (!key) continue;
      if (take_all || key > thr) ++nsel;
      else if (key == thr) ++neq;
    }
  }
  int tot;
  const int ex = block_excl_scan(nsel | (neq << 16), sm_scan, &tot);
  int ps = ex & 0xFFFF, pq = ex >> 16;
  int32_t *outr = out + (int64_t)r * k;
  // position p = 2 (w0 + e) + hh lies in this thread's block e / 4
  auto emit_col = [&](int e, int p) -> int32_t {
    return table ? (int32_t)(tab[e / 4] * 8 + (p & 7)) : (int32_t)p;
  };
#pragma unroll
  for (int e = 0; e < WPT; ++e) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const uint32_t key = hh ? (kv[e] >> 16) : (kv[e] & 0xFFFFu);
      if (!key) continue;
      const int pos = 2 * (w0 + e) + hh;
      if (take_all || key > thr) {
        if (ps < k) outr[ps] = emit_col(e, pos);
        ++ps;
      } else if (key == thr) {
        if (pq < need) outr[above + pq] = emit_col(e, pos);
        ++pq;
      }
    }
  }
  const int written = take_all ? (tot & 0xFFFF) : k;
  for (int i = written + threadIdx.x; i < k; i += kSelThreads) outr[i] = -1;
}

}  // namespace

int32_t topk_launch_count(int64_t stride, bool has_histogram, bool allow_cluster) {
  if (allow_cluster && stride <= kClRow) return 1;
  if (!has_histogram && stride <= kSmemRow) return 1;
  return has_histogram ? 2 : 3;
}

bool topk_batchable(const TopkCall *calls, int count) {
  if (count < 1 || count > kClMaxProb) return false;
  for (int i = 0; i < count; ++i)
    if (!calls[i].allow_cluster || calls[i].stride > kClRow) return false;
  return true;
}

namespace {

// One cluster launch for problems whose rows are all at most kClRow long;
// problem i takes workspace rows from the sum of the earlier problems' R.
dsa_status_t run_cluster_select(const TopkCall *calls, int count, cudaStream_t st) {
  char *ws = static_cast<char *>(calls[0].workspace);
  const int64_t wrows = calls[0].ws_rows;
  ClArgs ca{};
  ca.nprob = count;
  ca.cand = reinterpret_cast<unsigned long long *>(ws + WsLayout::cand_off(wrows));
  ca.ws_hist = reinterpret_cast<int32_t *>(ws + WsLayout::hist_off(wrows));
  ca.ws_fine = reinterpret_cast<int32_t *>(ws + WsLayout::fine_off(wrows));
  ca.status = reinterpret_cast<uint32_t *>(ws + WsLayout::kStatusOff);
  // More row clusters than one wave of two CTAs an SM holds: rows of at most
  // kClRow / 2 scores (an even count of them) go two to a cluster.
  int64_t row_clusters = 0;
  for (int i = 0; i < count; ++i)
    if (calls[i].stride > kClChunk) row_clusters += calls[i].R;
  static int sm_count = 0;
  if (sm_count == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && n > 0)
      sm_count = n;
    else
      sm_count = 152;
  }
  const bool pair_rows = row_clusters * kCl > 2 * (int64_t)sm_count;
  int64_t row0 = 0, clusters = 0;
  for (int i = 0; i < count; ++i) {
    const TopkCall &c = calls[i];
    ClProb &p = ca.p[i];
    p.logits = c.logits;
    p.stride = c.stride;
    p.ctx = c.context_lens;
    p.next_n = c.next_n;
    p.len_div = c.len_div;
    p.R = c.R;
    p.hist = c.histogram;
    p.reset_hist = c.reset_histogram ? 1 : 0;
    p.k = c.k;
    p.out = c.out_idx;
    p.flags = c.fallback_flags;
    p.bout = c.block_out;
    p.bflags = c.block_flags;
    p.bk = c.block_out ? c.block_k : 0;
    p.ws_row0 = (int)row0;
    p.local = c.stride <= kClChunk ? 1
              : (pair_rows && c.stride <= kClRow / 2 && c.R % 2 == 0) ? 2 : 0;
    p.bpt = c.block_out ? c.block_pt : nullptr;
    p.bpt_stride = c.block_pt_stride;
    p.bps = c.block_ps;
    p.bphys = c.block_phys;
    p.bvalid = c.block_valid;
    p.vec = ((reinterpret_cast<uintptr_t>(c.logits) & 15) == 0 && c.stride % 4 == 0) ? 1 : 0;
    ca.cl_begin[i] = (int)clusters;
    clusters += p.local == 1 ? (c.R + kCl - 1) / kCl : p.local == 2 ? c.R / 2 : c.R;
    row0 += c.R;
  }
  ca.cl_begin[count] = (int)clusters;
  if (row0 > wrows) return DSA_ERR_WORKSPACE;
  if (clusters == 0) return DSA_OK;
  if (clusters > 65535) return DSA_ERR_UNSUPPORTED;
  const int smem = (int)sizeof(ClSmem);
  if (!ensure_smem_attr(reinterpret_cast<const void *>(cluster_select_kernel), smem))
    return DSA_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kCl, (unsigned)clusters);
  cfg.blockDim = dim3(kClThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCl;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, cluster_select_kernel, ca);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    (void)cudaGetLastError();
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // namespace

namespace {
__global__ void bin_key_ranges_kernel(uint32_t *out) {
  const int T = blockIdx.x * blockDim.x + threadIdx.x;
  if (T > DSA_NUM_BINS) return;
  uint32_t lo, hi;
  bin_key_range(T, lo, hi);
  out[2 * T] = lo;
  out[2 * T + 1] = hi;
}
}  // namespace

dsa_status_t run_bin_key_ranges(uint32_t *out, cudaStream_t st) {
  bin_key_ranges_kernel<<<(DSA_NUM_BINS + 1 + 255) / 256, 256, 0, st>>>(out);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

dsa_status_t run_topk_batch(const TopkCall *calls, int count, cudaStream_t st) {
  if (topk_batchable(calls, count)) return run_cluster_select(calls, count, st);
  for (int i = 0; i < count; ++i) {  // stream order: each call may reuse the workspace rows
    const dsa_status_t e = run_topk(calls[i], st);
    if (e != DSA_OK) return e;
  }
  return DSA_OK;
}

dsa_status_t run_topk(const TopkCall &c, cudaStream_t st) {
  char *ws = static_cast<char *>(c.workspace);
  uint32_t *status = reinterpret_cast<uint32_t *>(ws + WsLayout::kStatusOff);
  int32_t *counters = reinterpret_cast<int32_t *>(ws + WsLayout::counters_off());
  unsigned long long *cand = reinterpret_cast<unsigned long long *>(ws + WsLayout::cand_off(c.ws_rows));
  int32_t *ws_hist = reinterpret_cast<int32_t *>(ws + WsLayout::hist_off(c.ws_rows));
  int32_t *fine = reinterpret_cast<int32_t *>(ws + WsLayout::fine_off(c.ws_rows));
  const int sms = num_sms();
  if (sms <= 0) return DSA_ERR_CUDA;
  // one pass iteration (8192 scores) per CTA; longer chunks only when the
  // grid would exceed the launch limit
  int64_t chunk = kIter;
  while ((c.stride + chunk - 1) / chunk > 65535) chunk *= 2;
  const int64_t nchunks = std::max<int64_t>(1, (c.stride + chunk - 1) / chunk);
  if (nchunks > 65535 || c.R > 65535) return DSA_ERR_UNSUPPORTED;
  if (topk_batchable(&c, 1)) return run_cluster_select(&c, 1, st);
  if (!c.histogram && c.stride <= kSmemRow) {
    // short rows, no histogram: one CTA per row, the row held in shared memory
    const int smem = kSmemRow * 4;
    if (!ensure_smem_attr(reinterpret_cast<const void *>(row_topk_kernel), smem))
      return DSA_ERR_CUDA;
    dsa_status_t e = launch_pdl(row_topk_kernel, dim3(c.R), dim3(kRowThreads), (size_t)smem, st,
                                c.logits, c.stride, c.context_lens, c.next_n, c.len_div, c.k,
                                c.out_idx, status);
    if (e == DSA_OK && c.fallback_flags)
      e = cudaMemsetAsync(c.fallback_flags, 0, sizeof(int32_t) * c.R, st) == cudaSuccess
              ? DSA_OK : DSA_ERR_CUDA;
    return e;
  }
  int32_t *hist = c.histogram;
  bool reset = c.reset_histogram;
  if (!hist) {
    hist = ws_hist;  // zero by contract; the select below clears it again
    reset = true;
    dsa_status_t e = launch_pdl(hist_build_kernel, dim3((unsigned)nchunks, (unsigned)c.R),
                                dim3(kSelThreads), 0, st, c.logits, c.stride, c.context_lens,
                                c.next_n, c.len_div, chunk, hist, status);
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
  a.fine = fine;
  a.status = status;
  a.chunk = chunk;
  if (!ensure_smem_attr(reinterpret_cast<const void *>(select_kernel<0>), kSelSmem) ||
      !ensure_smem_attr(reinterpret_cast<const void *>(select_kernel<1>), kSelSmem))
    return DSA_ERR_CUDA;
  const dim3 grid((unsigned)nchunks, (unsigned)c.R);
  dsa_status_t e = launch_pdl(select_kernel<0>, grid, dim3(kSelThreads), (size_t)kSelSmem, st, a);
  if (e != DSA_OK) return e;
  return launch_pdl(select_kernel<1>, grid, dim3(kSelThreads), (size_t)kSelSmem, st, a);
}

dsa_status_t run_topk_fp16(const Fp16TopkCall &c, cudaStream_t st) {
  // words a thread holds: the fewest that cover a row of `stride` scores
  auto fn = c.bf16 ? topk_fp16_kernel<true, 16> : topk_fp16_kernel<false, 16>;
  if (c.stride <= 2 * 4 * kSelThreads) fn = c.bf16 ? topk_fp16_kernel<true, 4> : topk_fp16_kernel<false, 4>;
  else if (c.stride <= 2 * 8 * kSelThreads) fn = c.bf16 ? topk_fp16_kernel<true, 8> : topk_fp16_kernel<false, 8>;
  return launch_pdl(fn, dim3(c.R), dim3(kSelThreads), 0, st, c.scores, c.stride, c.valid_lens,
                    c.k, c.block_table, c.kb, c.out_idx, c.status);
}

}  // namespace dsa
