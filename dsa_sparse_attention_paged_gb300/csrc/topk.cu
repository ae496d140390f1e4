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
//      loads, behind an early cluster-barrier arrive), or from one the CTAs
//      merge in the workspace (global reductions, resolved in L2)
//   2. the exact key range [loT, hiT] of bin T (coarse bins descend with the
//      key, so every bin is one key range), found by a warp-parallel search
//   3. when bin T holds more than kClDirect scores: a fine histogram over a
//      window of bin T's key range, merged in the workspace the same way, and
//      the fine threshold bin S
//   4. every CTA classifies its scores, reserves its output and candidate
//      ranges with one atomic per counter on CTA 0, and writes them
//   5. CTA 0 checks the counts and ranks the candidates (or refines them, or
//      runs the exact whole-row fallback)
// Short rows (stride <= kClChunk): each CTA of a cluster takes one row alone
// (the same steps inside one CTA, no cluster barrier), eight rows a cluster.
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
constexpr int kClRank = 64;                      // candidates ranked pairwise
constexpr int kClMaxProb = 4;                    // problems per launch
constexpr int kClFine = 1024;                    // fine bins
constexpr uint32_t kFineWindow = 1u << 26;       // keys one fine histogram spans at most
static_assert(kClThreads == kSelThreads, "block scans assume kSelThreads threads");

constexpr int kClBlk = kClChunk / 8;             // block maxima per CTA
constexpr int kClCandHalf = DSA_CAND_CAP / 2;    // candidate slots per select with block output

struct ClSmem {
  uint4 keys[kClVec * kClThreads];      // keys[q * kClThreads + tid] = slots 4q..4q+3 of tid
  int hist[DSA_NUM_BINS];               // local coarse / fine histogram, then the row's
  unsigned long long cand[kClDirect];   // the row's first candidates (CTA 0 / local CTA)
  uint32_t bkey[kClBlk];                // block maxima keys of this CTA's positions
  int bhist[DSA_NUM_BINS];              // local / merged histogram of the block maxima
  unsigned long long bcand[kClDirect];  // block select: first candidates (CTA 1 / local CTA)
  int ctr[8];                           // CTA 0: emitted, candidates, bin-T count; CTA 1: same
                                        // for the block select (ctr[4..6])
  uint32_t bmm[8];                      // (~min, max) of the maxima in each wide bin
  uint32_t red[4];                      // range reductions
};
static_assert(sizeof(uint4) * kClVec * kClThreads >= sizeof(unsigned long long) * DSA_CAND_CAP,
              "the refine reuses the key buffer for the candidates");

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
  int local;      // rows of at most kClChunk: one CTA per row
  int vec;        // rows 16-byte aligned: vector loads
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

// Index of the wide coarse bins (0: x >= 223, 1: +tiny, 2: -tiny, 3: x <= -223).
__device__ __forceinline__ int wide_bin_idx(int T) {
  return T == 0 ? 0 : T == 511 ? 1 : T == 512 ? 2 : T == 1023 ? 3 : -1;
}

// Workspace slots (inside the row's fine-histogram area) where every CTA of a
// cluster publishes the key range its scores take in a wide bin: (~min, max),
// both 0 when none; CTA r writes only its own slots.
constexpr int kSlotD = 3 * kClFine;      // score select: 2 per CTA
constexpr int kSlotB = kSlotD + 2 * kCl; // block select: 8 per CTA (4 wide bins)
static_assert(kSlotB + 8 * kCl <= kFineBins, "slots fit the row's fine area");

// (~min, max) of this CTA's keys inside [lo, hi] into red[0], red[1] (0 when
// none); every thread calls it; ends with a __syncthreads.
__device__ __noinline__ void cl_range_in(const uint4 *keys, int vq, uint32_t lo, uint32_t hi, uint32_t *red) {
  if (threadIdx.x == 0) {
    red[0] = 0;
    red[1] = 0;
  }
  __syncthreads();
  uint32_t nmin = 0, mx = 0;
  for (int q = 0; q < vq; ++q) {
    const uint4 k4 = keys[q * kClThreads + threadIdx.x];
    const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (kv[j] >= lo && kv[j] <= hi) {
        nmin = max(nmin, ~kv[j]);
        mx = max(mx, kv[j]);
      }
  }
  nmin = __reduce_max_sync(0xffffffffu, nmin);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if ((threadIdx.x & 31) == 0 && mx) {
    atomicMax(&red[0], nmin);
    atomicMax(&red[1], mx);
  }
  __syncthreads();
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

__device__ __forceinline__ void cl_store_keys(const float4 (&v)[kClVec], uint4 *keys) {
#pragma unroll
  for (int q = 0; q < kClVec; ++q)
    keys[q * kClThreads + threadIdx.x] = make_uint4(key_or_zero(v[q].x), key_or_zero(v[q].y),
                                                    key_or_zero(v[q].z), key_or_zero(v[q].w));
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

// Last step of a row, run by one CTA once every emit and candidate of the row
// is in place: check the counts, then rank or refine the candidates, or run
// the exact whole-row fallback.  Returns the fallback flag.
// Order key of the maximum of block b (scores 8b .. 8b+7) of a row of n
// scores: NaN scores do not count, a block with no other score has key 0
// (never selected), and the newest block (the last one) counts as +inf.
__device__ __forceinline__ uint32_t block_max_key(const float *row, int64_t n, int64_t b) {
  if (b == (n + 7) / 8 - 1) return kKeyPosInf;
  uint32_t m = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int64_t t = 8 * b + j;
    if (t < n) {
      const float x = row[t];
      if (!isnan(x)) m = max(m, f32_order_key(x));
    }
  }
  return m;
}

// Elements are the row's scores, or (maxima) the maxima of its blocks of 8
// scores: n elements, n_scores scores; `cap` candidate slots.
__device__ __noinline__ int cl_finish(const float *row, int64_t n, bool maxima, int64_t n_scores, int k,
                         int32_t *outr, bool take_all, int T, int above, int histT, bool fine,
                         int S, int above1, int fineS, int emitted, int ncand, int cap,
                         const unsigned long long *cand, const unsigned long long *cr,
                         unsigned long long *scratch, int *sm_h, int *sm_scan, int *sm_misc,
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
    } else if (ncand > kClRank && ncand <= kClDirect) {
      refine_candidates(cand, ncand, m, outr + base_out, sm_h, sm_misc, sm_u64);
    } else if (ncand <= kClDirect) {
      // candidate keys are unique (the column is part of the key): each
      // thread ranks one against all the others (quadratic: few candidates)
      if (threadIdx.x < ncand) {
        const unsigned long long v = cand[threadIdx.x];
        int rk = 0;
        for (int j = 0; j < ncand; ++j) rk += cand[j] > v;
        if (rk < m) outr[base_out + rk] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
      }
    } else {
      for (int i = threadIdx.x; i < ncand; i += kClThreads)
        scratch[i] = i < kClDirect ? cand[i] : __ldcg(cr + i);
      __syncthreads();
      refine_candidates(scratch, ncand, m, outr + base_out, sm_h, sm_misc, sm_u64);
    }
  } else if (maxima) {
    __syncthreads();
    block_radix_topk([row, n_scores](int64_t b) { return block_max_key(row, n_scores, b); }, n, k,
                     outr, sm_h, sm_scan, sm_misc);
  } else {
    __syncthreads();
    block_radix_topk_row(row, n, k, outr, sm_h, sm_scan, sm_misc);
  }
  return flag;
}

__global__ void __launch_bounds__(kClThreads, 2)
    cluster_select_kernel(const __grid_constant__ ClArgs a) {
  pdl_wait();  // predecessor grids complete before any global access
  extern __shared__ __align__(16) unsigned char cl_raw[];
  ClSmem &sm = *reinterpret_cast<ClSmem *>(cl_raw);
  __shared__ int sm_h[256];
  __shared__ int sm_scan[kSelWarps + 1];
  __shared__ int sm_misc[32];  // [0..2] T, [8..10] S, [16..18] Tb, [24..26] Sb, counters
  __shared__ unsigned long long sm_u64[2];
  const uint32_t rank = cluster_ctarank();
  const int lane = threadIdx.x & 31;
  const int y = blockIdx.y;
  int pi = 0;
  while (pi + 1 < a.nprob && y >= a.cl_begin[pi + 1]) ++pi;
  const ClProb &p = a.p[pi];
  const bool local = p.local != 0;
  const int r = local ? (y - a.cl_begin[pi]) * kCl + (int)rank : y - a.cl_begin[pi];
  if (local && r >= p.R) return;  // a local CTA passes no cluster barrier
  const int k = p.k;
  const int64_t n = row_len(p.ctx, p.next_n, p.len_div, r, p.stride, a.status);
  const float *row = p.logits + (int64_t)r * p.stride;
  int32_t *outr = p.out + (int64_t)r * k;
  const int64_t wr = (int64_t)p.ws_row0 + r;
  unsigned long long *cr = a.cand + wr * DSA_CAND_CAP;
  int32_t *wh = a.ws_hist + wr * DSA_NUM_BINS;
  int32_t *wf = a.ws_fine + wr * kFineBins;
  int32_t *wbh = wf + kClFine;       // the row's block-maxima histogram (workspace)
  int32_t *wbf = wf + 2 * kClFine;   // its fine histogram
  const int32_t *hrow = p.hist ? p.hist + (int64_t)r * DSA_NUM_BINS : nullptr;
  // this CTA's positions [c0, c1), in groups of 2048 (one float4 per thread)
  const int64_t chunk = ((local ? n : (n + kCl - 1) / kCl) + 2047) / 2048 * 2048;
  const int64_t c0 = local ? 0 : (int64_t)rank * chunk;
  const int64_t c1 = min(n, c0 + chunk);
  const int vq = (int)(chunk / 2048);  // <= kClVec
  const bool blk = p.bk > 0;           // block select alongside the score select
  const int bk = p.bk;
  const int dcap = blk ? kClCandHalf : DSA_CAND_CAP;  // candidate slots of the score select
  const int64_t nbk = (n + 7) / 8;     // blocks of the row
  const int64_t b0 = c0 / 8;           // this CTA's first block

  if (threadIdx.x < 8) sm.ctr[threadIdx.x] = 0;
  if (threadIdx.x < 8) sm.bmm[threadIdx.x] = 0;
  for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kClThreads) {
    sm.hist[i] = 0;
    sm.bhist[i] = 0;
  }
  float4 v[kClVec];
  cl_issue_loads(row, c0, c1, vq, p.vec != 0, v);

  // ---- 1. threshold bin T from the caller's histogram, while the row loads
  // (rows of at most k scores take every non-NaN score: T past the last bin)
  const bool take_all = n <= k;
  const bool early = hrow || take_all;  // T known without the row's own histogram
  int T = DSA_NUM_BINS, above = 0, histT = 0;
  if (early && !take_all) {
    threshold_from_hist<DSA_NUM_BINS>(hrow, k, sm_scan, sm_misc);
    T = sm_misc[0];
    above = sm_misc[1];
    histT = sm_misc[2];
  }
  cl_store_keys(v, sm.keys);
  __syncthreads();

  // ---- 2. local histograms: the scores' (when T is not known yet) and the
  // block maxima's (a block of 8 scores is two threads' slots), with the key
  // range each wide bin's maxima take
  if (!early) {
    for (int q = 0; q < vq; ++q) {
      const uint4 k4 = sm.keys[q * kClThreads + threadIdx.x];
      const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (kv[j]) atomicAdd(&sm.hist[coarse_bin_of_key(kv[j])], 1);
    }
  }
  if (blk) {
#pragma unroll 1
    for (int q = 0; q < kClVec; ++q) {
      const uint4 k4 = sm.keys[q * kClThreads + threadIdx.x];
      uint32_t mk = max(max(k4.x, k4.y), max(k4.z, k4.w));
      mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, 1));
      const int lb = q * (kClThreads / 2) + (threadIdx.x >> 1);
      const int b = (int)b0 + lb;           // blocks of a cluster row are below 2^28
      if (q >= vq || b >= (int)nbk) mk = 0;    // slots past this CTA's positions, blocks past the row
      else if (b == (int)nbk - 1) mk = kKeyPosInf;  // the newest block is always chosen
      if ((threadIdx.x & 1) == 0) {
        sm.bkey[lb] = mk;
        if (mk) {
          const int bb = coarse_bin_of_key(mk);
          atomicAdd(&sm.bhist[bb], 1);
          const int wi = wide_bin_idx(bb);
          if (wi >= 0) {
            atomicMax(&sm.bmm[2 * wi], ~mk);
            atomicMax(&sm.bmm[2 * wi + 1], mk);
          }
        }
      }
    }
  }
  uint32_t loT = 0, hiT = 0;  // loT > hiT: bin T empty (T past the last bin)
  bool fine = false, wide = false;
  if (early) {
    bin_key_range(T, loT, hiT);
    fine = (T < DSA_NUM_BINS) && histT > kClDirect;
    wide = fine && (hiT - loT) >= kFineWindow;
    if (wide) cl_range_in(sm.keys, vq, loT, hiT, sm.red);
  }
  __syncthreads();
  if (!local) {
    // publish into the workspace, then the first cluster barrier (it also
    // makes every CTA's counters safe to reach)
    if (!early) cl_flush(sm.hist, wh, DSA_NUM_BINS);
    if (blk) {
      cl_flush(sm.bhist, wbh, DSA_NUM_BINS);
      if (threadIdx.x < 8) wf[kSlotB + 8 * rank + threadIdx.x] = sm.bmm[threadIdx.x];
    }
    if (wide && threadIdx.x == 0) {
      wf[kSlotD + 2 * rank] = sm.red[0];
      wf[kSlotD + 2 * rank + 1] = sm.red[1];
    }
    cluster_arrive();
    cluster_wait();
  }

  // ---- 3. the score select's T when the row built its own histogram
  if (!early) {
    if (!local) {
      cl_fetch(sm.hist, wh, DSA_NUM_BINS);
      __syncthreads();
    }
    threshold_from_hist<DSA_NUM_BINS>(sm.hist, k, sm_scan, sm_misc);
    T = sm_misc[0];
    above = sm_misc[1];
    histT = sm_misc[2];
    bin_key_range(T, loT, hiT);
    fine = (T < DSA_NUM_BINS) && histT > kClDirect;
    wide = fine && (hiT - loT) >= kFineWindow;
    if (wide) {
      cl_range_in(sm.keys, vq, loT, hiT, sm.red);
      if (!local) {
        if (threadIdx.x == 0) {
          wf[kSlotD + 2 * rank] = sm.red[0];
          wf[kSlotD + 2 * rank + 1] = sm.red[1];
        }
        cluster_sync();
      }
    }
  }
  // ---- 4. the block select's threshold Tb and key ranges of wide bins
  const bool btake = nbk <= bk;
  int Tb = DSA_NUM_BINS, aboveb = 0, histTb = 0;
  if (blk) {
    if (!local) {
      cl_fetch(sm.bhist, wbh, DSA_NUM_BINS);
      __syncthreads();
    }
    if (!btake) {
      threshold_from_hist<DSA_NUM_BINS>(sm.bhist, bk, sm_scan, sm_misc + 16);
      Tb = sm_misc[16];
      aboveb = sm_misc[17];
      histTb = sm_misc[18];
    }
  }
  uint32_t bloT, bhiT;
  bin_key_range(Tb, bloT, bhiT);
  const bool bfine = blk && (Tb < DSA_NUM_BINS) && histTb > kClDirect;
  const int bwi = bfine ? wide_bin_idx(Tb) : -1;
  if (threadIdx.x == 0) {
    if (wide && !local) {
      uint32_t nm = 0, mx = 0;
      for (int c = 0; c < kCl; ++c) {
        nm = max(nm, (uint32_t)__ldcg(&wf[kSlotD + 2 * c]));
        mx = max(mx, (uint32_t)__ldcg(&wf[kSlotD + 2 * c + 1]));
      }
      sm.red[0] = nm;
      sm.red[1] = mx;
    }
    if (bwi >= 0) {
      uint32_t nm = sm.bmm[2 * bwi], mx = sm.bmm[2 * bwi + 1];
      if (!local) {
        nm = 0;
        mx = 0;
        for (int c = 0; c < kCl; ++c) {
          nm = max(nm, (uint32_t)__ldcg(&wf[kSlotB + 8 * c + 2 * bwi]));
          mx = max(mx, (uint32_t)__ldcg(&wf[kSlotB + 8 * c + 2 * bwi + 1]));
        }
      }
      sm.red[2] = nm;
      sm.red[3] = mx;
    }
  }
  __syncthreads();

  // ---- 5. fine histograms of bin T and bin Tb (one barrier for both)
  uint32_t flo = 0, bflo = 0;
  int fshift = 0, S = 0, above1 = 0, fineS = 0;
  int bfs = 0, Sb = 0, above1b = 0, fineSb = 0;
  if (fine || bfine) {
    if (fine) {
      cl_fine_window(T, loT, hiT, wide ? ~sm.red[0] : 0u, wide ? sm.red[1] : 0u, flo, fshift);
      for (int i = threadIdx.x; i < kClFine; i += kClThreads) sm.hist[i] = 0;
    }
    if (bfine) {
      cl_fine_window(Tb, bloT, bhiT, bwi >= 0 ? ~sm.red[2] : 0u, bwi >= 0 ? sm.red[3] : 0u, bflo,
                     bfs);
      for (int i = threadIdx.x; i < kClFine; i += kClThreads) sm.bhist[i] = 0;
    }
    __syncthreads();
    if (fine) {
      for (int q = 0; q < vq; ++q) {
        const uint4 k4 = sm.keys[q * kClThreads + threadIdx.x];
        const uint32_t kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (kv[j] >= loT && kv[j] <= hiT)
            atomicAdd(&sm.hist[cl_fine_idx(kv[j], flo, fshift)], 1);
      }
    }
    if (bfine) {
      for (int i = threadIdx.x; i < kClBlk; i += kClThreads) {
        const uint32_t mk = sm.bkey[i];
        if (mk >= bloT && mk <= bhiT) atomicAdd(&sm.bhist[cl_fine_idx(mk, bflo, bfs)], 1);
      }
    }
    __syncthreads();
    if (!local) {
      if (fine) cl_flush(sm.hist, wf, kClFine);
      if (bfine) cl_flush(sm.bhist, wbf, kClFine);
      cluster_sync();
      if (fine) cl_fetch(sm.hist, wf, kClFine);
      if (bfine) cl_fetch(sm.bhist, wbf, kClFine);
      __syncthreads();
    }
    if (fine) {
      threshold_from_hist<kClFine>(sm.hist, k - above, sm_scan, sm_misc + 8);
      S = sm_misc[8];
      above1 = sm_misc[9];
      fineS = sm_misc[10];
    }
    if (bfine) {
      threshold_from_hist<kClFine>(sm.bhist, bk - aboveb, sm_scan, sm_misc + 24);
      Sb = sm_misc[24];
      above1b = sm_misc[25];
      fineSb = sm_misc[26];
    }
  }

  // ---- 6. classify both selects, reserve output and candidate ranges
  // (score select on CTA 0, block select on CTA 1), write.  Emit: key > E;
  // candidate: C <= key <= E (bin T, or its fine bin S)
  uint32_t C = loT, E = hiT, CB = bloT, EB = bhiT;
  if (fine) fine_bin_keys(loT, hiT, flo, fshift, S, C, E);
  if (bfine) fine_bin_keys(bloT, bhiT, bflo, bfs, Sb, CB, EB);
  const unsigned long long kinds = cl_classify(sm.keys, vq, C, E);
  const int ne = __popcll(kinds & 0x5555555555555555ull);
  const int nc = __popcll(kinds & 0xAAAAAAAAAAAAAAAAull);
  constexpr int kBPer = kClBlk / kClThreads;  // maxima per thread: index tid + e * kClThreads
  uint32_t bkinds = 0;
  if (blk) {
#pragma unroll
    for (int e = 0; e < kBPer; ++e)
      bkinds |= cl_kind(sm.bkey[threadIdx.x + e * kClThreads], CB, EB) << (2 * e);
  }
  const int bne = __popc(bkinds & 0x55u), bnc = __popc(bkinds & 0xAAu);
  int tot, btot = 0, bex = 0;
  const int ex = block_excl_scan((nc << 16) | ne, sm_scan, &tot);  // per CTA < 2^15 each
  if (blk) bex = block_excl_scan((bnc << 16) | bne, sm_scan, &btot);
  int base_e = 0, base_c = 0, bbe = 0, bbc = 0;
  uint32_t cand0 = 0, bcand1 = 0;
  if (!local) {
    const uint32_t ctr0 = dsmem_map(smem_u32(&sm.ctr[0]), 0);
    const uint32_t bctr = dsmem_map(smem_u32(&sm.ctr[4]), 1);
    if (threadIdx.x == 0) {
      const int e0 = (tot & 0xFFFF) ? dsmem_atomic_add(ctr0, tot & 0xFFFF) : 0;
      const int e1 = (tot >> 16) ? dsmem_atomic_add(ctr0 + 4, tot >> 16) : 0;
      const int e2 = (btot & 0xFFFF) ? dsmem_atomic_add(bctr, btot & 0xFFFF) : 0;
      const int e3 = (btot >> 16) ? dsmem_atomic_add(bctr + 4, btot >> 16) : 0;
      sm_misc[5] = e0;
      sm_misc[6] = e1;
      sm_misc[21] = e2;
      sm_misc[22] = e3;
    }
    __syncthreads();
    base_e = sm_misc[5];
    base_c = sm_misc[6];
    bbe = sm_misc[21];
    bbc = sm_misc[22];
    cand0 = dsmem_map(smem_u32(&sm.cand[0]), 0);
    bcand1 = dsmem_map(smem_u32(&sm.bcand[0]), 1);
  }
  if (kinds)
    cl_write(kinds, sm.keys, c0, base_e + (ex & 0xFFFF), base_c + (ex >> 16), k, dcap, outr,
             !local, cand0, sm.cand, cr);
  int32_t *boutr = blk ? p.bout + (int64_t)r * bk : nullptr;
  unsigned long long *crb = cr + kClCandHalf;
  if (bkinds) {
    int pe = bbe + (bex & 0xFFFF), pc = bbc + (bex >> 16);
#pragma unroll
    for (int e = 0; e < kBPer; ++e) {
      const uint32_t kd = (bkinds >> (2 * e)) & 3u;
      if (!kd) continue;
      const int idx = threadIdx.x + e * kClThreads;
      const int64_t b = b0 + idx;
      if (kd == 1) {
        if (pe < bk) boutr[pe] = (int32_t)b;
        ++pe;
      } else {
        const unsigned long long cv = ((unsigned long long)sm.bkey[idx] << 32) |
                                      (unsigned long long)(0xFFFFFFFFu - (uint32_t)b);
        if (pc < kClDirect) {
          if (!local) dsmem_st64(bcand1 + 8u * (uint32_t)pc, cv);
          else sm.bcand[pc] = cv;
        } else if (pc < kClCandHalf) {
          crb[pc] = cv;
        }
        ++pc;
      }
    }
  }
  if (!local) cluster_sync();  // all emits and candidates are in place; histograms read
  else __syncthreads();

  // ---- 7. check, rank or refine, or fall back: the score select on CTA 0
  // (the local CTA), the block select on CTA 1 (the local CTA, after)
  unsigned long long *scratch = reinterpret_cast<unsigned long long *>(sm.keys);
  if (local || rank == 0) {
    const int emitted = local ? (tot & 0xFFFF) : sm.ctr[0];
    const int ncand = local ? (tot >> 16) : sm.ctr[1];
    const int flag = cl_finish(row, n, false, n, k, outr, take_all, T, above, histT, fine, S,
                               above1, fineS, emitted, ncand, dcap, sm.cand, cr, scratch, sm_h,
                               sm_scan, sm_misc, sm_u64);
    if (p.flags && threadIdx.x == 0) p.flags[r] = flag;
    // restore the zero workspace histograms; clear the caller's on request
    if (!local) {
      if (!early)
        for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kClThreads) wh[i] = 0;
      if (fine)
        for (int i = threadIdx.x; i < kClFine; i += kClThreads) wf[i] = 0;
      if (wide && threadIdx.x < 2 * kCl) wf[kSlotD + threadIdx.x] = 0;
    }
    if (p.reset_hist && p.hist) {
      int32_t *hw = p.hist + (int64_t)r * DSA_NUM_BINS;
      for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kClThreads) hw[i] = 0;
    }
  }
  if (blk && (local || rank == 1)) {
    __syncthreads();  // the local CTA: the score select's finish is done with the scratch
    const int emitted = local ? (btot & 0xFFFF) : sm.ctr[4];
    const int ncand = local ? (btot >> 16) : sm.ctr[5];
    const int flag = cl_finish(row, nbk, true, n, bk, boutr, btake, Tb, aboveb, histTb, bfine, Sb,
                               above1b, fineSb, emitted, ncand, kClCandHalf, sm.bcand, crb,
                               scratch, sm_h, sm_scan, sm_misc, sm_u64);
    if (p.bflags && threadIdx.x == 0) p.bflags[r] = flag;
    if (!local) {
      for (int i = threadIdx.x; i < DSA_NUM_BINS; i += kClThreads) wbh[i] = 0;
      if (bfine)
        for (int i = threadIdx.x; i < kClFine; i += kClThreads) wbf[i] = 0;
      if (threadIdx.x < 8 * kCl) wf[kSlotB + threadIdx.x] = 0;
    }
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
  const int lane = threadIdx.x & 31;
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
constexpr int kF16MaxRow = 16384;

template <bool BF16>
__global__ void __launch_bounds__(kSelThreads)
    topk_fp16_kernel(const uint16_t *scores, int64_t stride, const int32_t *valid_lens, int k,
                     const int32_t *table, int kb, int32_t *out, uint32_t *status) {
  pdl_wait();  // predecessor grids complete before any global access
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
  // keys, with positions >= n masked to the invalid key 0 (all loads issued
  // first); coarse histogram
  // words are handled in rounds of 4 per thread (all 4 loads in flight);
  // the round count depends only on the row, so every lane runs it
  constexpr int WR = 4;
  const int rounds = (nw + WR * kSelThreads - 1) / (WR * kSelThreads);
  for (int rd = 0; rd < rounds; ++rd) {
    uint32_t wv[WR];
#pragma unroll
    for (int e = 0; e < WR; ++e) {
      const int w = (rd * WR + e) * kSelThreads + threadIdx.x;
      wv[e] = (w < nw) ? row[w] : 0u;
    }
#pragma unroll
    for (int e = 0; e < WR; ++e) {
      const int w = (rd * WR + e) * kSelThreads + threadIdx.x;
      uint32_t kk = (w < nw) ? (BF16 ? bf16x2_order_keys(wv[e]) : f16x2_order_keys(wv[e])) : 0u;
      if (2 * w + 1 >= n) kk &= 0x0000FFFFu;
      keys2[w] = kk;
      const uint32_t lo = kk & 0xFFFFu, hi = kk >> 16;
      if (lo) atomicAdd(&h[lo >> 6], 1);
      if (hi) atomicAdd(&h[hi >> 6], 1);
    }
  }
  const int nw_r = rounds * WR * kSelThreads;  // words written above (zero past the row)
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
    for (int w0 = 0; w0 < nw_r; w0 += kSelThreads) {
      const uint32_t kk = keys2[w0 + threadIdx.x];  // 0 past the row
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
    p.local = c.stride <= kClChunk ? 1 : 0;
    p.vec = ((reinterpret_cast<uintptr_t>(c.logits) & 15) == 0 && c.stride % 4 == 0) ? 1 : 0;
    ca.cl_begin[i] = (int)clusters;
    clusters += p.local ? (c.R + kCl - 1) / kCl : c.R;
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
  return launch_pdl(c.bf16 ? topk_fp16_kernel<true> : topk_fp16_kernel<false>, dim3(c.R),
                    dim3(kSelThreads), 0, st, c.scores, c.stride,
                    c.valid_lens, c.k, c.block_table, c.kb, c.out_idx, c.status);
}

}  // namespace dsa
