// logits.cu -- paged MQA logits on sm_103a tensor cores, with the coarse
// score histogram fused into the epilogue, and the sparse variant that scores
// only the blocks of a candidate block table.
//
// [DG94] DeepGEMM PR #94 "What this adds": logits[r,t] = sum_h w[r,h] *
// ReLU(q[r,h].k[t] * kscale[t]) over an FP8 paged K cache, H = 32, D = 128,
// every live non-NaN score binned into 1024 descending bins while it is still
// in registers; verify rows (next_n > 1) share one K pass of their request
// (token Q tile, UMMA_N = 32 * next_n).
// [SG38944] SGLang PR #38944 "What this enables": the sparse logits score only
// the published 8-token blocks.
//
// One persistent CTA per SM over a ring of 256-token stages (32 KiB of K,
// 1 KiB of kscale each); 10 warps at next_n = 1, 18 at next_n > 1, one more
// in the sparse pass:
//   warp 0      producer: gathers the stage's K pages (or 8-token blocks)
//               through the page table with one multi-lane TMA instruction,
//               the matching kscale with one multi-lane bulk copy (sparse:
//               16-byte cp.async), and each request's Q tile and head weights
//               into one of two buffers; page-table entries are read one
//               group of stages ahead.  In the sparse pass a second producer
//               warp (the last one) issues half of each stage's block gathers.
//   warp 1      allocates TMEM and issues tcgen05.mma (one thread): per stage
//               two sub-tiles D[128 tokens x 32*next_n] = K[128 x 128] .
//               Q[32*next_n x 128]^T, FP8 x FP8 -> FP32, into a TMEM pair
//   warps 2..   epilogue, one warpgroup per 128-token sub-tile (two per
//               sub-tile at next_n > 1, taking alternate stages): each
//               thread owns one TMEM lane = one token, loads its 32 head dots
//               per row, applies kscale, ReLU and the head weights in
//               registers, stores the logit (coalesced across the warp) and
//               counts its bin in a shared histogram slot; the slots are
//               flushed with packed 64-bit global atomics whenever the CTA
//               moves on to another request.
// Work split: the flattened (request, stage) sequence is cut into gridDim.x
// contiguous ranges, one per CTA; each CTA derives its range from a prefix sum
// over context_lens (no separate metadata kernel).  Ring positions advance
// by counters (no division per stage).
#include <algorithm>

#include <type_traits>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {

namespace {

constexpr int kStageTok = 256;               // tokens per pipeline stage
constexpr int kSubTok = 128;                 // tokens per MMA sub-tile (TMEM lanes)
constexpr int kStageK = kStageTok * 128;     // bytes of K per stage
constexpr int kSubK = kSubTok * 128;
constexpr int kStageKs = kStageTok * 4;      // bytes of kscale per stage
constexpr int kMaxStages = 8;
// Epilogue warps: two warpgroups (one per 128-token sub-tile) at next_n = 1;
// four at next_n > 1, where the epilogue carries next_n rows per token: the
// two groups of a sub-tile take alternate stages.  Eight warps consume each
// stage either way.
__host__ __device__ constexpr int epi_warps(int nn) { return nn == 1 ? 8 : 16; }
// One more warp after the epilogue warps: a second producer (the sparse
// pass; dense FP8 keys at next_n = 1) or, with MXFP4 keys, the scale-factor
// warp.
__host__ __device__ constexpr int threads_for(int nn, bool sparse, bool mx = false) {
  return 64 + 32 * epi_warps(nn) + ((sparse || mx || nn == 1) ? 32 : 0);
}
constexpr int kStageEpiWarps = 8;
constexpr int kSmemLimit = 232448;           // 227 KiB opt-in per CTA

struct LogitsArgs {
  const int32_t *context_lens;
  const int32_t *page_table;
  int64_t pt_stride;
  const float *kscale;
  const float *weights;
  int32_t B;
  int32_t req_next_n;   // rows per request
  int32_t page_size;
  int32_t log2_ps;      // page_size is 64 or 128
  int32_t num_pages;
  int32_t num_units;    // dense: requests; sparse: rows
  int32_t sparse_tpu;   // sparse: stages per row (ceil(kb / 32))
  const int32_t *block_table;
  int32_t kb;
  const int32_t *phys;        // sparse: physical blocks (pool slot / 8) of the table, or NULL
  const int32_t *valid_lens;  // sparse, with phys: live positions form the prefix [0, len)
  // sparse, paired rows (next_n = 2 instantiation): unit u is rows 2m, 2m+1
  // of request u / upr (an odd last row alone); `phys` is then the union of
  // their tables, `upos` per union entry (pos_a + 1) | (pos_b + 1) << 16
  const int32_t *upos;
  const int32_t *ulen;        // union entries per unit, or NULL (unpaired)
  int32_t upr;                // units per request: ceil(next_n / 2)
  int32_t tab_stride;         // entries per unit in `phys`: kb, or 2 kb paired
  // unpaired, kb a multiple of 32, `phys` 16-byte aligned: the entries of
  // flattened stage g are phys[32 g .. 32 g + 31], read by 16-byte loads
  int32_t phys_vec;
  void *out;
  int64_t out_stride;
  int32_t *histogram;
  float *amax;          // dense only: block maxima over 8 scores, or NULL
  int64_t amax_stride;
  int32_t amax_skip;    // rows with at most this many blocks are skipped (0: none)
  uint32_t *status;
  int32_t num_stages;
  int32_t num_acc;
  int32_t num_ks;       // kscale ring depth
  uint32_t tmem_cols;
  long long wait_limit;
};

struct SmemPlan {
  int kst, q, ks, w, hist, bar, misc, sptab, sfst, total;
};

constexpr int kSpTab = 32;  // sparse: stages whose K rows the producer holds in shared memory

// Histogram slots per epilogue warpgroup: one per warp at next_n = 1, one
// shared by the group's four warps otherwise (shared memory goes to stages).
// A slot holds 16-bit counts, two bins to a 32-bit word (bin 2p in the low
// half of word p), and is flushed on every change of request and at least
// every kHistFlushStages stages, so no count reaches 2^16: a slot counts at
// most 128 tokens a stage.
__host__ __device__ constexpr int hist_slots_per_group(int nn) { return nn == 1 ? 4 : 1; }
constexpr int kHistWords = DSA_NUM_BINS / 2;  // 32-bit words of one slot row
constexpr int kHistFlushStages = 256;

// MXFP4 keys: per K stage, the block exponents of its two sub-tiles as the
// 32-row x 16-byte tables the scale-factor copy into TMEM reads (2 x 512 B).
constexpr int kSfStage = 1024;

__host__ __device__ inline SmemPlan smem_plan(int nn, bool hist, bool sparse, int stages, int nacc,
                                              int nks, bool mx = false) {
  SmemPlan p;
  int off = 0;
  p.kst = off;
  off += stages * kStageK;
  p.q = off;
  off += 2 * nn * 32 * 128;
  p.ks = off;
  off += nks * kStageKs;
  p.w = off;
  off += 2 * nn * 32 * 4;
  p.hist = off;
  off += hist ? 2 * hist_slots_per_group(nn) * nn * kHistWords * 4 : 0;
  off = (off + 7) & ~7;
  p.bar = off;
  off += (2 * stages + 2 * nks + 4 + 2 * nacc + 3 + (mx ? stages : 0)) * 8;
  p.misc = off;
  off += 64 + 2 * 32 * 4;  // flags/schedule + the producer's two row tables
  off = (off + 15) & ~15;  // 16-byte stores into the sparse row table
  p.sptab = off;
  off += sparse ? kSpTab * 32 * 4 : 0;
  off = (off + 127) & ~127;
  p.sfst = off;
  off += mx ? stages * kSfStage : 0;
  p.total = off + 1024;  // slack to align the base to 1024 bytes
  return p;
}

__device__ __forceinline__ int64_t eff_ctx(const LogitsArgs &a, int b) {
  int64_t c = __ldg(&a.context_lens[b]);
  const int64_t cap = a.pt_stride * a.page_size;
  if (c < 0) c = 0;
  if (c > cap) c = cap;
  return c;
}

// Pool row of physical block `raw` (pool slot / 8), or -1 for padding; an id
// past the pool is flagged and skipped.
__device__ __forceinline__ int phys_block_row(const LogitsArgs &a, int raw) {
  if (raw == INT32_MAX || raw < 0) return -1;
  if ((int64_t)raw * 8 + 8 > (int64_t)a.num_pages * a.page_size) {
    set_status(a.status, DSA_DEV_BOUNDS);
    return -1;
  }
  return raw * 8;
}

template <bool SPARSE>
__device__ __forceinline__ int unit_tiles(const LogitsArgs &a, int u) {
  if (SPARSE) {
    if (!a.ulen) return a.sparse_tpu;
    // paired: the union, and at least kb entries so that every padding
    // position of both rows' outputs is visited once
    const int n = min(max(__ldg(&a.ulen[u]), a.kb), a.tab_stride);
    return (n + 31) / 32;
  }
  return static_cast<int>((eff_ctx(a, u) + kStageTok - 1) / kStageTok);
}

template <bool SPARSE>
struct TileIter {
  int u, i, tiles;
  __device__ void init(const LogitsArgs &a, int u0, int i0) {
    u = u0;
    i = i0;
    tiles = (u < a.num_units) ? unit_tiles<SPARSE>(a, u) : 1;
  }
  __device__ void next(const LogitsArgs &a) {
    if (++i >= tiles) {
      i = 0;
      do {
        ++u;
        tiles = (u < a.num_units) ? unit_tiles<SPARSE>(a, u) : 1;
      } while (tiles == 0);
    }
  }
};

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Position in a ring of `size` slots with the mbarrier phase bit of the
// current lap: advanced by one per tile (no division in the loops).
struct Ring {
  int idx;
  uint32_t ph;
  int size;
  __device__ __forceinline__ void init(int n) {
    idx = 0;
    ph = 0;
    size = n;
  }
  __device__ __forceinline__ void next() {
    if (++idx == size) {
      idx = 0;
      ph ^= 1;
    }
  }
  // slot and phase of the tile `back` positions before the current one (back <= size)
  __device__ __forceinline__ void prev(int back, int &i, uint32_t &p) const {
    i = idx - back;
    p = ph;
    if (i < 0) {
      i += size;
      p ^= 1;
    }
  }
};

// One warp: this CTA's contiguous range [g0, g1) of the flattened tile
// sequence, as (first unit, first tile in it, tile count).
template <bool SPARSE>
__device__ void compute_sched(const LogitsArgs &a, int *out_u0, int *out_i0, long long *out_cnt) {
  const int lane = threadIdx.x & 31;
  long long T = 0;
  const bool fixed = SPARSE && !a.ulen;  // same stage count for every unit
  if (fixed) {
    T = (long long)a.num_units * a.sparse_tpu;
  } else {
    for (int base = 0; base < a.num_units; base += 32) {
      const int b = base + lane;
      int t = (b < a.num_units) ? unit_tiles<SPARSE>(a, b) : 0;
      if (!SPARSE && b < a.num_units && a.context_lens[b] > a.pt_stride * a.page_size)
        set_status(a.status, DSA_DEV_BOUNDS);
      T += __shfl_sync(0xffffffffu, warp_incl_scan(t), 31);
    }
  }
  // (32-bit divisions when the products fit: a 64-bit one is a long
  // software sequence on the start of every CTA)
  long long g0, g1;
  if (T * gridDim.x < (1ll << 31)) {
    g0 = (int)(blockIdx.x * (unsigned)T) / (int)gridDim.x;
    g1 = (int)((blockIdx.x + 1) * (unsigned)T) / (int)gridDim.x;
  } else {
    g0 = (long long)blockIdx.x * T / gridDim.x;
    g1 = (long long)(blockIdx.x + 1) * T / gridDim.x;
  }
  int u0 = a.num_units, i0 = 0;
  if (g1 > g0) {
    if (fixed) {
      u0 = g0 < (1ll << 31) ? (int)g0 / a.sparse_tpu : (int)(g0 / a.sparse_tpu);
      i0 = (int)(g0 - (long long)u0 * a.sparse_tpu);
    } else {
      long long acc = 0;
      for (int base = 0; base < a.num_units; base += 32) {
        const int b = base + lane;
        const int t = (b < a.num_units) ? unit_tiles<SPARSE>(a, b) : 0;
        const int incl = warp_incl_scan(t);
        const int tot = __shfl_sync(0xffffffffu, incl, 31);
        if (g0 < acc + tot) {
          const unsigned m = __ballot_sync(0xffffffffu, acc + incl > g0);
          const int l = __ffs(m) - 1;
          const int excl_l = __shfl_sync(0xffffffffu, incl - t, l);
          u0 = base + l;
          i0 = (int)(g0 - acc - excl_l);
          break;
        }
        acc += tot;
      }
    }
  }
  *out_u0 = u0;
  *out_i0 = i0;
  *out_cnt = g1 - g0;
}

// Packed FP32 pairs (sm_100 family): two lanes of arithmetic per instruction.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Sum over the 32 heads of one row: kscale, ReLU, head weight.  Four
// independent accumulation chains (heads h = 4i + c go to chain c), combined
// as (c0 + c1) + (c2 + c3).  For a finite kscale s >= 0, ReLU(d * s) = s *
// ReLU(d), so s is applied once to the sum; any other s takes the formula
// term by term.  Dense and sparse logits share this function, so they are
// bitwise equal.  The head weights come in registers (the row's 32, read
// once per request).
__device__ __forceinline__ float head_sum(const uint32_t (&v)[32], float ks, const float (&w)[32]) {
  uint64_t a01 = pk2(0.0f, 0.0f), a23 = pk2(0.0f, 0.0f);
  if (ks >= 0.0f && ks <= 3.4028234e38f) {
#pragma unroll
    for (int h = 0; h < 32; h += 4) {
      a01 = fma2(pk2(w[h + 0], w[h + 1]),
                 pk2(fmaxf(__uint_as_float(v[h + 0]), 0.0f), fmaxf(__uint_as_float(v[h + 1]), 0.0f)),
                 a01);
      a23 = fma2(pk2(w[h + 2], w[h + 3]),
                 pk2(fmaxf(__uint_as_float(v[h + 2]), 0.0f), fmaxf(__uint_as_float(v[h + 3]), 0.0f)),
                 a23);
    }
    float c0, c1, c2, c3;
    upk2(a01, c0, c1);
    upk2(a23, c2, c3);
    return ks * ((c0 + c1) + (c2 + c3));
  }
  const uint64_t ks2 = pk2(ks, ks);
#pragma unroll
  for (int h = 0; h < 32; h += 4) {
    float p0, p1, p2, p3;
    upk2(mul2(pk2(__uint_as_float(v[h + 0]), __uint_as_float(v[h + 1])), ks2), p0, p1);
    upk2(mul2(pk2(__uint_as_float(v[h + 2]), __uint_as_float(v[h + 3])), ks2), p2, p3);
    a01 = fma2(pk2(w[h + 0], w[h + 1]), pk2(fmaxf(p0, 0.0f), fmaxf(p1, 0.0f)), a01);
    a23 = fma2(pk2(w[h + 2], w[h + 3]), pk2(fmaxf(p2, 0.0f), fmaxf(p3, 0.0f)), a23);
  }
  float c0, c1, c2, c3;
  upk2(a01, c0, c1);
  upk2(a23, c2, c3);
  return (c0 + c1) + (c2 + c3);
}

// MX: the keys are MXFP4 (E2M1 codes through a 4-bit unpacking tensor map,
// one UE8M0 exponent per 32 dimensions in place of kscale), multiplied by
// the block-scaled MMA; dense logits only.
// head_sum in two calls of 16 heads each (heads 16p .. 16p+15 for p = 0, 1,
// in that order): the same chains in the same order, so the same float.
// ALLOK (chosen per warp by the caller): every lane's kscale is finite and
// >= 0, so the sum is taken without it and the caller applies it.  Otherwise
// each lane takes its own case by selects, not branches (the warp's TMEM
// loads around this call need it converged): a lane whose kscale qualifies
// (`ksok`) still sums without it, the others apply it term by term.
template <bool ALLOK>
__device__ __forceinline__ void head_sum_part(const uint32_t (&v)[16], float ks, bool ksok,
                                              const float *w, uint64_t &a01, uint64_t &a23) {
  if (ALLOK) {
#pragma unroll
    for (int h = 0; h < 16; h += 4) {
      const float4 wv = *reinterpret_cast<const float4 *>(w + h);
      a01 = fma2(pk2(wv.x, wv.y),
                 pk2(fmaxf(__uint_as_float(v[h + 0]), 0.0f), fmaxf(__uint_as_float(v[h + 1]), 0.0f)),
                 a01);
      a23 = fma2(pk2(wv.z, wv.w),
                 pk2(fmaxf(__uint_as_float(v[h + 2]), 0.0f), fmaxf(__uint_as_float(v[h + 3]), 0.0f)),
                 a23);
    }
    return;
  }
  const uint64_t ks2 = pk2(ks, ks);
#pragma unroll
  for (int h = 0; h < 16; h += 4) {
    const float4 wv = *reinterpret_cast<const float4 *>(w + h);
    float p0, p1, p2, p3;
    upk2(mul2(pk2(__uint_as_float(v[h + 0]), __uint_as_float(v[h + 1])), ks2), p0, p1);
    upk2(mul2(pk2(__uint_as_float(v[h + 2]), __uint_as_float(v[h + 3])), ks2), p2, p3);
    p0 = ksok ? __uint_as_float(v[h + 0]) : p0;
    p1 = ksok ? __uint_as_float(v[h + 1]) : p1;
    p2 = ksok ? __uint_as_float(v[h + 2]) : p2;
    p3 = ksok ? __uint_as_float(v[h + 3]) : p3;
    a01 = fma2(pk2(wv.x, wv.y), pk2(fmaxf(p0, 0.0f), fmaxf(p1, 0.0f)), a01);
    a23 = fma2(pk2(wv.z, wv.w), pk2(fmaxf(p2, 0.0f), fmaxf(p3, 0.0f)), a23);
  }
}

template <int NN, bool SPARSE, int OUT, bool HIST, bool MX = false>
__global__ void __launch_bounds__(threads_for(NN, SPARSE, MX), 1)
    logits_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                  const LogitsArgs a) {
  static_assert(!(MX && SPARSE), "MXFP4 keys: dense logits only");
  // the dense pass waits for its predecessors at once; the sparse pass sets up
  // (barriers, schedule, TMEM, tensor maps: nothing a predecessor writes) first
  // dense, and paired sparse (whose schedule reads the union lengths): the
  // predecessor's outputs are needed from the start
  constexpr bool kWaitFirst = !SPARSE || NN > 1;
  if (kWaitFirst) pdl_wait();
  constexpr int N = 32 * NN;
  constexpr uint32_t IDESC = idesc_e4m3_f32(128, N);
  constexpr int HS = hist_slots_per_group(NN);
  constexpr int EW = epi_warps(NN);
  constexpr int NPAR = EW / kStageEpiWarps;  // groups sharing a sub-tile (alternate stages)
  constexpr int kThr = threads_for(NN, SPARSE, MX);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

  const int S = a.num_stages;
  const int A = a.num_acc;
  const int KS = a.num_ks;
  const SmemPlan P = smem_plan(NN, HIST, SPARSE, S, A, KS, MX);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t kst = smem_u32(smem + P.kst);
  const uint32_t qst = smem_u32(smem + P.q);
  float *ks_s = reinterpret_cast<float *>(smem + P.ks);
  float *w_s = reinterpret_cast<float *>(smem + P.w);
  uint32_t *hist_s = reinterpret_cast<uint32_t *>(smem + P.hist);
  const uint32_t bar0 = smem_u32(smem + P.bar);
  // barrier map
  auto FULL = [&](int s) { return bar0 + 8u * s; };                       // K landed
  auto EMPTY = [&](int s) { return bar0 + 8u * (S + s); };                // MMA done with K
  auto KSF = [&](int k) { return bar0 + 8u * (2 * S + k); };              // kscale landed
  auto KSE = [&](int k) { return bar0 + 8u * (2 * S + KS + k); };         // epilogue done
  const uint32_t qb0 = bar0 + 8u * (2 * S + 2 * KS);
  auto QFULL = [&](int q) { return qb0 + 8u * q; };
  auto QEMPTY = [&](int q) { return qb0 + 8u * (2 + q); };
  auto AFULL = [&](int x) { return qb0 + 8u * (4 + x); };
  auto AEMPTY = [&](int x) { return qb0 + 8u * (4 + A + x); };
  const uint32_t DRAIN = qb0 + 8u * (4 + 2 * A);
  auto GSYNC = [&](int g) { return qb0 + 8u * (5 + 2 * A + g); };
  auto SFR = [&](int s) { return qb0 + 8u * (7 + 2 * A + s); };  // MX: scale factors staged
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + P.misc);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + P.misc + 4);
  int *sched = reinterpret_cast<int *>(smem + P.misc + 16);
  long long *sched_cnt = reinterpret_cast<long long *>(smem + P.misc + 32);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), 1);
    }
    for (int k = 0; k < KS; ++k) {
      mbar_init(KSF(k), SPARSE ? 32 : 1);  // sparse: one cp.async arrival per producer lane
      mbar_init(KSE(k), MX ? 1 : kStageEpiWarps);  // MX: the scale-factor warp reads the exponents
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(QFULL(q), 1);
      mbar_init(QEMPTY(q), 1 + EW);
    }
    for (int x = 0; x < A; ++x) {
      mbar_init(AFULL(x), 1);
      mbar_init(AEMPTY(x), kStageEpiWarps);
    }
    mbar_init(DRAIN, 1);
    if (MX)
      for (int s = 0; s < S; ++s) mbar_init(SFR(s), 1);
    mbar_init(GSYNC(0), 4 * NPAR);
    mbar_init(GSYNC(1), 4 * NPAR);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) compute_sched<SPARSE>(a, &sched[0], &sched[1], sched_cnt);
  if (HIST) {
    for (int i = threadIdx.x; i < 2 * HS * NN * kHistWords; i += kThr) hist_s[i] = 0;
  }
  __syncthreads();
  const long long count = *sched_cnt;
  if (count <= 0) return;  // uniform across the CTA: nothing to do, no TMEM taken
  const int u_start = sched[0], i_start = sched[1];

  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), a.tmem_cols);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_q);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!kWaitFirst) pdl_wait();  // the block table, physical blocks and live lengths are ready
  const uint32_t tmem_base = *tmem_slot;
  // MX TMEM beyond the accumulators: the A scale factors of the two
  // sub-tiles (4 columns each, rewritten every stage in issue order with the
  // MMAs), then the B scale factors, all 2^0 (UE8M0 127): queries are plain E4M3
  const uint32_t sfa0 = tmem_base + 2u * (uint32_t)A * (uint32_t)N;
  const uint32_t sfb = sfa0 + 64u;
  if (MX) {
    if (warp >= 2 && warp < 6) {  // one warp per TMEM lane quarter
      const uint32_t lq = (uint32_t)(32 * (warp & 3)) << 16;
      tmem_st4(sfb + lq, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st4(sfb + lq + 4u, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      tmem_st_wait();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  const WaitCtl ctl{abort_flag, a.status, a.wait_limit};

  // FP8 dense keys at next_n = 1 in pages of 64 tokens (four page copies a
  // stage): two producer warps take alternate stages, warp 0 also loading Q
  // and the weights.  One warp issuing every stage's copies caps the gather
  // below what the memory delivers (measured: two warps gather random 8 KiB
  // pages about 8 % faster).  With pages of 128 tokens (two copies a stage)
  // or next_n > 1 (the epilogue bounds the pass) one producer does it all.
  constexpr bool kTwoProd = !SPARSE && !MX && NN == 1;
  const int nprod = (kTwoProd && a.page_size == 64) ? 2 : 1;
  if (warp == 0 || (kTwoProd && warp == 2 + EW)) {
    // ------------------------------------------------------------ producer
    // (the second producer warp is idle when one producer does it all)
    const int role = warp == 0 ? 0 : 1;
    const bool idle = role == 1 && nprod == 1;
    auto mine = [&](long long m) { return nprod == 1 || (int)(m & 1) == role; };
    // ppt load slots per stage (4 or 2 pages, or 32 blocks of 8 tokens), one
    // per lane; tpg = 32 / ppt stages per prefetch group.  Each lane reads its
    // slot's table entry one group ahead of use.
    const int ppt = SPARSE ? 32 : (kStageTok / a.page_size);
    const int tpg = 32 / ppt;
    const int my_o = lane / ppt, my_sl = lane % ppt;
    constexpr int kNone = INT32_MIN;
    TileIter<SPARSE> it;
    it.init(a, u_start, i_start);
    TileIter<SPARSE> git = it;  // first stage of the group being prefetched
    // raw table entry of this lane's slot in the group starting at (g0, n0)
    auto fetch = [&](TileIter<SPARSE> g0, long long n0, int &unit) -> int {
      unit = -1;
      if (n0 + my_o >= count) return kNone;
      for (int k = 0; k < my_o; ++k) g0.next(a);
      unit = g0.u;
      if (SPARSE) {
        const int blk = g0.i * 32 + my_sl;
        if (blk >= a.tab_stride) return kNone;
        return __ldg(&(a.phys ? a.phys : a.block_table)[(int64_t)g0.u * a.tab_stride + blk]);
      }
      const int64_t p = (int64_t)g0.i * ppt + my_sl;
      if (p * a.page_size >= eff_ctx(a, g0.u)) return kNone;
      return __ldg(&a.page_table[(int64_t)g0.u * a.pt_stride + p]);
    };
    // physical row of a slot (or -1 when nothing is loaded)
    auto to_row = [&](int raw, int unit) -> int {
      if (raw == kNone || unit < 0) return -1;
      if (SPARSE && a.phys) return phys_block_row(a, raw);  // no page-table read
      if (SPARSE) {
        const int b = unit / a.req_next_n;
        const int j = unit - b * a.req_next_n;
        const int64_t n_live = eff_ctx(a, b) - (a.req_next_n - 1 - j);
        if (raw == INT32_MAX || raw < 0 || (int64_t)raw * 8 >= n_live) return -1;
        const int64_t tok = (int64_t)raw * 8;
        int32_t pg = __ldg(&a.page_table[(int64_t)b * a.pt_stride + (tok >> a.log2_ps)]);
        if (pg < 0 || pg >= a.num_pages) {
          set_status(a.status, DSA_DEV_BOUNDS);
          pg = 0;
        }
        return pg * a.page_size + (int)(tok & (a.page_size - 1));
      }
      int32_t pg = raw;
      if (pg < 0 || pg >= a.num_pages) {
        set_status(a.status, DSA_DEV_BOUNDS);
        pg = 0;
      }
      return pg * a.page_size;
    };
    const uint64_t pol = policy_evict_first();
    const int blk_rows = SPARSE ? 8 : a.page_size;
    int nxt_unit;
    // sparse with physical blocks: the K rows of the next kSpTab stages sit in
    // a shared table, refilled with one round of loads every kSpTab stages
    const bool sptab = SPARSE && a.phys != nullptr;
    int *sp_tab = reinterpret_cast<int *>(smem + P.sptab);
    int tab_i = 0;
    int nxt = sptab ? kNone : fetch(git, 0, nxt_unit);
    int cur_row = -1;
    int prev_u = -1, unit_ord = -1;
    long long n_done = 0;  // stages walked; this warp's among them were issued
    int q_issued = 0;
    bool ok = true;
    Ring rs, rk;
    rs.init(S);
    rk.init(KS);
    int o = 0;
    for (long long n = 0; n < count && ok && !idle; ++n, it.next(a), rs.next(), rk.next(),
                   o = (o + 1 == tpg) ? 0 : o + 1) {
      const int u = it.u;
      int row;
      if (sptab) {
        if (tab_i == 0) {
          // flattened stage g = (row, tile) in closed form, so the loads of
          // eight stages are in flight together
          // (paired: stage counts differ per unit, so a copy of the
          // iterator walks the next stages instead)
          const long long gbase = (long long)u_start * a.sparse_tpu + i_start + n;
          TileIter<SPARSE> wt = it;
          if (NN == 1 && a.phys_vec) {
            // the next nst stages' entries are one contiguous run: eight
            // 16-byte loads a stage, converted in place (the row table's
            // layout, stage-major, is the run's own)
            const int nq = 8 * (int)min((long long)kSpTab, count - n);
            const int4 *src = reinterpret_cast<const int4 *>(a.phys + gbase * 32);
            int4 *dst = reinterpret_cast<int4 *>(sp_tab);
#pragma unroll 2
            for (int q = lane; q < nq; q += 32) {
              const int4 v = __ldg(src + q);
              dst[q] = make_int4(phys_block_row(a, v.x), phys_block_row(a, v.y),
                                 phys_block_row(a, v.z), phys_block_row(a, v.w));
            }
          }
          for (int j0 = 0; !(NN == 1 && a.phys_vec) && j0 < kSpTab && n + j0 < count; j0 += 8) {
            int raw[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              raw[jj] = kNone;
              if (n + j0 + jj < count) {
                int uu, ti;
                if (NN == 1) {  // stage numbers fit 32 bits: rows x (kb / 32)
                  const int g = (int)(gbase + j0 + jj);
                  uu = g / a.sparse_tpu;
                  ti = g - uu * a.sparse_tpu;
                } else {
                  uu = wt.u;
                  ti = wt.i;
                  wt.next(a);
                }
                const int blk = ti * 32 + lane;
                if (blk < a.tab_stride) raw[jj] = __ldg(&a.phys[(int64_t)uu * a.tab_stride + blk]);
              }
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) sp_tab[(j0 + jj) * 32 + lane] = to_row(raw[jj], 0);
          }
          __syncwarp();
        }
        row = sp_tab[tab_i * 32 + lane];
        tab_i = (tab_i + 1 == kSpTab) ? 0 : tab_i + 1;
      } else {
        if (o == 0) {
          cur_row = to_row(nxt, nxt_unit);
          for (int k = 0; k < tpg; ++k) git.next(a);
          nxt = fetch(git, n + tpg, nxt_unit);
        }
        row = __shfl_sync(0xffffffffu, cur_row, (o * ppt + my_sl) & 31);
        if (lane >= ppt) row = -1;
      }
      if (role == 0 && u != prev_u) {
        ++unit_ord;
        prev_u = u;
        const int qb = unit_ord & 1;
        int qrow0 = SPARSE ? u * 32 : u * N;
        int nw = N;  // head weights loaded
        if (SPARSE && NN == 2) {
          // paired unit: rows 2m, 2m+1 of its request; an odd last row loads
          // its own weights only (the Q tile's second half is not used)
          const int b = u / a.upr, m2 = 2 * (u - b * a.upr);
          qrow0 = (b * a.req_next_n + m2) * 32;
          if (m2 + 1 >= a.req_next_n) nw = 32;
        }
        if (lane == 0) {
          ok = mbar_wait(QEMPTY(qb), ((unit_ord >> 1) & 1) ^ 1, ctl);
          if (ok) {
            mbar_arrive_expect_tx(QFULL(qb), N * 128 + nw * 4);
            tma_load_2d(qst + qb * (N * 128), &tm_q, QFULL(qb), 0, qrow0);
            bulk_load(smem_u32(w_s + qb * N), a.weights + (int64_t)qrow0, nw * 4, QFULL(qb));
            ++q_issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      if (!mine(n)) {  // the other producer's stage
        n_done = n + 1;
        continue;
      }
      const int s = rs.idx;
      const int kx = rk.idx;
      if (lane == 0) ok = mbar_wait(EMPTY(s), rs.ph ^ 1, ctl) && mbar_wait(KSE(kx), rk.ph ^ 1, ctl);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      const uint32_t nload = (uint32_t)__popc(__ballot_sync(0xffffffffu, row >= 0));
      if (lane == 0) {
        // MX: the 4-bit unpacking copy counts the 64 packed bytes of a row
        mbar_arrive_expect_tx(FULL(s), nload * (uint32_t)(blk_rows * (MX ? 64 : 128)));
        if (!SPARSE) mbar_arrive_expect_tx(KSF(kx), nload * (uint32_t)(blk_rows * 4));
      }
      __syncwarp();
      // sparse with physical blocks: blocks 16..31 go to the second producer
      if (row >= 0 && !(sptab && lane >= 16))
        tma_load_2d_hint(kst + s * kStageK + lane * blk_rows * 128, &tm_k, FULL(s), 0, row, pol);
      if (SPARSE) {
        // kscale of the 32 blocks (32 bytes each) by 16-byte cp.async, two
        // per lane, each lane's completion arriving on KSF by itself: a bulk
        // copy per block would add a second operation per block on the SM's
        // TMA unit, which bounds the sparse pass (about 40 ns per operation)
        const uint32_t sdst = smem_u32(ks_s + kx * kStageTok);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = 16 * h + (lane >> 1), half = lane & 1;
          const int rj = __shfl_sync(0xffffffffu, row, j);
          if (rj >= 0)
            cp_async16_hint(sdst + (uint32_t)((j * 8 + half * 4) * 4),
                            a.kscale + (int64_t)rj + half * 4, pol);
        }
        cp_async_arrive_noinc(KSF(kx));
      } else if (row >= 0) {
        bulk_load(smem_u32(ks_s + kx * kStageTok + lane * blk_rows), a.kscale + (int64_t)row,
                  blk_rows * 4, KSF(kx));
      }
      n_done = n + 1;
    }
    if (SPARSE) cp_async_wait_all();  // this warp's kscale copies land before it moves on
    if (!ok && lane == 0) {
      // drain our own TMA copies still in flight before the CTA exits (the
      // sparse pass's kscale cp.async copies were waited for above)
      // (stage m sits in K slot m % S, phase (m / S) & 1; kscale likewise)
      const long long lim = a.wait_limit;
      for (long long m = n_done > S ? n_done - S : 0; m < n_done; ++m)
        if (mine(m)) mbar_wait_drain(FULL((int)(m % S)), (uint32_t)((m / S) & 1), lim);
      for (long long m = n_done > KS ? n_done - KS : 0; !SPARSE && m < n_done; ++m)
        if (mine(m)) mbar_wait_drain(KSF((int)(m % KS)), (uint32_t)((m / KS) & 1), lim);
      for (int k2 = (q_issued > 2 ? q_issued - 2 : 0); k2 < q_issued; ++k2)
        mbar_wait_drain(QFULL(k2 & 1), (uint32_t)((k2 >> 1) & 1), lim);
    }
  } else if (warp == 1 && MX) {
    // ------------------------------------------------------------ MMA issuer, MXFP4 keys
    // Per stage: the scale-factor warp's two staged tables go to the sub-tiles'
    // A scale-factor columns of TMEM (tcgen05.cp, in issue order with the
    // MMAs that read them), then four block-scaled MMAs a sub-tile, the MMA
    // for dimensions 32kk .. 32kk+31 taking exponent byte kk.
    if (lane == 0) {
      TileIter<SPARSE> it;
      it.init(a, u_start, i_start);
      int prev_u = -1, unit_ord = -1, qb = 0;
      bool ok = true;
      long long mmas = 0;
      Ring rs, ra;
      rs.init(S);
      ra.init(A);
      for (long long n = 0; n < count; ++n, it.next(a), rs.next(), ra.next()) {
        if (it.u != prev_u) {
          ++unit_ord;
          prev_u = it.u;
          qb = unit_ord & 1;
          if (!(ok = mbar_wait(QFULL(qb), (unit_ord >> 1) & 1, ctl))) break;
        }
        const int s = rs.idx;
        const int x = ra.idx;
        if (!(ok = mbar_wait(AEMPTY(x), ra.ph ^ 1, ctl) && mbar_wait(FULL(s), rs.ph, ctl) &&
                   mbar_wait(SFR(s), rs.ph, ctl)))
          break;
        tc_fence_after();
        const uint8_t *stg = smem + P.sfst + s * kSfStage;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tmem_cp_32x128b_x4(sfa0 + 32u * h, sdesc_plain(smem_u32(stg + h * 512), 128, 128));
        const uint64_t bd = sdesc_sw128(qst + qb * (N * 128));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t d = tmem_base + (uint32_t)((2 * x + h) * N);
          const uint64_t ad = sdesc_sw128(kst + s * kStageK + h * kSubK);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 128 E2M1 = 4 steps of 32 (one exponent each)
            mma_mx(d, ad + 2 * kk, bd + 2 * kk, idesc_mx_e2m1_e4m3(128, N, kk, kk), sfa0 + 32u * h,
                   sfb, kk > 0 ? 1u : 0u);
        }
        ++mmas;
        mma_commit(EMPTY(s));
        mma_commit(AFULL(x));
        if (it.i == it.tiles - 1 || n == count - 1) mma_commit(QEMPTY(qb));
      }
      if (!ok && mmas > 0) {
        mma_commit(DRAIN);
        mbar_wait_drain(DRAIN, 0, a.wait_limit);
      }
    }
    __syncwarp();
  } else if (MX && warp == 2 + EW) {
    // ------------------------------------------------------------ scale-factor warp, MXFP4 keys
    // Turns each stage's 256 token exponent words (token order, byte j = the
    // exponent of dimensions 32j .. 32j+31) into the two tables the
    // scale-factor copy reads: row i of sub-tile h holds the words of tokens
    // i, i+32, i+64, i+96 of the sub-tile, which lands token m's exponents in
    // TMEM lane m, column m / 32 of the sub-tile's A scale factors.  Running
    // ahead of the MMA warp, it keeps these loads, stores and the proxy fence
    // off the MMA's per-stage path.  The stage's table slot is free once its
    // exponents have landed: the producer copied them only after the slot's
    // previous MMAs (and the scale-factor copy before them) had completed.
    const uint32_t *kraw = reinterpret_cast<const uint32_t *>(ks_s);
    bool ok = true;
    Ring rs, rk;
    rs.init(S);
    rk.init(KS);
    for (long long n = 0; n < count; ++n, rs.next(), rk.next()) {
      const int s = rs.idx;
      const int kx = rk.idx;
      if (lane == 0) ok = mbar_wait(KSF(kx), rk.ph, ctl);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      uint8_t *stg = smem + P.sfst + s * kSfStage;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint32_t *src = kraw + kx * kStageTok + h * kSubTok + lane;
        *reinterpret_cast<uint4 *>(stg + h * 512 + 16 * lane) =
            make_uint4(src[0], src[32], src[64], src[96]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(KSE(kx));  // the exponents of this ring slot are read
        mbar_arrive(SFR(s));   // the stage's tables are staged
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      TileIter<SPARSE> it;
      it.init(a, u_start, i_start);
      int prev_u = -1, unit_ord = -1, qb = 0;
      bool ok = true;
      long long mmas = 0;
      Ring rs, ra;
      rs.init(S);
      ra.init(A);
      for (long long n = 0; n < count; ++n, it.next(a), rs.next(), ra.next()) {
        if (it.u != prev_u) {
          ++unit_ord;
          prev_u = it.u;
          qb = unit_ord & 1;
          if (!(ok = mbar_wait(QFULL(qb), (unit_ord >> 1) & 1, ctl))) break;
        }
        const int s = rs.idx;
        const int x = ra.idx;
        if (!(ok = mbar_wait(AEMPTY(x), ra.ph ^ 1, ctl))) break;
        if (!(ok = mbar_wait(FULL(s), rs.ph, ctl))) break;
        tc_fence_after();
        const uint64_t bd = sdesc_sw128(qst + qb * (N * 128));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t d = tmem_base + (uint32_t)((2 * x + h) * N);
          const uint64_t ad = sdesc_sw128(kst + s * kStageK + h * kSubK);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 128 FP8 = 4 steps of 32 bytes
            mma_f8(d, ad + 2 * kk, bd + 2 * kk, IDESC, kk > 0 ? 1u : 0u);
        }
        ++mmas;
        mma_commit(EMPTY(s));
        mma_commit(AFULL(x));
        if (it.i == it.tiles - 1 || n == count - 1) mma_commit(QEMPTY(qb));
      }
      if (!ok && mmas > 0) {
        mma_commit(DRAIN);
        mbar_wait_drain(DRAIN, 0, a.wait_limit);
      }
    }
    __syncwarp();
  } else if (SPARSE && warp == 2 + EW) {
    // ------------------------------------------------------------ second producer
    // sparse with physical blocks: the K gathers of blocks 16..31 of every
    // stage (lanes 16..31); warp 0 issues blocks 0..15, the kscale and the
    // barrier accounting.  One TMA operation per 1 KiB block holds the
    // issuing warp for about 80 cycles, so two warps share a stage's issue.
    if (a.phys != nullptr) {
      TileIter<SPARSE> it;
      it.init(a, u_start, i_start);
      const uint64_t pol = policy_evict_first();
      int rq[8];  // this lane's block rows for the next stages, oldest first
      int avail = 0;
      bool ok = true;
      Ring rs;
      rs.init(S);
      long long issued = 0;
      for (long long n = 0; n < count && ok; ++n, it.next(a), rs.next()) {
        if (avail == 0 && NN == 1 && a.phys_vec) {
          // one 16-byte load a lane: lane l holds blocks 16 + 4 (l % 4) ..
          // + 3 of stage l / 4 of the next eight; each lane 16..31 takes its
          // block of every stage from the lane holding it
          const long long gbase = (long long)u_start * a.sparse_tpu + i_start + n;
          int4 v = make_int4(INT32_MAX, INT32_MAX, INT32_MAX, INT32_MAX);
          if (n + (lane >> 2) < count)
            v = __ldg(reinterpret_cast<const int4 *>(a.phys + (gbase + (lane >> 2)) * 32 + 16) +
                      (lane & 3));
          const int src0 = (lane - 16) >> 2, e = lane & 3;
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const int sl = (4 * jj + src0) & 31;
            const int x = __shfl_sync(0xffffffffu, v.x, sl), y = __shfl_sync(0xffffffffu, v.y, sl);
            const int z = __shfl_sync(0xffffffffu, v.z, sl), w = __shfl_sync(0xffffffffu, v.w, sl);
            const int r = e == 0 ? x : e == 1 ? y : e == 2 ? z : w;
            rq[jj] = phys_block_row(a, lane >= 16 ? r : INT32_MAX);
          }
          avail = 8;
        } else if (avail == 0) {
          const long long gbase = (long long)u_start * a.sparse_tpu + i_start + n;
          TileIter<SPARSE> wt = it;
          int raw[8];
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            raw[jj] = INT32_MAX;
            if (n + jj < count) {
              int uu, ti;
              if (NN == 1) {
                const int g = (int)(gbase + jj);
                uu = g / a.sparse_tpu;
                ti = g - uu * a.sparse_tpu;
              } else {
                uu = wt.u;
                ti = wt.i;
                wt.next(a);
              }
              const int blk = ti * 32 + lane;
              if (lane >= 16 && blk < a.tab_stride)
                raw[jj] = __ldg(&a.phys[(int64_t)uu * a.tab_stride + blk]);
            }
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) rq[jj] = phys_block_row(a, raw[jj]);
          avail = 8;
        }
        const int row = rq[0];
#pragma unroll
        for (int k = 0; k < 7; ++k) rq[k] = rq[k + 1];
        --avail;
        const int s = rs.idx;
        // Wait for the slot only in a stage this warp loads into.  A stage
        // whose blocks 16..31 are all padding completes without this warp
        // (warp 0 arms its barrier for the other blocks alone), so the MMA
        // may release the slot before this warp gets there, and a wait on it
        // would then be for a phase already past.  A stage this warp loads
        // into cannot complete without it, so that wait is never behind.
        if (__ballot_sync(0xffffffffu, row >= 0) != 0) {
          if (lane == 0) ok = mbar_wait(EMPTY(s), rs.ph ^ 1, ctl);
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (row >= 0)
            tma_load_2d_hint(kst + s * kStageK + lane * 8 * 128, &tm_k, FULL(s), 0, row, pol);
        }
        ++issued;
      }
      if (!ok && lane == 0) {
        // drain this warp's own copies still in flight
        Ring ds = rs;
        ds.idx = (int)(issued % S);
        ds.ph = (uint32_t)((issued / S) & 1);
        for (int back = 1; back <= S && back <= issued; ++back) {
          int i2;
          uint32_t p2;
          ds.prev(back, i2, p2);
          mbar_wait_drain(FULL(i2), p2, a.wait_limit);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // warpgroup gi takes sub-tile g = gi % 2 of the stages of parity gi / 2
    // (every stage at next_n = 1); warp w reads TMEM lanes 32*(w%4) .. +31,
    // i.e. one token per thread.  Every warp walks every stage for the
    // bookkeeping (unit changes, histogram flushes, Q release).
    const int gi = (warp - 2) >> 2;
    const int g = gi & 1;        // sub-tile
    const int par = gi >> 1;     // stage parity (0 when NPAR == 1)
    const int quarter = warp & 3;
    const int lane_base = 32 * quarter;
    const int tok = g * kSubTok + lane_base + lane;   // token within the stage
    const int gtid = par * 128 + ((warp - 2) & 3) * 32 + lane;  // within the sub-tile's warps
    const uint64_t out_pol = policy_evict_last();
    uint32_t *grp_hist = hist_s + g * HS * NN * kHistWords;
    uint32_t *my_hist = grp_hist + (HS == 4 ? quarter : 0) * NN * kHistWords;
    TileIter<SPARSE> it;
    it.init(a, u_start, i_start);
    int prev_u = -1, unit_ord = -1, qb = 0;
    uint32_t gsync_ph = 0;
    int64_t ctx_b = 0, n_row = 0;
    // dense: the current request's rows (their first logit) and, per row, the
    // positions stored: below min(live length, row stride), set per request
    float *orow = nullptr;
    float wr[32];  // next_n = 1: the current row's head weights
    uint32_t lim[NN];
#pragma unroll
    for (int j = 0; j < NN; ++j) lim[j] = 0;
    int row_base = 0;
    bool ok = true;
    // paired unit: its rows, their live lengths and the union length
    int row_a = 0, row_b = -1, nu = 0;
    int64_t v_a = 0, v_b = 0;
    // one sparse score, in the output format
    auto sp_store = [&](int64_t row, int64_t p, float val) {
      if (OUT == DSA_OUT_F16) {
        reinterpret_cast<__half *>(a.out)[row * a.out_stride + p] = __float2half_rn(val);
      } else if (OUT == DSA_OUT_BF16) {
        reinterpret_cast<__nv_bfloat16 *>(a.out)[row * a.out_stride + p] = __float2bfloat16_rn(val);
      } else {
        reinterpret_cast<float *>(a.out)[row * a.out_stride + p] = val;
      }
    };
    // a paired row's share of a union position: its own table slot p_tab
    // (live below its valid length, -inf past it), and the padding slots
    // [blocks * 8, kb * 8) of its output, which the union walk visits once
    auto pair_store = [&](int row, int p_tab, int64_t pos, int64_t v, float val) {
      if (p_tab >= 0 && p_tab < a.kb) {
        const int64_t p = (int64_t)p_tab * 8 + (pos & 7);
        sp_store(row, p, p < v ? val : -INFINITY);
      }
      if (pos >= ((v + 7) >> 3) * 8 && pos < (int64_t)a.kb * 8) sp_store(row, pos, -INFINITY);
    };

    auto ewait = [&](uint32_t bar, uint32_t parity) -> bool {
      const bool r = mbar_wait(bar, parity, ctl);
      return __all_sync(0xffffffffu, r) != 0;
    };
    auto group_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(GSYNC(g));
      const bool r = ewait(GSYNC(g), gsync_ph);
      gsync_ph ^= 1;
      return r;
    };
    // add this group's counts of the current request to the global
    // histogram (packed 64-bit atomics on bin pairs) and clear its slots
    auto flush = [&](int rb) -> bool {
      if (!group_sync()) return false;
      for (int j = 0; j < NN; ++j) {
        for (int p = gtid; p < kHistWords; p += 128 * NPAR) {
          uint32_t c0 = 0, c1 = 0;
#pragma unroll
          for (int w = 0; w < HS; ++w) {
            uint32_t *sl = grp_hist + (w * NN + j) * kHistWords + p;
            c0 += *sl & 0xFFFFu;
            c1 += *sl >> 16;
            *sl = 0;
          }
          if (c0 | c1) {
            unsigned long long *gp = reinterpret_cast<unsigned long long *>(
                a.histogram + (int64_t)(rb + j) * DSA_NUM_BINS + 2 * p);
            atomicAdd(gp, ((unsigned long long)c1 << 32) | c0);
          }
        }
      }
      return group_sync();
    };

    Ring ra, rk;
    ra.init(A);
    rk.init(KS);
    int since_flush = 0;  // stages counted into the slots since their last flush
    for (long long n = 0; n < count; ++n, it.next(a), ra.next(), rk.next()) {
      const int u = it.u, i = it.i;
      if (HIST && u == prev_u && ++since_flush >= kHistFlushStages) {
        if (!(ok = flush(row_base))) break;  // every warp of the group walks every stage
        since_flush = 0;
      }
      if (u != prev_u) {
        if (HIST && prev_u >= 0) {
          if (!(ok = flush(row_base))) break;
        }
        since_flush = 0;
        ++unit_ord;
        prev_u = u;
        qb = unit_ord & 1;
        if (SPARSE && NN == 2) {
          const int b = u / a.upr, m2 = 2 * (u - b * a.upr);
          row_a = b * a.req_next_n + m2;
          row_b = (m2 + 1 < a.req_next_n) ? row_a + 1 : -1;
          nu = min(__ldg(&a.ulen[u]), a.tab_stride);
          v_a = __ldg(&a.valid_lens[row_a]);
          v_b = row_b >= 0 ? __ldg(&a.valid_lens[row_b]) : 0;
        } else if (SPARSE && a.valid_lens) {
          n_row = __ldg(&a.valid_lens[u]);  // live positions of the sparse row
        } else if (SPARSE) {
          const int b = u / a.req_next_n;
          const int j = u - b * a.req_next_n;
          n_row = eff_ctx(a, b) - (a.req_next_n - 1 - j);
          if (n_row < 0) n_row = 0;
        } else {
          ctx_b = eff_ctx(a, u);
          row_base = u * NN;
          orow = reinterpret_cast<float *>(a.out) + (int64_t)row_base * a.out_stride;
#pragma unroll
          for (int j = 0; j < NN; ++j) {
            const int64_t n_rj = ctx_b - (NN - 1 - j);
            lim[j] = (uint32_t)max((int64_t)0, min(n_rj, a.out_stride));
          }
          // a live position past the row stride is flagged, not stored
          if (lane == 0 && ctx_b > a.out_stride) set_status(a.status, DSA_DEV_BOUNDS);
        }
        if (!(ok = ewait(QFULL(qb), (unit_ord >> 1) & 1))) break;
        if constexpr (EW == 8) {  // next_n = 1: the row's head weights into registers
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 wv = *reinterpret_cast<const float4 *>(w_s + qb * N + h);
            wr[h + 0] = wv.x;
            wr[h + 1] = wv.y;
            wr[h + 2] = wv.z;
            wr[h + 3] = wv.w;
          }
        }
      }
      const bool mine = NPAR == 1 || ((int)(n & 1) == par);
      if (mine) {
      const int x = ra.idx;
      const int kx = rk.idx;
      const int64_t pos = (int64_t)i * kStageTok + tok;
      int32_t blk = INT32_MAX;
      uint32_t pw = 0;  // paired: the union entry's two table positions
      if (SPARSE && NN == 2 && (pos >> 3) < nu)
        pw = (uint32_t)__ldg(&a.upos[(int64_t)u * a.tab_stride + (pos >> 3)]);
      if (SPARSE && NN == 1 && !a.valid_lens && pos < (int64_t)a.kb * 8)
        blk = __ldg(&a.block_table[(int64_t)u * a.kb + pos / 8]);
      float ks = 1.0f;  // MX: the block exponents were applied by the MMA
      if (!MX) {
        if (!(ok = ewait(KSF(kx), rk.ph))) break;
        ks = ks_s[kx * kStageTok + tok];
        __syncwarp();
        if (lane == 0) mbar_arrive(KSE(kx));
      }
      if (!(ok = ewait(AFULL(x), ra.ph))) break;
      tc_fence_after();
      // head dots leave TMEM in batches of up to two rows; with 16 epilogue
      // warps (576 threads leave 96 registers a thread) in half rows of 16
      // heads, the load of the next half in flight while one is summed.  The
      // accumulator goes back to the MMA as soon as the last load is in.
      float acc[NN];
      const uint32_t tcol = tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)((2 * x + g) * N);
      constexpr int kB = NN == 1 ? 1 : (EW == 8 ? 2 : 1);
      if constexpr (EW == 16) {
        const float *wq = w_s + qb * N;
        uint32_t hv[2][16];
        uint64_t c01 = 0, c23 = 0;
        tmem_ld16(tcol, hv[0]);
        tmem_ld_wait();
        const bool ksok = ks >= 0.0f && ks <= 3.4028234e38f;
        // one unrolled pass per case, chosen per warp (the TMEM loads in it
        // need the whole warp; padding tokens may carry any kscale)
        auto run = [&](auto allok_tag) {
          constexpr bool ALLOK = decltype(allok_tag)::value;
#pragma unroll
          for (int step = 0; step < 2 * NN; ++step) {  // row step / 2, heads 16 (step % 2) ..
            if (step + 1 < 2 * NN) {
              tmem_ld16(tcol + (uint32_t)((step + 1) * 16), hv[(step + 1) & 1]);
            } else {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(AEMPTY(x));
            }
            if ((step & 1) == 0) c01 = c23 = pk2(0.0f, 0.0f);
            head_sum_part<ALLOK>(hv[step & 1], ks, ksok, wq + 16 * step, c01, c23);
            if (step & 1) {
              float c0, c1, c2, c3;
              upk2(c01, c0, c1);
              upk2(c23, c2, c3);
              const float sm = (c0 + c1) + (c2 + c3);
              acc[step >> 1] = (ALLOK || ksok) ? ks * sm : sm;
            }
            if (step + 1 < 2 * NN) tmem_ld_wait();
          }
        };
        if (__all_sync(0xffffffffu, ksok)) run(std::true_type{});
        else run(std::false_type{});
      } else {
#pragma unroll
      for (int j0 = 0; j0 < NN; j0 += kB) {
        uint32_t v[kB][32];
#pragma unroll
        for (int jj = 0; jj < kB; ++jj)
          if (j0 + jj < NN) tmem_ld32(tcol + (uint32_t)((j0 + jj) * 32), v[jj]);
        tmem_ld_wait();
        if (j0 + kB >= NN) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(AEMPTY(x));
        }
#pragma unroll
        for (int jj = 0; jj < kB; ++jj)
          if (j0 + jj < NN) acc[j0 + jj] = head_sum(v[jj], ks, wr);
      }
      }

      if (SPARSE && NN == 2) {
        pair_store(row_a, (int)(pw & 0xffffu) - 1, pos, v_a, acc[0]);
        if (row_b >= 0) pair_store(row_b, (int)(pw >> 16) - 1, pos, v_b, acc[NN - 1]);
      } else if (SPARSE) {
        if (pos < (int64_t)a.kb * 8) {
          const int64_t t = (int64_t)blk * 8 + (pos & 7);
          const bool live = a.valid_lens ? pos < n_row : (blk != INT32_MAX && blk >= 0 && t < n_row);
          sp_store(u, pos, live ? acc[0] : -INFINITY);
        }
      } else {
        const uint32_t t32 = (uint32_t)i * kStageTok + (uint32_t)tok;  // position in the row
#pragma unroll
        for (int j = 0; j < NN; ++j) {
          if (t32 < lim[j]) {
            // kept in L2 for the select that reads the row next (the K stream
            // around it is marked evict-first)
            st_f32_hint(orow + j * a.out_stride + t32, acc[j], out_pol);
            if (HIST) {
              const int bin = coarse_bin(acc[j]);
              if (bin >= 0) atomicAdd(&my_hist[j * kHistWords + (bin >> 1)], 1u << (16 * (bin & 1)));
            }
          }
          if (a.amax != nullptr) {
            // block maximum of 8 consecutive scores (8 consecutive lanes), in
            // the value order of the select (-0 below +0, NaN ignored); the
            // newest block is +inf, nothing is written past the block count
            const int64_t t = pos;
            const int64_t n_rj = ctx_b - (NN - 1 - j);
            const int64_t nb = n_rj > 0 ? (n_rj + 7) >> 3 : 0;
            uint32_t key = (t < n_rj && !isnan(acc[j])) ? f32_order_key(acc[j]) : 0u;
            key = max(key, __shfl_xor_sync(0xffffffffu, key, 1));
            key = max(key, __shfl_xor_sync(0xffffffffu, key, 2));
            key = max(key, __shfl_xor_sync(0xffffffffu, key, 4));
            const int64_t blk = t >> 3;
            if ((lane & 7) == 0 && blk < nb && (a.amax_skip <= 0 || nb > a.amax_skip)) {
              float m;
              if (blk == nb - 1) {
                m = INFINITY;
              } else {
                const uint32_t bits = (key & 0x80000000u) ? (key ^ 0x80000000u) : ~key;
                m = key ? __uint_as_float(bits) : __int_as_float(0x7fc00000);
              }
              if (blk < a.amax_stride) a.amax[(int64_t)(row_base + j) * a.amax_stride + blk] = m;
              else set_status(a.status, DSA_DEV_BOUNDS);
            }
          }
        }
      }
      }  // mine
      if (i == it.tiles - 1 || n == count - 1) {
        __syncwarp();
        if (lane == 0) mbar_arrive(QEMPTY(qb));
      }
    }
    if (HIST && ok && prev_u >= 0) flush(row_base);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, a.tmem_cols);
  }
}

// Stage count and ring depths for one instantiation: as many 32 KiB K stages
// as fit next to the Q/weight buffers, the histogram slots and a kscale ring
// deep enough (stages + accumulators + 2) never to hold the producer back.
struct LaunchPlan {
  int stages, nacc, nks, cols, smem;
};

inline LaunchPlan plan_for(int nn, bool hist, bool sparse, bool mx = false) {
  LaunchPlan L;
  const int N = 32 * nn;
  // TMEM pairs (two 128-lane sub-tiles each); MX keeps 96 columns after the
  // pairs for the scale factors (two A regions and the B region, 32 apart)
  L.nacc = std::min(4, 512 / (2 * N));
  if (mx)
    while (L.nacc > 1 && 2 * L.nacc * N + 96 > 512) --L.nacc;
  L.cols = 32;
  while (L.cols < 2 * L.nacc * N + (mx ? 96 : 0)) L.cols <<= 1;
  L.stages = kMaxStages;
  while (L.stages > 2 &&
         smem_plan(nn, hist, sparse, L.stages, L.nacc, L.stages + L.nacc + 2, mx).total > kSmemLimit)
    --L.stages;
  L.nks = L.stages + L.nacc + 2;
  L.smem = smem_plan(nn, hist, sparse, L.stages, L.nacc, L.nks, mx).total;
  return L;
}

template <int NN, bool SPARSE, int OUT, bool HIST, bool MX = false>
dsa_status_t launch_one(const CUtensorMap &tk, const CUtensorMap &tq, const LogitsArgs &a0,
                        int grid, cudaStream_t st) {
  LogitsArgs a = a0;
  const LaunchPlan L = plan_for(NN, HIST, SPARSE, MX);
  a.num_acc = L.nacc;
  a.num_ks = L.nks;
  a.tmem_cols = (uint32_t)L.cols;
  a.num_stages = L.stages;
  auto kfn = logits_kernel<NN, SPARSE, OUT, HIST, MX>;
  if (!ensure_smem_attr(reinterpret_cast<const void *>(kfn), L.smem)) return DSA_ERR_CUDA;
  return launch_pdl(kfn, dim3(grid), dim3(threads_for(NN, SPARSE, MX)), (size_t)L.smem, st, tk, tq, a);
}

}  // namespace

int logits_stages_for(int next_n, bool hist, bool mx) {
  return plan_for(next_n, hist, false, mx).stages;
}

dsa_status_t run_paged_logits(const LogitsCall &c, cudaStream_t st) {
  CUtensorMap tk, tq;
  if (c.mx && c.sparse) return DSA_ERR_UNSUPPORTED;
  dsa_status_t e = c.mx ? make_tmap_rows_e2m1(&tk, c.kv, (uint64_t)c.num_pages * c.page_size,
                                               c.page_size)
                        : make_tmap_rows128(&tk, c.kv, (uint64_t)c.num_pages * c.page_size,
                                            c.sparse ? 8 : c.page_size);
  if (e != DSA_OK) return e;
  const int nn = c.sparse ? (c.union_len ? 2 : 1) : c.next_n;
  e = make_tmap_rows128(&tq, c.q, (uint64_t)c.B * c.next_n * 32, 32 * nn);
  if (e != DSA_OK) return e;
  LogitsArgs a{};
  a.context_lens = c.context_lens;
  a.page_table = c.page_table;
  a.pt_stride = c.pt_stride;
  a.kscale = c.kscale;
  a.weights = c.weights;
  a.B = c.B;
  a.req_next_n = c.next_n;
  a.page_size = c.page_size;
  a.log2_ps = (c.page_size == 128) ? 7 : 6;
  a.num_pages = c.num_pages;
  a.block_table = c.block_table;
  a.kb = c.kb;
  a.phys = c.sparse ? c.phys : nullptr;
  a.valid_lens = c.sparse ? c.valid_lens : nullptr;
  a.tab_stride = c.kb;
  a.phys_vec = 0;
  a.upr = 1;
  const bool paired = c.sparse && c.union_len != nullptr;
  if (paired) {
    a.phys = c.union_phys;
    a.upos = c.union_pos;
    a.ulen = c.union_len;
    a.tab_stride = 2 * c.kb;
    a.upr = (c.next_n + 1) / 2;
  }
  a.out = c.out;
  a.out_stride = c.out_stride;
  a.histogram = c.histogram;
  a.amax = c.sparse ? nullptr : c.amax;
  a.amax_stride = c.amax_stride;
  a.amax_skip = c.amax_skip;
  a.status = c.status;
  a.wait_limit = c.wait_limit;
  const int sms = num_sms();
  if (sms <= 0) return DSA_ERR_CUDA;
  if (paired) {
    // stage counts per unit come from the union lengths on the device
    a.num_units = c.B * a.upr;
    a.sparse_tpu = (c.kb + 31) / 32;
    const long long tiles = (long long)a.num_units * 2 * a.sparse_tpu;
    const int grid = (int)std::max<long long>(1, std::min<long long>(sms, tiles));
    if (c.out_fmt == DSA_OUT_F16) return launch_one<2, true, DSA_OUT_F16, false>(tk, tq, a, grid, st);
    if (c.out_fmt == DSA_OUT_BF16)
      return launch_one<2, true, DSA_OUT_BF16, false>(tk, tq, a, grid, st);
    return launch_one<2, true, DSA_OUT_F32, false>(tk, tq, a, grid, st);
  }
  if (c.sparse) {
    a.num_units = c.B * c.next_n;
    a.sparse_tpu = (c.kb + 31) / 32;
    a.phys_vec = (a.phys && c.kb % 32 == 0 && (reinterpret_cast<uintptr_t>(a.phys) & 15) == 0) ? 1 : 0;
    const long long tiles = (long long)a.num_units * a.sparse_tpu;
    const int grid = (int)std::max<long long>(1, std::min<long long>(sms, tiles));
    if (c.out_fmt == DSA_OUT_F16) return launch_one<1, true, DSA_OUT_F16, false>(tk, tq, a, grid, st);
    if (c.out_fmt == DSA_OUT_BF16)
      return launch_one<1, true, DSA_OUT_BF16, false>(tk, tq, a, grid, st);
    return launch_one<1, true, DSA_OUT_F32, false>(tk, tq, a, grid, st);
  }
  a.num_units = c.B;
  a.sparse_tpu = 0;
  const int grid = sms;
  const bool h = c.histogram != nullptr;
  if (c.mx) {
    switch (c.next_n) {
      case 1:
        return h ? launch_one<1, false, DSA_OUT_F32, true, true>(tk, tq, a, grid, st)
                 : launch_one<1, false, DSA_OUT_F32, false, true>(tk, tq, a, grid, st);
      case 2:
        return h ? launch_one<2, false, DSA_OUT_F32, true, true>(tk, tq, a, grid, st)
                 : launch_one<2, false, DSA_OUT_F32, false, true>(tk, tq, a, grid, st);
      case 3:
        return h ? launch_one<3, false, DSA_OUT_F32, true, true>(tk, tq, a, grid, st)
                 : launch_one<3, false, DSA_OUT_F32, false, true>(tk, tq, a, grid, st);
      case 4:
        return h ? launch_one<4, false, DSA_OUT_F32, true, true>(tk, tq, a, grid, st)
                 : launch_one<4, false, DSA_OUT_F32, false, true>(tk, tq, a, grid, st);
      default:
        return DSA_ERR_UNSUPPORTED;
    }
  }
  switch (c.next_n) {
    case 1:
      return h ? launch_one<1, false, DSA_OUT_F32, true>(tk, tq, a, grid, st)
               : launch_one<1, false, DSA_OUT_F32, false>(tk, tq, a, grid, st);
    case 2:
      return h ? launch_one<2, false, DSA_OUT_F32, true>(tk, tq, a, grid, st)
               : launch_one<2, false, DSA_OUT_F32, false>(tk, tq, a, grid, st);
    case 3:
      return h ? launch_one<3, false, DSA_OUT_F32, true>(tk, tq, a, grid, st)
               : launch_one<3, false, DSA_OUT_F32, false>(tk, tq, a, grid, st);
    case 4:
      return h ? launch_one<4, false, DSA_OUT_F32, true>(tk, tq, a, grid, st)
               : launch_one<4, false, DSA_OUT_F32, false>(tk, tq, a, grid, st);
    default:
      return DSA_ERR_UNSUPPORTED;
  }
}

}  // namespace dsa
