// dsa_device.cuh -- device-side building blocks shared by the sm_103a kernels:
// inline-PTX wrappers for mbarriers, TMA (cp.async.bulk[.tensor]), the
// tcgen05 tensor-core/TMEM instructions, bounded waits that record a status
// bit instead of hanging, and the coarse score bin / order-key functions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"  // include/ is on the include path

namespace dsa {

// ---------------------------------------------------------------- workspace
// Byte layout of the caller's workspace (see dsa_workspace_size).
struct WsLayout {
  static constexpr size_t kStatusOff = 0;         // uint32 status word (+ padding)
  static constexpr size_t kHeader = 256;
  // per row: 4 x int32 counters {emitted, candidates, done CTAs, spare}
  static size_t counters_off() { return kHeader; }
  static size_t counters_bytes(int64_t R) { return (size_t)R * 16; }
  // per row: DSA_CAND_CAP x uint64 (key << 32 | ~column) candidates
  static size_t cand_off(int64_t R) { return align(counters_off() + counters_bytes(R)); }
  static size_t cand_bytes(int64_t R) { return (size_t)R * DSA_CAND_CAP * 8; }
  // per row: 1024 int32 histogram for selects given no histogram
  static size_t hist_off(int64_t R) { return align(cand_off(R) + cand_bytes(R)); }
  static size_t hist_bytes(int64_t R) { return (size_t)R * DSA_NUM_BINS * 4; }
  // per row: 4096 int32 fine histogram of a threshold bin over capacity
  static size_t fine_off(int64_t R) { return align(hist_off(R) + hist_bytes(R)); }
  static size_t fine_bytes(int64_t R) { return (size_t)R * 4096 * 4; }
  static size_t total(int64_t R) { return align(fine_off(R) + fine_bytes(R)); }
  static size_t align(size_t x) { return (x + 255) & ~(size_t)255; }
};

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------- smem / sync
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm volatile("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

// ---------------------------------------------------------------- launches
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while its predecessor on the stream finishes.
// pdl_wait() blocks until every predecessor grid has completed and its memory
// is visible; each kernel calls it before touching memory a predecessor
// writes.  Kernels do not release their dependents early as a rule
// (griddepcontrol.launch_dependents): CTAs of the next grid that became
// resident while a large grid was still running slowed that grid down by more
// than the launch latency they hid, so dependents launch as the running
// grid's CTAs exit.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// The one exception: a small grid whose successor can set itself up on the
// SMs the small grid leaves idle releases it at once (sort -> sparse logits).
__device__ __forceinline__ void pdl_release_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- clusters
// Distributed shared memory: map a shared address of this CTA to the same
// variable in CTA `rank` of the cluster, and access it there.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t dsmem_map(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ int dsmem_atomic_add(uint32_t addr, int v) {
  int old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v)
               : "memory");
  return old;
}
__device__ __forceinline__ void dsmem_red_add(uint32_t addr, int v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ int dsmem_ld(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int4 dsmem_ld4(uint32_t addr) {
  int4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_st64(uint32_t addr, unsigned long long v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void dsmem_st32(uint32_t addr, int v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// All threads of all CTAs of the cluster meet (shared-memory writes before it
// are visible to every CTA after it).
// The two halves of cluster_sync(), for work placed between them: a thread's
// writes before its arrive are visible to every CTA after that CTA's wait.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared abort flag + global status for one CTA's bounded waits.
struct WaitCtl {
  volatile int *abort_flag;  // shared memory
  uint32_t *status;          // global
  long long limit;           // clock64 cycles
};

// Wait for the phase with `parity` to complete.  Gives up (returns false) when
// another role of the CTA aborted, or after ctl.limit cycles, in which case it
// records DSA_DEV_TIMEOUT and raises the CTA's abort flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl &ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*ctl.abort_flag) return false;
    if (clock64() - t0 > ctl.limit) {
      *ctl.abort_flag = 1;
      set_status(ctl.status, DSA_DEV_TIMEOUT);
      return false;
    }
  }
}

// Same, without abort propagation: used while draining after an abort.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar, int32_t x, int32_t y,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// The same with an L2 eviction policy for the source lines.
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void *src, uint32_t bytes,
                                               uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Arrive on `bar` once all cp.async copies issued so far by this thread have
// landed (the barrier's expected count must include this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 16-byte asynchronous copy global -> shared through the LSU path, with an
// L2 cache policy.
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void *src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Global store / read-only vector load with an L2 eviction policy.
__device__ __forceinline__ void st_f32_hint(float *ptr, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(ptr), "f"(v), "l"(policy)
               : "memory");
}
__device__ __forceinline__ float4 ld_f4_hint(const float *ptr, uint64_t policy) {
  float4 v;
  asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0, %1, %2, %3}, [%4], %5;"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(ptr), "l"(policy));
  return v;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, FP8 E4M3 x E4M3 -> FP32, issued by one thread.
__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// Instruction descriptor for kind::f8f6f4: D = FP32, A = B = E4M3, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= (A[smem] * sA) * (B[smem] * sB)^T with block scale factors:
// A E2M1 (MXFP4 keys, one UE8M0 exponent per 32 K-elements), B E4M3, FP32
// accumulate; the scale factors are read from TMEM (sfa / sfb columns), the
// byte within each 32-bit cell chosen by the scale-factor ids of `idesc`.
__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                       uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Instruction descriptor of the block-scaled kind::mxf8f6f4 MMA: A = E2M1,
// B = E4M3, both K-major, D = FP32, N >> 3 at bit 17, UE8M0 scale factors
// (bit 23), M >> 4 at bit 24, the A scale-factor byte id at bits 29-30 and
// the B one at bits 4-5.
__host__ __device__ constexpr uint32_t idesc_mx_e2m1_e4m3(int M, int N, int a_sf_id, int b_sf_id) {
  return ((uint32_t)b_sf_id << 4) | (5u << 7) | (0u << 10) | ((uint32_t)(N >> 3) << 17) |
         (1u << 23) | ((uint32_t)(M >> 4) << 24) | ((uint32_t)a_sf_id << 29);
}

// Copy a 32-row x 16-byte shared-memory matrix into 32 TMEM lanes x 4 columns,
// repeated in all four lane quarters (issued by one thread, ordered before the
// MMAs it issues after it).
__device__ __forceinline__ void tmem_cp_32x128b_x4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// 32 lanes x 4 columns of 32-bit data from registers: thread i of the warp
// writes columns taddr .. taddr + 3 of TMEM lane (warp's lane base + i).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2,
                                         uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(v0), "r"(v1), "r"(v2), "r"(v3)
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Generic-proxy shared-memory writes become visible to the async proxy
// (tcgen05.cp / TMA reads) issued after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor of a plain (no swizzle) K-major operand:
// core matrices of 8 rows x 16 bytes stored contiguously, `sbo` bytes between
// 8-row groups, `lbo` bytes between core matrices along K.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(lbo >> 4) << 16;
  d |= (uint64_t)(sbo >> 4) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version (sm_100 family); swizzle none
  return d;
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle
// layout TMA writes (rows of 128 bytes, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading byte offset (unused for SW128 K-major)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                    // swizzle mode: 128 B
  return d;
}

// 32 lanes x 32 columns of 32-bit TMEM data: thread i of the warp receives
// the 32 consecutive columns of TMEM lane (warp's lane base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// 32 lanes x 16 columns: thread i receives 16 consecutive columns of its lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- scores
// Coarse bin of one score ([DG94] "What this adds"): 1024 descending bins,
// bin 0 = largest.  |x| >= 223 -> magnitude code 511; 16 <= |x| < 223 ->
// 304 + floor(|x|) - 16; |x| < 16 -> FP16-RN(|x|) >> 6.  bin = 511 - m for a
// clear sign bit, 512 + m otherwise; -1 for NaN.
__device__ __forceinline__ int coarse_bin(float x) {
  const float a = fabsf(x);
  int m = static_cast<int>(__half_as_ushort(__float2half_rn(a)) >> 6);  // |x| < 16
  // 16 <= |x| < 223: floor(a) as the low bits of a + 2^23 rounded down (an
  // add instead of a float-to-int conversion; exact below 2^23)
  const int mu = __float_as_int(__fadd_rd(a, 8388608.0f)) - (0x4B000000 - 288);
  m = a >= 16.0f ? mu : m;
  m = a >= 223.0f ? 511 : m;
  // 511 - m for a clear sign bit, 512 + m for a set one: m ^ 511 or m ^ 512 (m < 512)
  const int bin = m ^ (511 + static_cast<int>(__float_as_uint(x) >> 31));
  return isnan(x) ? -1 : bin;
}

// Ascending order key of an FP32 value: unsigned compare == value compare,
// -inf lowest, -0 just below +0.
__device__ __forceinline__ uint32_t f32_order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Order keys of the two FP16 halves of a 32-bit word at once ([VL52696]
// "Why": both packed halves are transformed with one 32-bit operation).  A
// set sign bit flips all 16 bits, a clear one flips only the sign bit.  NaN
// halves become key 0, below every non-NaN key (-inf has key 0x03FF).
template <uint32_t kNanAdd>
__device__ __forceinline__ uint32_t x16x2_order_keys(uint32_t w) {
  const uint32_t sign = (w >> 15) & 0x00010001u;
  uint32_t k = w ^ ((sign * 0x7FFFu) | 0x80008000u);
  // NaN (magnitude above the infinity pattern) iff (h & 0x7FFF) + kNanAdd
  // carries into bit 15: kNanAdd = 0x03FF for FP16 (inf 0x7C00), 0x007F for
  // BF16 (inf 0x7F80)
  const uint32_t nan_bits = ((w & 0x7FFF7FFFu) + (kNanAdd * 0x00010001u)) & 0x80008000u;
  const uint32_t nan_mask = (nan_bits >> 15) * 0xFFFFu;
  return k & ~nan_mask;
}
__device__ __forceinline__ uint32_t f16x2_order_keys(uint32_t w) {
  return x16x2_order_keys<0x03FFu>(w);
}
// The same for two BF16 halves (the same sign-magnitude order).
__device__ __forceinline__ uint32_t bf16x2_order_keys(uint32_t w) {
  return x16x2_order_keys<0x007Fu>(w);
}

}  // namespace dsa
