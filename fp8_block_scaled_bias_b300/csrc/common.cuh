// Shared device helpers for the sm_103a kernels: status reporting, bounded mbarrier
// waits, TMA loads, tcgen05 (TMEM allocation, MMA issue, commit, TMEM loads) and FP8
// conversion.  Inline PTX only; no library code.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/moe_fp8.h"

#define MOE_DEV __device__ __forceinline__

namespace moe {

// ---- status --------------------------------------------------------------------------

// First device error wins: only a 0 status is overwritten.
MOE_DEV void set_status(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

MOE_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A wait that lasts this long means the pipeline is broken; the kernel then stops,
// reports MOE_ERR_DEVICE_TIMEOUT and returns instead of hanging the GPU.
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// ---- shared-memory addresses and mbarriers --------------------------------------------

MOE_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MOE_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

MOE_DEV void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

MOE_DEV void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

MOE_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

MOE_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

MOE_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Same, with cluster-scope acquire: for barriers that the other CTA of a pair arrives on.
MOE_DEV bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with `parity` has completed.  Returns false (after setting
// *abort and the status word) if the wait exceeds kWaitLimitNs, or if another thread
// of the block has already aborted.
// CLUSTER: cluster-scope acquire (the barrier receives arrivals from the other CTA of a
// pair).  limit_ns: the wait limit (kWaitLimitNs unless a caller asks for less).
template <bool CLUSTER = false>
MOE_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* status,
                       uint64_t limit_ns = kWaitLimitNs) {
  auto poll = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (poll()) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (poll()) return true;
    if ((i & 255u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        set_status(status, MOE_ERR_DEVICE_TIMEOUT);
        return false;
      }
    }
  }
}

// Warp-wide wait: lane 0 polls the barrier (the other lanes do not compete for shared
// memory while they wait), then the warp resynchronises.  All lanes get the result.
template <bool CLUSTER = false>
MOE_DEV bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* status,
                            uint64_t limit_ns = kWaitLimitNs) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait<CLUSTER>(bar, parity, abort, status, limit_ns) ? 1 : 0;
  ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
  return ok != 0;
}

// ---- TMA -----------------------------------------------------------------------------

MOE_DEV void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load of one box into shared memory; completion is signalled on `bar` as
// transaction bytes.  x is the innermost (contiguous) coordinate in elements.
MOE_DEV void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Same, with an L2 eviction-priority hint (a createpolicy result).
MOE_DEV void tma_load_2d_hint(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

// ---- cp.async (per-thread asynchronous global -> shared copies) ----------------------------

MOE_DEV void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

MOE_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Arrive on `bar` once every cp.async this thread issued so far has landed (the barrier's
// expected count includes this arrival: .noinc).
MOE_DEV void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Wait until at most N of this thread's committed groups are still in flight.
template <int N>
MOE_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ---- CTA pairs (clusters of two CTAs sharing one tcgen05 MMA) -------------------------

MOE_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

MOE_DEV uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

MOE_DEV uint32_t ncluster_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// All threads of both CTAs of the cluster (release/acquire ordering of shared memory).
MOE_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// The shared::cluster address of the object at shared::cta address `a` in CTA `rank`.
MOE_DEV uint32_t mapa_shared(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}

// Arrive on an mbarrier that may sit in the other CTA of the pair.  Default (CTA-scope)
// release: what the arrival orders are this thread's tcgen05 loads, through
// tcgen05.fence::before_thread_sync, and no generic-proxy data.  A cluster-scope release
// waits for the thread's outstanding memory operations to become visible cluster-wide;
// measured on this B300 it added ~900 cycles to every TMEM-buffer release of the pair.
MOE_DEV void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

MOE_DEV void mbar_arrive_expect_tx_cluster(uint32_t cluster_bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_bar),
               "r"(bytes)
               : "memory");
}

// 2-D tiled load into this CTA's shared memory whose completion (transaction bytes) is
// signalled on an mbarrier of either CTA of the pair.
MOE_DEV void tma_load_2d_pair(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                              uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(cluster_bar)
      : "memory");
}

MOE_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

MOE_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---- tcgen05 / TMEM ------------------------------------------------------------------

// Whole warp: allocate `ncols` TMEM columns (power of two >= 32); the TMEM address is
// written to shared memory at `dst`.
MOE_DEV void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

MOE_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

MOE_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

MOE_DEV void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row swizzle atoms of 1024 bytes stacked along
// M/N (stride byte offset 1024).  The leading byte offset is unused for this layout.
// Bits: [0,14) start >> 4, [16,30) LBO >> 4, [32,46) SBO >> 4, [46,48) version 1,
// [61,64) layout 2 = 128-byte swizzle.  The tile must start on a 1024-byte boundary;
// K steps inside the 128-byte row advance the start address.
MOE_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

// Instruction descriptor for a dense MMA with FP32 accumulation, both operands K-major.
// a_fmt/b_fmt: kind::f8f6f4 E4M3 = 0; kind::f16 BF16 = 1.
// Bits: [4,6) D format (1 = F32), [7,10) A format, [10,13) B format, [15] A major,
// [16] B major, [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, uint32_t a_fmt, uint32_t b_fmt) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// One tcgen05 MMA, issued by a single thread: D[tmem] (+)= A[smem] . B[smem]^T.
MOE_DEV void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

MOE_DEV void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                      uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every MMA issued so far by this thread has completed.
MOE_DEV void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Warp-wide: 32 lanes x 32 consecutive FP32 columns from TMEM (lane window set by the
// warp's rank within its warpgroup).
MOE_DEV void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Warp-wide: 32 lanes x 16 consecutive FP32 columns.
MOE_DEV void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

MOE_DEV void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Named barrier over `nthreads` threads (id 1..15; 0 is __syncthreads), whole warps,
// returning the OR of every participating thread's `v`.  A hardware barrier: it does not
// touch shared memory.  It cannot time out, so the participants must execute it the same
// number of times by construction.
MOE_DEV bool named_bar_sync_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ---- number formats ------------------------------------------------------------------

// Two FP32 values -> two E4M3 bytes (round to nearest even, saturate to +-448, NaN ->
// 0x7F); `lo` lands in the low byte.
MOE_DEV uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

MOE_DEV float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// 32-byte global store (sm_100+); the address must be 32-byte aligned.
MOE_DEV void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                          uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

MOE_DEV uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The scale of a 1x128 / 128x128 group: amax / 448, correctly rounded; 1 for amax 0.
MOE_DEV float e4m3_scale_from_amax(float amax) {
  return amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
}

// Power-of-two scale rule (the MX-native variant and the 128x1 backward tiles): the
// smallest s = 2^k with 448 * s >= amax, found exactly from amax's exponent and mantissa
// (448 = 1.75 * 2^8), at least 2^-126; s = 1 for amax == 0.  Division by it is exact.
MOE_DEV float pow2_scale_from_amax(float amax) {
  if (amax == 0.0f) return 1.0f;
  uint32_t b = __float_as_uint(amax);
  int e = static_cast<int>((b >> 23) & 0xFFu) - 127;
  if (((b >> 23) & 0xFFu) == 0) {                         // subnormal amax: rescale exactly
    b = __float_as_uint(amax * 18446744073709551616.0f);  // * 2^64
    e = static_cast<int>((b >> 23) & 0xFFu) - 127 - 64;
  }
  const int k = max(e - 8 + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0), -126);
  return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

}  // namespace moe
