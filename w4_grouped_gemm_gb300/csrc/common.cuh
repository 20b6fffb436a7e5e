// common.cuh -- sm_103a device helpers: mbarriers with bounded waits, TMA,
// tcgen05 (TMEM alloc / MMA / commit / load) and small bit utilities.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lily_internal.h"

namespace lily {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// ------------------------------------------------------------------ mbarrier
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

// try_wait that may suspend the thread in hardware for up to hint_ns while
// the phase is incomplete (no issue slots spent spinning).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  The waiting thread
// sleeps in try_wait (up to 100 us per attempt); the wait gives up after
// kWaitLimitNs of wall time, or early when *abort is set by another role of
// the same CTA; on giving up it sets *abort and the TIMEOUT status bit and
// returns false.  Never traps, never spins forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kSleepHintNs = 100000u;        // 100 us
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      set_status(status, LILY_STATUS_TIMEOUT);
      return false;
    }
  }
}

// Wait by lane 0 only, result broadcast: keeps every warp-collective op
// (tcgen05.ld, __syncwarp, shuffles) convergent even when a wait gives up.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status) {
  int ok = 1;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait run by every lane of a converged warp: all lanes poll
// test_wait and a vote keeps the outcome warp-uniform, so the warp stays
// converged without a divergent lane-0 loop and a broadcast.  Used by the
// warp that issues MMAs, where every synchronising instruction waits for
// the MMAs already issued to drain, so the fewer the better.  Same limits and
// abort protocol as mbar_wait.
__device__ __forceinline__ bool warp_wait_all(uint32_t bar, uint32_t parity, volatile int* abort,
                                              uint32_t* status) {
  if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, parity))) return true;
    if ((n & 255u) == 0) {
      if (__any_sync(0xffffffffu, *abort != 0)) return false;
      if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitLimitNs)) {
        if ((threadIdx.x & 31) == 0) {
          *abort = 1;
          set_status(status, LILY_STATUS_TIMEOUT);
        }
        return false;
      }
    }
  }
}

// Both phases (bar0, parity0) and (bar1, parity1), or only the first when
// !need1: one converged poll and one vote per attempt (see warp_wait_all).
__device__ __forceinline__ bool warp_wait_all2(uint32_t bar0, uint32_t parity0, uint32_t bar1,
                                               uint32_t parity1, bool need1, volatile int* abort,
                                               uint32_t* status) {
  auto ready = [&]() {
    return mbar_test_wait(bar0, parity0) && (!need1 || mbar_test_wait(bar1, parity1));
  };
  if (__all_sync(0xffffffffu, ready())) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (__all_sync(0xffffffffu, ready())) return true;
    if ((n & 255u) == 0) {
      if (__any_sync(0xffffffffu, *abort != 0)) return false;
      if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitLimitNs)) {
        if ((threadIdx.x & 31) == 0) {
          *abort = 1;
          set_status(status, LILY_STATUS_TIMEOUT);
        }
        return false;
      }
    }
  }
}

// The same two-phase wait with mbarrier.try_wait, which suspends the
// waiting threads instead of polling: for warps whose waits should leave the
// issue slots of their SM sub-partition to other warps.
__device__ __forceinline__ bool warp_wait_all2_blocking(uint32_t bar0, uint32_t parity0,
                                                        uint32_t bar1, uint32_t parity1,
                                                        bool need1, volatile int* abort,
                                                        uint32_t* status) {
  auto ready = [&]() {
    return mbar_try_wait(bar0, parity0) && (!need1 || mbar_try_wait(bar1, parity1));
  };
  if (__all_sync(0xffffffffu, ready())) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (__all_sync(0xffffffffu, ready())) return true;
    if ((n & 7u) == 0) {
      if (__any_sync(0xffffffffu, *abort != 0)) return false;
      if (__any_sync(0xffffffffu, globaltimer_ns() - t0 > kWaitLimitNs)) {
        if ((threadIdx.x & 31) == 0) {
          *abort = 1;
          set_status(status, LILY_STATUS_TIMEOUT);
        }
        return false;
      }
    }
  }
}

// One lane of the converged warp (elect.sync): the producer issues a whole
// K-step's expect-tx and TMA copies from it in one branch, which measured
// faster than one election per copy.
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "elect.sync _|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(e));
  return e != 0;
}

// ------------------------------------------------------------------ dependent launch
// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor in the
// stream still runs.  pdl_wait() returns once the predecessor has completed
// and its memory is visible (immediately when there is no such predecessor);
// loads of data the predecessor does not write (weights) may go before it.
// pdl_trigger() lets this kernel's own dependent start; it is called after
// pdl_wait(), so a dependent never overlaps anything older than its direct
// predecessor.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier `id` (1..15) over the first `n` threads of the CTA (a multiple of 32).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ------------------------------------------------------------------ proxies
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int32_t c0,
                                            int32_t c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// Shared memory -> global through a 2-D tensor map (bulk group of this
// thread), and the waits on this thread's bulk groups: until their reads of
// shared memory are done (the buffer may be rewritten), or fully written.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* tm, int32_t c0, int32_t c1,
                                             uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tm),
      "r"(c0), "r"(c1), "r"(src)
      : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int32_t c0,
                                            int32_t c1, int32_t c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tm), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// Plain bulk copy (no tensor map) of `bytes` (a multiple of 16; both
// addresses 16-byte aligned) from global to this CTA's shared memory,
// completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Bring `bytes` (a multiple of 16; 16-byte aligned address) of global memory
// into L2 without waiting for it.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tm) : "memory");
}

// ------------------------------------------------------------------ tcgen05
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

// Shared-memory matrix descriptor, K-major operand with 128-byte swizzle:
// rows of 128 B, 8-row atoms of 1024 B (stride byte offset), version 1.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);  // start address
  d |= (uint64_t)1u << 16;                   // leading byte offset (unused, 16 B)
  d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset
  d |= (uint64_t)1u << 46;                   // descriptor version
  d |= (uint64_t)2u << 61;                   // SWIZZLE_128B
  return d;
}

// Instruction descriptor: kind::f16 with A = B = bf16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor: kind::f16 with A = B = fp16, D = f32, both K-major.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]^T: A (128 rows = TMEM lanes, K packed two
// 16-bit elements per 32-bit column) is read from tensor memory.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-collective commit: every lane of a converged warp executes it and one
// elected lane issues it (for single commits outside the per-step issue
// branches, which use elect_one()).
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          bar)
      : "memory");
}

// Arrive on an mbarrier once all earlier tcgen05 ops of this thread finish.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns (as tmem_ld32, half the width).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
// 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (warp quadrant * 32 + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Store 32 / 16 consecutive 32-bit columns of this thread's TMEM lane
// (32x32b shape: warp w writes lanes 32*(w%4) .. +31).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// The same wait, tied to the source registers of the stores it waits for,
// so that they stay unused until the stores have completed.
__device__ __forceinline__ void tmem_st_wait_regs(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::st.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]),
                 "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                 "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
                 "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                 "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// The same wait, tied to the destination registers of the loads it waits
// for ("+r"), so that no use of them can be scheduled above it while further
// loads are in flight into other registers.
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]),
                 "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[8], uint32_t (&q)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]),
                 "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(q[0]), "+r"(q[1]), "+r"(q[2]), "+r"(q[3]),
                 "+r"(q[4]), "+r"(q[5]), "+r"(q[6]), "+r"(q[7])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t (&r)[16], uint32_t (&q)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]),
                 "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                 "+r"(q[0]), "+r"(q[1]), "+r"(q[2]), "+r"(q[3]),
                 "+r"(q[4]), "+r"(q[5]), "+r"(q[6]), "+r"(q[7]),
                 "+r"(q[8]), "+r"(q[9]), "+r"(q[10]), "+r"(q[11]),
                 "+r"(q[12]), "+r"(q[13]), "+r"(q[14]), "+r"(q[15])
               :
               : "memory");
}

// ------------------------------------------------------------------ bits
// f16x2 helpers on raw 32-bit words (low half = first element).
__device__ __forceinline__ uint32_t h2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t h2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  // (a & mask) | orv in one LOP3 (immLut 0xEA = (a & b) | c)
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
  return d;
}
// bf16 bit pattern -> fp16 bit pattern (round to nearest; exact for
// magnitudes in [2^-17, 65504], the range of group scales and biases).
__device__ __forceinline__ uint16_t bf16_to_f16_bits(uint16_t b) {
  return __half_as_ushort(__float2half_rn(__uint_as_float((uint32_t)b << 16)));
}

// Eight 4-bit codes (one 32-bit word, element i in bits 4i..4i+3) times one
// fp16 scale plus one fp16 bias, as 8 fp16 in the "pair-interleaved" chunk
// order (q0, q4, q1, q5, q2, q6, q3, q7) -- the order in which one LOP3 per
// pair extracts them.  The other GEMM operand stores every 8-element K chunk
// in the same order (kchunk_pos), so the dot products are unchanged.  Each
// weight is round_fp16(scale * q + bias).  A code in bits 0..3 of a 16-bit
// half OR-ed into fp16 1024 (0x6400, unit spacing) reads as 1024 + q; a code
// in bits 4..7 OR-ed into fp16 64 (0x5400, spacing 1/16) reads as 64 + q, so
// two of the four pairs need no shift.  Both sums and the subtractions are
// exact; the f16x2 FMA rounds once.
__device__ __forceinline__ void dequant8(uint32_t w, uint32_t s2, uint32_t b2, uint32_t (&o)[4]) {
  const uint32_t kMagicLo = 0x64006400u;  // fp16 pair (1024, 1024)
  const uint32_t kMagicHi = 0x54005400u;  // fp16 pair (64, 64)
  const uint32_t kMaskLo = 0x000F000Fu, kMaskHi = 0x00F000F0u;
  const uint32_t w8 = w >> 8;
  o[0] = h2_fma(s2, h2_sub(lop3_and_or(w, kMaskLo, kMagicLo), kMagicLo), b2);   // (q0, q4)
  o[1] = h2_fma(s2, h2_sub(lop3_and_or(w, kMaskHi, kMagicHi), kMagicHi), b2);   // (q1, q5)
  o[2] = h2_fma(s2, h2_sub(lop3_and_or(w8, kMaskLo, kMagicLo), kMagicLo), b2);  // (q2, q6)
  o[3] = h2_fma(s2, h2_sub(lop3_and_or(w8, kMaskHi, kMagicHi), kMagicHi), b2);  // (q3, q7)
}
// Position of element e (0..7) of an 8-element K chunk in that order.
__host__ __device__ __forceinline__ int kchunk_pos(int e) { return ((e & 3) << 1) | (e >> 2); }

// 8 bf16 (one 16-byte chunk of a row of x) -> 8 fp16 in the grouped GEMM's
// K-chunk order (element e at position kchunk_pos(e)).
__device__ __forceinline__ uint4 bf8_to_h8_kchunk(uint4 v, bool& ok) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float f[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    f[2 * j] = __uint_as_float(w[j] << 16);
    f[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
  }
  uint16_t h[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ok &= fabsf(f[e]) <= 65504.f;
    h[kchunk_pos(e)] = __half_as_ushort(__float2half_rn(f[e]));
  }
  uint4 o;
  o.x = h[0] | ((uint32_t)h[1] << 16);
  o.y = h[2] | ((uint32_t)h[3] << 16);
  o.z = h[4] | ((uint32_t)h[5] << 16);
  o.w = h[6] | ((uint32_t)h[7] << 16);
  return o;
}

}  // namespace lily
