// Inline-PTX device primitives for sm_103a: mbarriers with bounded waits, TMA
// tensor loads, tcgen05 (TMEM allocation, MMA, commit, fences) and the shared
// memory / instruction descriptors the MMAs consume.  Written from the public
// PTX ISA description of these instructions.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "tmem_ldst.cuh"

namespace ta {

// ------------------------------------------------------------------ errors
// Bits of the device error word that kernels set instead of trapping.
enum : uint32_t {
  kErrTimeoutTma = 1u << 0,    // a wait for TMA data ran out
  kErrTimeoutMma = 1u << 1,    // a wait for an MMA result ran out
  kErrTimeoutSoftmax = 1u << 2,  // a wait for softmax/producer output ran out
  kErrTimeoutOther = 1u << 3,
  kErrSmemLayout = 1u << 4,    // a kernel could not lay out its shared memory (did not run)
};

struct WaitCtl {
  uint32_t* err;         // global error word (nullable)
  uint64_t timeout_ns;   // per-wait limit
  volatile int* abort;   // CTA-wide abort flag in shared memory
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// try_wait with a suspend-time hint: a thread whose phase is not complete
// sleeps in hardware until the phase completes (or ~kSuspendNs passes)
// instead of spinning, so idle waiters do not take issue slots or shared
// memory bandwidth from the MMA issuer and the tensor core.
constexpr uint32_t kSuspendNs = 1000000;  // 1 ms

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Never
// spins forever: after ctl.timeout_ns (or once another role of the CTA set
// the abort flag) it records `code` in the error word, raises the abort flag
// and returns false, so the caller can unwind without trapping.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                          uint32_t code) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (*ctl.abort) return false;
    if (globaltimer_ns() - t0 > ctl.timeout_ns) {
      if (ctl.err) atomicOr(ctl.err, code);
      *ctl.abort = 1;
      return false;
    }
  }
}

// The same wait taken by all 32 lanes of a warp, with a warp-uniform result,
// for waits that guard warp-collective (.sync.aligned) tcgen05 instructions.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl, uint32_t code) {
  const bool ok = mbar_wait(bar, parity, ctl, code);
  return __all_sync(0xffffffffu, ok);
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is counted in
// bytes on `bar`.  Coordinates are element indices (innermost first).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2) {
  if (!TA_CHECK_V((smem_u32(dst) & 1023u) == 0u && guard_in_dyn_smem(smem_u32(dst)) && (c0 & 15) == 0 && c1 >= 0 &&
                      c2 >= 0,
                  smem_u32(dst)))
    return;
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// 3-D tiled store of one box from shared memory (in the map's swizzled
// layout) to global memory, tracked as a bulk async-group of this thread.
// Parts of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  if (!TA_CHECK_V((smem_u32(src) & 1023u) == 0u && guard_in_dyn_smem(smem_u32(src)) && (c0 & 15) == 0 && c1 >= 0 &&
                      c2 >= 0,
                  smem_u32(src)))
    return;
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// Closes this thread's pending bulk stores into one group, then waits until
// every group has finished reading its shared-memory source (the source may
// then be reused or freed; the global writes complete asynchronously).
__device__ __forceinline__ void tma_store_commit_and_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\n cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// 16-byte store to a shared-memory address.
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Barrier over `count` threads (a multiple of 32) on hardware barrier `id`
// (1..15; 0 is __syncthreads').
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// 32-bit store to a shared-memory address.
__device__ __forceinline__ void sts_b32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Generic-proxy writes to shared memory -> visible to the async proxy (MMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// D(tmem) = A(smem) * B(smem) (+ D if accumulate).
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D(tmem) = A(tmem) * B(smem) (+ D if accumulate).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// ------------------------------------------------- batched MMA issue
// N MMAs of one K-loop issued from ONE asm block by the elected lane of a
// fully converged warp (every lane executes the call; elect.sync picks one).
// The first MMA accumulates iff `acc` != 0, the rest always do.  Issuing a
// whole K-loop this way keeps the issuing thread's instruction stream to the
// MMAs themselves, which lets the tensor core run back to back; separate asm
// statements per MMA from a single divergent lane issue far more slowly.

__device__ __forceinline__ void mma_ss_x2(uint32_t d, const uint64_t (&a)[2], const uint64_t (&b)[2], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %6, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %3, %5, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %4, %5, p1;\n"
      "}\n"
      ::"r"(d), "l"(a[0]), "l"(a[1]), "l"(b[0]), "l"(b[1]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ss_x4(uint32_t d, const uint64_t (&a)[4], const uint64_t (&b)[4], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %10, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %9, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %9, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %9, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %9, p1;\n"
      "}\n"
      ::"r"(d), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ss_x8(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %18, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %9, %17, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %10, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %11, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %12, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %5, %13, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %6, %14, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %7, %15, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %8, %16, %17, p1;\n"
      "}\n"
      ::"r"(d), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts_x2(uint32_t d, const uint32_t (&a)[2], const uint64_t (&b)[2], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %6, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %3, %5, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %4, %5, p1;\n"
      "}\n"
      ::"r"(d), "r"(a[0]), "r"(a[1]), "l"(b[0]), "l"(b[1]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts_x4(uint32_t d, const uint32_t (&a)[4], const uint64_t (&b)[4], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %10, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %9, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %9, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %9, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %9, p1;\n"
      "}\n"
      ::"r"(d), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts_x8(uint32_t d, const uint32_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc,
                                          uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %18, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %9, %17, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %10, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %11, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %12, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %13, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%6], %14, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %15, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%8], %16, %17, p1;\n"
      "}\n"
      ::"r"(d), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ss_f8_x2(uint32_t d, const uint64_t (&a)[2], const uint64_t (&b)[2], uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %6, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %3, %5, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %2, %4, %5, p1;\n"
      "}\n"
      ::"r"(d), "l"(a[0]), "l"(a[1]), "l"(b[0]), "l"(b[1]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ss_f8_x4(uint32_t d, const uint64_t (&a)[4], const uint64_t (&b)[4], uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %10, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %5, %9, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %2, %6, %9, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %7, %9, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %4, %8, %9, p1;\n"
      "}\n"
      ::"r"(d), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ss_f8_x8(uint32_t d, const uint64_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %18, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %9, %17, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %2, %10, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %3, %11, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %4, %12, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %5, %13, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %6, %14, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %7, %15, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %8, %16, %17, p1;\n"
      "}\n"
      ::"r"(d), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts_f8_x2(uint32_t d, const uint32_t (&a)[2], const uint64_t (&b)[2], uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %6, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %3, %5, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%2], %4, %5, p1;\n"
      "}\n"
      ::"r"(d), "r"(a[0]), "r"(a[1]), "l"(b[0]), "l"(b[1]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts_f8_x4(uint32_t d, const uint32_t (&a)[4], const uint64_t (&b)[4], uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %10, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %5, %9, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%2], %6, %9, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%3], %7, %9, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%4], %8, %9, p1;\n"
      "}\n"
      ::"r"(d), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void mma_ts_f8_x8(uint32_t d, const uint32_t (&a)[8], const uint64_t (&b)[8], uint32_t idesc,
                                             uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p0, p1;\n elect.sync _|e, 0xffffffff;\n"
      " setp.ne.b32 p0, %18, 0;\n setp.eq.u32 p1, 1, 1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %9, %17, p0;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%2], %10, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%3], %11, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%4], %12, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%5], %13, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%6], %14, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%7], %15, %17, p1;\n"
      " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%8], %16, %17, p1;\n"
      "}\n"
      ::"r"(d), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(acc)
      : "memory");
}

template <int N>
__device__ __forceinline__ void mma_ss_n(uint32_t d, const uint64_t (&a)[N], const uint64_t (&b)[N], uint32_t idesc,
                                         uint32_t acc) {
  static_assert(N == 2 || N == 4 || N == 8, "batch of 2, 4 or 8");
#ifdef TA_GUARD
  // value: the accumulator address, or 0x80000000 | the first rejected descriptor's address field
  uint32_t bad = (guard_tmem_cols(d, 1) && (d >> 16) == 0u) ? 0u : (d | 1u);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if (!bad && !guard_sdesc(a[i])) bad = 0x80000000u | static_cast<uint32_t>(a[i] & 0x3FFFu);
    if (!bad && !guard_sdesc(b[i])) bad = 0xC0000000u | static_cast<uint32_t>(b[i] & 0x3FFFu);
  }
  if (!TA_CHECK_V(bad == 0u, bad)) return;
#endif
  if constexpr (N == 8) mma_ss_x8(d, a, b, idesc, acc);
  else if constexpr (N == 4) mma_ss_x4(d, a, b, idesc, acc);
  else mma_ss_x2(d, a, b, idesc, acc);
}
template <int N>
__device__ __forceinline__ void mma_ts_n(uint32_t d, const uint32_t (&a)[N], const uint64_t (&b)[N], uint32_t idesc,
                                         uint32_t acc) {
  static_assert(N == 2 || N == 4 || N == 8, "batch of 2, 4 or 8");
#ifdef TA_GUARD
  uint32_t bad = (guard_tmem_cols(d, 1) && (d >> 16) == 0u) ? 0u : (d | 1u);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if (!bad && !(guard_tmem_cols(a[i], 1) && (a[i] >> 16) == 0u)) bad = a[i] | 1u;
    if (!bad && !guard_sdesc(b[i])) bad = 0xC0000000u | static_cast<uint32_t>(b[i] & 0x3FFFu);
  }
  if (!TA_CHECK_V(bad == 0u, bad)) return;
#endif
  if constexpr (N == 8) mma_ts_x8(d, a, b, idesc, acc);
  else if constexpr (N == 4) mma_ts_x4(d, a, b, idesc, acc);
  else mma_ts_x2(d, a, b, idesc, acc);
}
template <int N>
__device__ __forceinline__ void mma_ss_f8_n(uint32_t d, const uint64_t (&a)[N], const uint64_t (&b)[N], uint32_t idesc,
                                            uint32_t acc) {
  static_assert(N == 2 || N == 4 || N == 8, "batch of 2, 4 or 8");
#ifdef TA_GUARD
  // value: the accumulator address, or 0x80000000 | the first rejected descriptor's address field
  uint32_t bad = (guard_tmem_cols(d, 1) && (d >> 16) == 0u) ? 0u : (d | 1u);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if (!bad && !guard_sdesc(a[i])) bad = 0x80000000u | static_cast<uint32_t>(a[i] & 0x3FFFu);
    if (!bad && !guard_sdesc(b[i])) bad = 0xC0000000u | static_cast<uint32_t>(b[i] & 0x3FFFu);
  }
  if (!TA_CHECK_V(bad == 0u, bad)) return;
#endif
  if constexpr (N == 8) mma_ss_f8_x8(d, a, b, idesc, acc);
  else if constexpr (N == 4) mma_ss_f8_x4(d, a, b, idesc, acc);
  else mma_ss_f8_x2(d, a, b, idesc, acc);
}
template <int N>
__device__ __forceinline__ void mma_ts_f8_n(uint32_t d, const uint32_t (&a)[N], const uint64_t (&b)[N],
                                            uint32_t idesc, uint32_t acc) {
  static_assert(N == 2 || N == 4 || N == 8, "batch of 2, 4 or 8");
#ifdef TA_GUARD
  uint32_t bad = (guard_tmem_cols(d, 1) && (d >> 16) == 0u) ? 0u : (d | 1u);
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if (!bad && !(guard_tmem_cols(a[i], 1) && (a[i] >> 16) == 0u)) bad = a[i] | 1u;
    if (!bad && !guard_sdesc(b[i])) bad = 0xC0000000u | static_cast<uint32_t>(b[i] & 0x3FFFu);
  }
  if (!TA_CHECK_V(bad == 0u, bad)) return;
#endif
  if constexpr (N == 8) mma_ts_f8_x8(d, a, b, idesc, acc);
  else if constexpr (N == 4) mma_ts_f8_x4(d, a, b, idesc, acc);
  else mma_ts_f8_x2(d, a, b, idesc, acc);
}

// tcgen05.commit by the elected lane of a fully converged warp.
__device__ __forceinline__ void commit_el(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(smem_u32(bar))
      : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout a TMA load
// with CU_TENSOR_MAP_SWIZZLE_128B produces).  Byte offsets: `lbo` is the
// leading-dimension offset, `sbo` the stride-dimension offset (8-row groups).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16 with fp32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ----------------------------------------------------------------- math
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------ packed fp32
// Two fp32 lanes per instruction (the .f32x2 forms of sm_100 and later).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mov.b64 rc, {%6, %7};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}\n"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// max(a, b, c) in one instruction (three-input form, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16) {
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  } else {
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  }
  return r;
}

}  // namespace ta
