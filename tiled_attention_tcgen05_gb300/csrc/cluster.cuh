// Device helpers for thread-block clusters on sm_103a, written from the
// public PTX ISA description of these instructions.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace ta {

// Thread-block clusters: rank of this CTA, a barrier over every thread of the
// cluster (like __syncthreads; the cluster's CTAs are co-scheduled, so it
// completes once every thread reaches it), shared-memory addresses of a peer
// CTA, loads from them, and arrivals on a peer's mbarrier.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// This CTA's shared address `addr` -> the same offset in CTA `rank`'s shared
// memory, as a shared::cluster address.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float4 ld_cluster_v4(uint32_t caddr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(caddr)
               : "memory");
  return v;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t caddr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(caddr) : "memory");
  return v;
}

// Arrive on an mbarrier in another CTA of the cluster, releasing this
// thread's earlier shared-memory writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

// mbar_wait for a barrier that a peer CTA arrives on: the completed phase
// acquires at cluster scope (the peer's released writes become visible).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, const WaitCtl& ctl,
                                                  uint32_t code) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity), "r"(kSuspendNs)
        : "memory");
    if (ok) return true;
    if (*ctl.abort) return false;
    if (globaltimer_ns() - t0 > ctl.timeout_ns) {
      if (ctl.err) atomicOr(ctl.err, code);
      *ctl.abort = 1;
      return false;
    }
  }
}

}  // namespace ta
