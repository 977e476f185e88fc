// Guard checks: device-side checks of the kernels' index arithmetic and of
// the operands they hand the TMA and tensor-core instructions, compiled in
// only when TA_GUARD is defined (the test build libtattn_guard.so).  A check
// that fails records kErrGuard and its source line in its translation unit's
// guard word, and the checked access is skipped, so a broken invariant
// shows up as a status (TA_ERR_GUARD from ta_sync_status) instead of a
// fault.  In the product build TA_CHECK is the constant true and no code is
// generated for it.
//
// What is checked, and where:
//  - TMA loads (tma_load_3d): the shared-memory destination lies in the
//    block's dynamic shared memory on a 1024-byte boundary (the 128-byte
//    swizzle's atom); the innermost coordinate is a multiple of 16 elements
//    and no coordinate is negative.
//  - TMEM loads and stores: the lane field is the calling warp's quadrant
//    (warp % 4) and the columns stay inside the 512 allocated.
//  - MMA batches: the accumulator's and a TMEM operand's columns lie inside
//    the allocation with lane 0; every shared-memory descriptor starts inside
//    the dynamic shared memory.
//  - Global stores through the row-store helpers: 16-byte alignment; the
//    kernels check each stored row and column against the problem's extents.
//  - Work decode: every CTA's (head, tile) lies inside the grid's problem.
#pragma once
#include <cstdint>

namespace ta {

constexpr uint32_t kErrGuard = 1u << 5;

#ifdef TA_GUARD
constexpr bool kGuardBuild = true;

// [0]: kErrGuard once a check has failed; of the first failure: [1] its
// source line, [2] the value it rejected (0 where the check has none), [3]
// the block's dynamic shared memory base and [4] its size.  One copy per
// translation unit (each unit is its own device module); the unit's
// TA_GUARD_ACCESSOR reads and clears it from the host.
static __device__ uint32_t g_guard_word[5];

extern __shared__ uint8_t ta_guard_dyn_smem[];  // aliases every kernel's dynamic shared memory

static __device__ __noinline__ void guard_fail(uint32_t line, uint32_t value) {
  atomicOr(&g_guard_word[0], kErrGuard);
  if (atomicCAS(&g_guard_word[1], 0u, line) == 0u) {
    uint32_t size;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
    g_guard_word[2] = value;
    g_guard_word[3] = static_cast<uint32_t>(__cvta_generic_to_shared(ta_guard_dyn_smem));
    g_guard_word[4] = size;
  }
}

#define TA_CHECK(cond) (__builtin_expect(!!(cond), 1) || (::ta::guard_fail(__LINE__, 0u), false))
// The same, recording `value` (an address or index the check rejected).
#define TA_CHECK_V(cond, value) \
  (__builtin_expect(!!(cond), 1) || (::ta::guard_fail(__LINE__, static_cast<uint32_t>(value)), false))

__device__ __forceinline__ bool guard_in_dyn_smem(uint32_t saddr) {
  uint32_t size;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(size));
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(ta_guard_dyn_smem));
  return saddr >= base && saddr < base + size;
}

// TMEM address: lane in bits 16..31, column in bits 0..15.
__device__ __forceinline__ bool guard_tmem_cols(uint32_t taddr, uint32_t ncols) {
  return (taddr & 0xFFFFu) + ncols <= 512u;
}

__device__ __forceinline__ bool guard_tmem_warp(uint32_t taddr, uint32_t ncols) {
  const uint32_t warp = threadIdx.x >> 5;
  return ((taddr >> 16) >> 5) == (warp & 3u) && guard_tmem_cols(taddr, ncols);
}

// Start address field (bits 0..13, in 16-byte units) of a shared-memory
// descriptor: the low 18 bits of the operand's shared address.  In a cluster
// launch the block's shared addresses carry bits above those (the window's
// place in the cluster's), so the full address is the window's upper bits
// with the field below them (a block's window never crosses a 256 KB
// boundary).
__device__ __forceinline__ bool guard_sdesc(uint64_t desc) {
  const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(ta_guard_dyn_smem));
  return guard_in_dyn_smem((base & ~0x3FFFFu) | (static_cast<uint32_t>(desc & 0x3FFFu) << 4));
}
#else
constexpr bool kGuardBuild = false;
#define TA_CHECK(cond) true
#define TA_CHECK_V(cond, value) true
#endif

}  // namespace ta

// Host accessor of a translation unit's guard word (guard build only):
// returns the failure bits and copies words [1..4] (line, value, shared
// memory base and size of the first failure) to info, clearing them all.
#ifdef TA_GUARD
#define TA_GUARD_ACCESSOR(NAME)                                                       \
  namespace ta {                                                                      \
  uint32_t guard_take_##NAME(uint32_t* info) {                                        \
    uint32_t w[5] = {0u, 0u, 0u, 0u, 0u};                                             \
    if (cudaMemcpyFromSymbol(w, g_guard_word, sizeof(w)) != cudaSuccess) return 0u;  \
    if (w[0] != 0u) {                                                                 \
      const uint32_t z[5] = {0u, 0u, 0u, 0u, 0u};                                     \
      cudaMemcpyToSymbol(g_guard_word, z, sizeof(z));                                 \
    }                                                                                 \
    for (int i = 0; i < 4; ++i) info[i] = w[i + 1];                                   \
    return w[0];                                                                      \
  }                                                                                   \
  }
#else
#define TA_GUARD_ACCESSOR(NAME)
#endif
