// attn_bwd_noalloc: the attention backward for callers that cannot hand the
// library a workspace.
//
// attn_bwd needs scratch memory for delta = rowsum(dO o O) (one float per
// query row), which it expects in a caller-provided buffer.  Some callers
// cannot provide one: a host framework that has reserved all device memory
// for its own pool and does not expose an allocator to plug-ins, or a step
// loop that must not call cudaMalloc because the call synchronises the
// device and its latency is unbounded.  This entry point keeps that scratch
// in a fixed-size array that lives in this library's device image instead, so
// the call itself allocates nothing.
#include <mutex>

#include "tattn.h"
#include "common.cuh"

namespace ta {

// Room for delta of up to kNoAllocRows query rows (B * H * M), 8 MiB.  Every
// GPU that loads the library holds this array until the process exits.
constexpr long long kNoAllocRows = 1ll << 21;
static __device__ __align__(256) float g_noalloc_delta[kNoAllocRows];

// Device address of g_noalloc_delta for the current device.  In host code the
// array's name only stands in for the symbol, so the address is looked up once
// per device (with that device current) and cached.
static ta_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || p == nullptr) return TA_ERR_CUDA;
    cache[dev] = p;
  }
  *out = cache[dev];
  return TA_OK;
}

}  // namespace ta

extern "C" ta_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dO, void* dq, void* dk, void* dv, int B,
                                      int H, int M, int N, int D, ta_dtype dt, int causal, float sm_scale,
                                      void* stream) {
  if (B < 0 || H < 0 || M < 0) return TA_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H * M > ta::kNoAllocRows) return TA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  const ta_status st = ta::noalloc_scratch(&scratch);
  if (st != TA_OK) return st;
  return attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, static_cast<size_t>(ta::kNoAllocRows) * sizeof(float),
                  B, H, M, N, D, dt, causal, sm_scale, stream);
}
