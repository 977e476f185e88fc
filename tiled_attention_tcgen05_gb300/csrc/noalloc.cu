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
// the call itself allocates nothing.  It runs the two-pass backward (dK/dV
// pass, then dQ pass), whose only scratch is delta; attn_bwd's fused pass
// would also need an fp32 dQ accumulator of B*H*M*D floats.
#include <climits>
#include <mutex>

#include "tattn.h"
#include "common.cuh"
#include "launch.h"

namespace ta {

// Room for delta of up to kNoAllocRows query rows (B * H * M), 8 MiB.  Every
// GPU that loads the library holds this array until the process exits.
constexpr long long kNoAllocRows = 1ll << 21;
static __device__ __align__(256) float g_noalloc_delta[kNoAllocRows];

typedef CUresult (*NaCtxGetCurrentFn)(CUcontext*);

// The calling thread's current context (null when it has none or the driver
// entry point is unavailable).
static CUcontext current_context() {
  static NaCtxGetCurrentFn get = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get = reinterpret_cast<NaCtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (get && get(&c) != CUDA_SUCCESS) c = nullptr;
  return c;
}

// Device address of g_noalloc_delta for the current device.  In host code the
// array's name only stands in for the symbol, so the address is looked up
// with the device current and cached per device, together with the context
// it was looked up in: after cudaDeviceReset (or under another context) the
// module is loaded afresh and the next call looks the address up again.
static ta_status noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* cache[kMaxDevices] = {};
  static CUcontext cache_ctx[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(mu);
  const CUcontext ctx = current_context();
  if (!cache[dev] || ctx == nullptr || ctx != cache_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || p == nullptr) return TA_ERR_CUDA;
    cache[dev] = p;
    cache_ctx[dev] = current_context();  // the lookup binds a context if the thread had none
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
  const long long BH = static_cast<long long>(B) * H;  // < 2^62: no overflow
  if (BH > INT_MAX) return TA_ERR_INVALID_ARG;
  if (BH * M > ta::kNoAllocRows) return TA_ERR_UNSUPPORTED;  // BH * M < 2^62
  void* scratch = nullptr;
  const ta_status st = ta::noalloc_scratch(&scratch);
  if (st != TA_OK) return st;
  return ta::bwd_entry(false, q, k, v, o, lse, dO, dq, dk, dv, scratch,
                       static_cast<size_t>(ta::kNoAllocRows) * sizeof(float), B, H, M, N, D, dt, causal, sm_scale,
                       stream);
}
