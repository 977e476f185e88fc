// Merge of two partial attention states over disjoint key sets (split-KV or
// context-parallel combine), forward and backward, after the
// "backward_phase_2" page (reference_forward and the merge backward kernel):
//   m = max(L1, L2), a = exp(L1 - m), b = exp(L2 - m),
//   alpha = a / (a + b), beta = b / (a + b),
//   O = alpha O1 + beta O2, L = m + ln(a + b);
//   dO1 = alpha dO, dO2 = beta dO, t = sum_d dO (O1 - O2),
//   dL1 = alpha dL + alpha beta t, dL2 = beta dL - alpha beta t.
// A row whose parts both saw no key (L1 = L2 = -inf) gives O = 0, L = -inf and
// zero gradients.
//
// Memory-bound: one group of G = D * sizeof(T) / 16 threads per row, each
// thread moving 16 bytes of every D-wide operand, so a warp touches whole
// 128-byte lines; the backward's row dot product is a butterfly over the
// group.  Arithmetic in fp32 for every element type.
#include "common.cuh"
#include "launch.h"

namespace ta {

template <typename T>
struct Vec16;  // 16 bytes of T as fp32 values
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const void* p, float (&f)[4]) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p));
    f[0] = v.x, f[1] = v.y, f[2] = v.z, f[3] = v.w;
  }
  __device__ static void store(void* p, const float (&f)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(f[0], f[1], f[2], f[3]);
  }
};
template <typename H, bool BF>
struct Vec16Half {
  static constexpr int N = 8;
  __device__ static void load(const void* p, float (&f)[8]) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const H* h = reinterpret_cast<const H*>(&v);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = static_cast<float>(h[i]);
  }
  __device__ static void store(void* p, const float (&f)[8]) {
    uint4 v;
    v.x = pack2<BF>(f[0], f[1]);
    v.y = pack2<BF>(f[2], f[3]);
    v.z = pack2<BF>(f[4], f[5]);
    v.w = pack2<BF>(f[6], f[7]);
    *reinterpret_cast<uint4*>(p) = v;
  }
};
template <>
struct Vec16<__half> : Vec16Half<__half, false> {};
template <>
struct Vec16<__nv_bfloat16> : Vec16Half<__nv_bfloat16, true> {};

// alpha, beta, merged L of one row.
__device__ __forceinline__ void merge_weights(float l1, float l2, float& alpha, float& beta, float& L) {
  const float m = fmaxf(l1, l2);
  if (m == -INFINITY) {
    alpha = beta = 0.f;
    L = -INFINITY;
    return;
  }
  const float a = expf(l1 - m), b = expf(l2 - m);
  const float inv = 1.f / (a + b);
  alpha = a * inv;
  beta = b * inv;
  L = m + logf(a + b);
}

template <typename T, int D>
__global__ void __launch_bounds__(256) merge_fwd_kernel(const T* __restrict__ o1, const float* __restrict__ l1,
                                                        const T* __restrict__ o2, const float* __restrict__ l2,
                                                        T* __restrict__ o, float* __restrict__ lse, long long rows) {
  using V = Vec16<T>;
  constexpr int G = D / V::N;  // threads per row
  constexpr int RPB = 256 / G;
  const int g = threadIdx.x % G;
  const long long stride = static_cast<long long>(gridDim.x) * RPB;
  for (long long r = static_cast<long long>(blockIdx.x) * RPB + threadIdx.x / G; r < rows; r += stride) {
    float alpha, beta, L;
    merge_weights(__ldg(l1 + r), __ldg(l2 + r), alpha, beta, L);
    const size_t off = static_cast<size_t>(r) * D + g * V::N;
    float x[V::N], y[V::N];
    V::load(o1 + off, x);
    V::load(o2 + off, y);
#pragma unroll
    for (int i = 0; i < V::N; ++i) x[i] = alpha * x[i] + beta * y[i];
    V::store(o + off, x);
    if (g == 0) lse[r] = L;
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(256) merge_bwd_kernel(const T* __restrict__ o1, const float* __restrict__ l1,
                                                        const T* __restrict__ o2, const float* __restrict__ l2,
                                                        const T* __restrict__ dO, const float* __restrict__ dl,
                                                        T* __restrict__ do1, float* __restrict__ dl1,
                                                        T* __restrict__ do2, float* __restrict__ dl2, long long rows) {
  using V = Vec16<T>;
  constexpr int G = D / V::N;
  constexpr int RPB = 256 / G;
  const int g = threadIdx.x % G;
  const long long stride = static_cast<long long>(gridDim.x) * RPB;
  // The loop bound is the block's first row, the same for every lane, so
  // the butterfly below always runs with the whole warp; rows past the end
  // only skip their loads and stores.
  for (long long rb = static_cast<long long>(blockIdx.x) * RPB; rb < rows; rb += stride) {
    const long long r = rb + threadIdx.x / G;
    const bool act = r < rows;
    float alpha = 0.f, beta = 0.f, L = 0.f;
    float x[V::N] = {}, y[V::N] = {}, d[V::N] = {};
    const size_t off = static_cast<size_t>(act ? r : 0) * D + g * V::N;
    if (act) {
      merge_weights(__ldg(l1 + r), __ldg(l2 + r), alpha, beta, L);
      V::load(o1 + off, x);
      V::load(o2 + off, y);
      V::load(dO + off, d);
    }
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < V::N; ++i) t = fmaf(d[i], x[i] - y[i], t);
#pragma unroll
    for (int sh = G / 2; sh > 0; sh >>= 1) t += __shfl_xor_sync(0xffffffffu, t, sh);
    if (!act) continue;
#pragma unroll
    for (int i = 0; i < V::N; ++i) {
      x[i] = alpha * d[i];
      y[i] = beta * d[i];
    }
    V::store(do1 + off, x);
    V::store(do2 + off, y);
    if (g == 0) {
      const float dlr = dl ? __ldg(dl + r) : 0.f;
      const float ab = alpha * beta * t;
      dl1[r] = alpha * dlr + ab;
      dl2[r] = beta * dlr - ab;
    }
  }
}

// SM count of the current device (cached per device).
static int merge_sm_count() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  std::atomic<int>* n = (dev >= 0 && dev < kMaxDevices) ? &cache[dev] : nullptr;
  int v = n ? n->load(std::memory_order_relaxed) : 0;
  if (v <= 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    if (n) n->store(v, std::memory_order_relaxed);
  }
  return v;
}

template <typename T, int D>
static long long merge_blocks(long long rows) {
  constexpr int RPB = 256 / (D / Vec16<T>::N);
  long long b = (rows + RPB - 1) / RPB;
  const long long cap = static_cast<long long>(merge_sm_count()) * 8;
  return b > cap ? cap : b;
}

template <typename T, int D>
static cudaError_t merge_fwd_t(const MergePtrs& p, long long rows, cudaStream_t s) {
  merge_fwd_kernel<T, D><<<merge_blocks<T, D>(rows), 256, 0, s>>>(
      static_cast<const T*>(p.o1), p.l1, static_cast<const T*>(p.o2), p.l2, static_cast<T*>(p.o), p.lse, rows);
  return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t merge_bwd_t(const MergePtrs& p, long long rows, cudaStream_t s) {
  merge_bwd_kernel<T, D><<<merge_blocks<T, D>(rows), 256, 0, s>>>(
      static_cast<const T*>(p.o1), p.l1, static_cast<const T*>(p.o2), p.l2, static_cast<const T*>(p.dO), p.dl,
      static_cast<T*>(p.do1), p.dl1, static_cast<T*>(p.do2), p.dl2, rows);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t merge_dispatch(bool bwd, int D, const MergePtrs& p, long long rows, cudaStream_t s) {
  switch (D) {
    case 16: return bwd ? merge_bwd_t<T, 16>(p, rows, s) : merge_fwd_t<T, 16>(p, rows, s);
    case 32: return bwd ? merge_bwd_t<T, 32>(p, rows, s) : merge_fwd_t<T, 32>(p, rows, s);
    case 64: return bwd ? merge_bwd_t<T, 64>(p, rows, s) : merge_fwd_t<T, 64>(p, rows, s);
    case 128: return bwd ? merge_bwd_t<T, 128>(p, rows, s) : merge_fwd_t<T, 128>(p, rows, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_merge(bool bwd, int dtype, int D, const MergePtrs& p, long long rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (dtype == 0) return merge_dispatch<__half>(bwd, D, p, rows, s);
  if (dtype == 1) return merge_dispatch<__nv_bfloat16>(bwd, D, p, rows, s);
  return merge_dispatch<float>(bwd, D, p, rows, s);
}

}  // namespace ta

TA_GUARD_ACCESSOR(merge)
