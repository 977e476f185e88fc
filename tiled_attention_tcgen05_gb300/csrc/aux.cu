// Memory-bound helper kernels: the backward preprocess delta = rowsum(dO o O)
// ("Triton fused attention tutorial, updated with JVP support",
// _attn_bwd_preprocess; "FlagAttention piecewise.py", _bwd_preprocess), the
// fill for rows that see no key (piecewise _fwd_kernel, empty lines: O = 0,
// L = -inf) and a zero fill.
#include "common.cuh"
#include "launch.h"

namespace ta {

// One group of D/8 threads per row; each thread reads 16 bytes of O and of
// dO (8 elements), so a warp reads whole 128-byte lines of both tensors.
template <typename T, int D>
__global__ void __launch_bounds__(256) delta_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dO,
                                                    float* __restrict__ delta, long long rows) {
  constexpr int G = D / 8;  // threads per row
  constexpr int RPB = 256 / G;
  const int g = threadIdx.x % G;
  const long long stride = static_cast<long long>(gridDim.x) * RPB;
  // Block-uniform loop bound: the butterfly always runs with the whole warp.
  for (long long rb = static_cast<long long>(blockIdx.x) * RPB; rb < rows; rb += stride) {
    const long long row = rb + threadIdx.x / G;
    const bool act = row < rows;
    float acc = 0.f;
    if (act) {
      const uint4 a = __ldg(o + row * G + g);
      const uint4 b = __ldg(dO + row * G + g);
      const T* ap = reinterpret_cast<const T*>(&a);
      const T* bp = reinterpret_cast<const T*>(&b);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(static_cast<float>(ap[i]), static_cast<float>(bp[i]), acc);
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (act && g == 0) delta[row] = acc;
  }
}

static int sm_count() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

cudaError_t launch_delta(bool bf16, int D, const void* o, const void* dO, float* delta, long long rows,
                         cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int rpb = 256 / (D / 8);
  long long blocks = (rows + rpb - 1) / rpb;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  const uint4* a = static_cast<const uint4*>(o);
  const uint4* b = static_cast<const uint4*>(dO);
  if (D == 16) {
    if (bf16) delta_kernel<__nv_bfloat16, 16><<<blocks, 256, 0, s>>>(a, b, delta, rows);
    else delta_kernel<__half, 16><<<blocks, 256, 0, s>>>(a, b, delta, rows);
  } else if (D == 32) {
    if (bf16) delta_kernel<__nv_bfloat16, 32><<<blocks, 256, 0, s>>>(a, b, delta, rows);
    else delta_kernel<__half, 32><<<blocks, 256, 0, s>>>(a, b, delta, rows);
  } else if (D == 64) {
    if (bf16) delta_kernel<__nv_bfloat16, 64><<<blocks, 256, 0, s>>>(a, b, delta, rows);
    else delta_kernel<__half, 64><<<blocks, 256, 0, s>>>(a, b, delta, rows);
  } else if (D == 128) {
    if (bf16) delta_kernel<__nv_bfloat16, 128><<<blocks, 256, 0, s>>>(a, b, delta, rows);
    else delta_kernel<__half, 128><<<blocks, 256, 0, s>>>(a, b, delta, rows);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

__global__ void empty_rows_kernel(uint4* o, float* lse, uint4* to, long long rows, int vec_per_row) {
  const long long n = rows * vec_per_row;
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n; i += 256ll * gridDim.x) {
    o[i] = make_uint4(0, 0, 0, 0);
    if (to) to[i] = make_uint4(0, 0, 0, 0);
  }
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < rows; i += 256ll * gridDim.x) lse[i] = -INFINITY;
}

cudaError_t launch_empty_rows(int esize, int D, void* o, float* lse, void* to, long long rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int vpr = D * esize / 16;
  long long blocks = (rows * vpr + 255) / 256;
  if (blocks > sm_count() * 8) blocks = sm_count() * 8;
  empty_rows_kernel<<<blocks, 256, 0, s>>>(static_cast<uint4*>(o), lse, static_cast<uint4*>(to), rows, vpr);
  return cudaGetLastError();
}

__global__ void zero_kernel(uint4* p, long long nvec) {
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < nvec; i += 256ll * gridDim.x) p[i] = make_uint4(0, 0, 0, 0);
}

cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s) {
  const long long nvec = static_cast<long long>(bytes / 16);
  if (nvec <= 0) return cudaSuccess;
  long long blocks = (nvec + 255) / 256;
  if (blocks > sm_count() * 8) blocks = sm_count() * 8;
  zero_kernel<<<blocks, 256, 0, s>>>(static_cast<uint4*>(p), nvec);
  return cudaGetLastError();
}

}  // namespace ta
