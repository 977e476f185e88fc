// Epilogue helpers shared by the backward kernels: fp32 accumulator rows
// read from TMEM, scaled, rounded to the 16-bit element type and stored.
#pragma once
#include "common.cuh"
#include "tmem_ldst.cuh"

namespace ta {

// Stores the first 8 * ng (ng <= 4) of 32 fp32 values (x scale) as T.
template <typename T>
__device__ __forceinline__ void store_chunk32(T* dst, const uint32_t* v, float scale, int ng) {
  constexpr bool BF = DT<T>::bf16;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack2<BF>(__uint_as_float(v[8 * q + 0]) * scale, __uint_as_float(v[8 * q + 1]) * scale);
    u.y = pack2<BF>(__uint_as_float(v[8 * q + 2]) * scale, __uint_as_float(v[8 * q + 3]) * scale);
    u.z = pack2<BF>(__uint_as_float(v[8 * q + 4]) * scale, __uint_as_float(v[8 * q + 5]) * scale);
    u.w = pack2<BF>(__uint_as_float(v[8 * q + 6]) * scale, __uint_as_float(v[8 * q + 7]) * scale);
    if (q < ng) d4[q] = u;
  }
}

// Reads columns [c0, c0 + D/2) of a D-column fp32 accumulator row from TMEM
// and stores those below dg (x scale) into the matching half of one row of T
// (dg columns in memory); `touched` false writes zeros.  Warp-collective.
template <typename T, int D>
__device__ __forceinline__ void epilogue_half(uint32_t taddr, T* row, int c0, bool store, bool touched,
                                              float scale, int dg) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t v[32];
    tmem_ld_x32(taddr + c0 + 32 * c, v);
    tmem_ld_wait(v);
    if (store) store_chunk32<T>(row + c0 + 32 * c, v, touched ? scale : 0.f, chunk_groups(dg, c0 + 32 * c));
  }
}

template <typename T, int D>
__device__ __forceinline__ void zero_half(T* row, int c0, int dg) {
  uint32_t z[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) z[e] = 0;
#pragma unroll
  for (int c = 0; c < D / 64; ++c) store_chunk32<T>(row + c0 + 32 * c, z, 0.f, chunk_groups(dg, c0 + 32 * c));
}

#define TB_CHUNK(arr, c) (*reinterpret_cast<uint32_t(*)[32]>(&(arr)[32 * (c)]))
#define TB_CHUNK16(arr, c) (*reinterpret_cast<uint32_t(*)[16]>(&(arr)[16 * (c)]))

}  // namespace ta
