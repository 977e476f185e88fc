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
  if (!TA_CHECK((reinterpret_cast<uintptr_t>(dst) & 15u) == 0u && ng >= 0 && ng <= 4)) return;
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


// ------------------------------------------- TMA and MMA helpers
template <int D>
__device__ __forceinline__ void load_tile_b(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row0, int bh) {
#pragma unroll
  for (int kb = 0; kb < D / 64; ++kb) tma_load_3d(dst + kb * (kBM * 128), map, bar, kb * 64, row0, bh);
}

// d = A B^T over D: A, B are 128-row x D K-major swizzled tiles in smem.
template <int D>
__device__ __forceinline__ void mma_abT(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, uint32_t idesc) {
  const uint64_t da0 = sdesc_sw128(a_smem, 16, 1024);
  const uint64_t db0 = sdesc_sw128(b_smem, 16, 1024);
  uint64_t da[D / 16], db[D / 16];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
    da[kk] = da0 + off;
    db[kk] = db0 + off;
  }
  mma_ss_n<D / 16>(d_tmem, da, db, idesc, 0u);
}

// K-steps of chunk group g (the 32-key / 32-query chunk g of both column
// halves): {2g, 2g + 1, 2g + 4, 2g + 5}.
__device__ __forceinline__ constexpr int chunk_kstep(int g, int i) { return 2 * g + (i & 1) + 4 * (i >> 1); }

// d (+)= X Y over the K-steps of chunk group G only, X with interleaved
// K-steps: step kk at x + (kk / 2) * 32 + (kk % 2) * 8 (16 packed columns in
// each 32-column chunk); Y a 128-row x D tile in smem read as an MN-major B
// operand (rows = K).  Whole converged warp.
template <int G>
__device__ __forceinline__ void mma_tY_il_g(uint32_t d_tmem, uint32_t x_tmem, uint32_t y_smem, uint32_t idesc,
                                            bool accumulate) {
  const uint64_t dy = sdesc_sw128(y_smem, kBM * 128, 1024);
  uint32_t a[4];
  uint64_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int kk = chunk_kstep(G, i);
    a[i] = x_tmem + (kk >> 1) * 32 + (kk & 1) * 8;
    b[i] = dy + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<4>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}

// Copies row r of a 128 x D 16-bit K-major 128-byte-swizzled tile from shared
// memory into TMEM lane r, columns taddr .. taddr + D/2 (two elements per
// column, lower index in the low half): the layout an A operand is read in.
// Warp-collective.
template <int D>
__device__ __forceinline__ void tile_row_to_tmem(const uint8_t* tile, int r, uint32_t taddr) {
#pragma unroll
  for (int kb = 0; kb < D / 64; ++kb) {
    uint32_t v[32];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 c = *reinterpret_cast<const uint4*>(tile + kb * (kBM * 128) + r * 128 + ((j ^ (r & 7)) * 16));
      v[4 * j + 0] = c.x;
      v[4 * j + 1] = c.y;
      v[4 * j + 2] = c.z;
      v[4 * j + 3] = c.w;
    }
    tmem_st_x32(taddr + 32 * kb, v);
  }
}

#define TB_CHUNK(arr, c) (*reinterpret_cast<uint32_t(*)[32]>(&(arr)[32 * (c)]))
#define TB_CHUNK16(arr, c) (*reinterpret_cast<uint32_t(*)[16]>(&(arr)[16 * (c)]))

}  // namespace ta
