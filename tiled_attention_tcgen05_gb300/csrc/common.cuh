// Shared definitions for the attention kernels: problem parameters, tile
// constants and the mode tags.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace ta {

constexpr int kBM = 128;  // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;  // keys per tile
constexpr int kSmemMax = 232448;  // opt-in dynamic shared memory per block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// The running row maximum is only raised (and O rescaled) when a new score
// exceeds it by more than this many powers of two; below that the stale
// maximum is kept, which is exact because O and l share it.
constexpr float kRescaleThreshold = 8.0f;

enum Mode : int { kStd = 0, kPiecewise = 1, kJvp = 2 };

struct FwdArgs {
  void* o;
  float* lse;
  void* to;       // JVP tangent output (kJvp only)
  float* tlse;    // JVP tangent of L (kJvp only; may be null)
  int BH, M, N, P_SEQ;
  int num_q_tiles;
  int causal;
  int w;          // piecewise threshold
  int group_heads;   // heads per group of the two-tile forward's tile order (grouped_tile)
  float scale_log2;  // sm_scale * log2(e)
  float sm_scale;
  int dg;            // head dimension of the tensors in memory (row stride, columns stored)
  uint32_t* err;
  uint64_t timeout_ns;
};

struct BwdArgs {
  void* dq;   // dq  (dq1 in piecewise)
  void* dq2;  // piecewise only
  void* dk;   // dk  (dk1 in piecewise)
  void* dk2;  // piecewise only
  void* dv;
  const float* lse;
  const float* delta;  // backward of the JVP: <dO, O> + <dtO, tO>
  const float* mu;     // backward of the JVP only: tL = rowsum(P o T)
  const float* eps;    // backward of the JVP only: <dtO, O>
  void* dtq;           // backward of the JVP: the tangents' gradients (where TMEM has room)
  void* dtk;
  void* dtv;
  int BH, M, N, P_SEQ;
  int causal;
  int w;
  float scale_log2;
  float sm_scale;
  int dg;  // head dimension of the tensors in memory (row stride, columns stored)
  float* dq_acc;  // fused backward: fp32 dQ accumulator [BH, M, D] (zeroed by the delta pass)
  float* delta_out;  // standard dQ pass: form delta = rowsum(dO o O) from O and store it here
  uint32_t* err;
  uint64_t timeout_ns;
};

// Number of 8-column (16-byte) groups of the 32-column chunk starting at
// column c0 that exist in a row of dg columns (0 to 4).
__host__ __device__ inline int chunk_groups(int dg, int c0) {
  const int n = (dg - c0) >> 3;
  return n < 0 ? 0 : (n > 4 ? 4 : n);
}

// Number of key tiles that query tile [q0, q0 + kBM) visits.
__host__ __device__ inline int kv_tiles_for(int q0, int M, int N, int P_SEQ, int causal) {
  int n_all = (N + kBN - 1) / kBN;
  if (!causal) return n_all;
  int last = q0 + kBM - 1 + P_SEQ;  // largest visible key of the tile
  if (last < 0) return 0;
  if (last > N - 1) last = N - 1;
  return last / kBN + 1;
}

// First query tile that key tile [k0, k0 + kBN) is visible from.
__host__ __device__ inline int first_q_tile_for(int k0, int P_SEQ, int causal) {
  if (!causal) return 0;
  int first_row = k0 - P_SEQ;  // smallest i with k0 <= i + P_SEQ
  if (first_row < 0) first_row = 0;
  return first_row / kBM;
}

// Linear block index -> (head, rank of the tile within its head): heads are
// taken in groups of G (so the resident CTAs of one wave share the K/V or
// Q/dO of only G heads and reuse them through L2), and within a group rank 0
// (the caller's heaviest tile) comes first for every head.
// Returns false (a guard-build check) when the block index decodes outside
// the problem; the caller's CTA then does nothing.
__device__ __forceinline__ bool grouped_tile(int id, int BH, int ntiles, int G, int* bh, int* rank) {
  const int per_group = G * ntiles;
  const int grp = id / per_group;
  const int h0 = grp * G;
  const int gh = min(G, BH - h0);  // heads in this (possibly last, smaller) group
  const int within = id - grp * per_group;
  *rank = within / gh;
  *bh = h0 + within % gh;
  return TA_CHECK(gh > 0 && *bh >= 0 && *bh < BH && *rank >= 0 && *rank < ntiles);
}
constexpr int kGroupHeads = 8;

// Stages 32 fp32 values (x scale, rounded to 16 bits) of row r, columns
// [32 c, 32 c + 32), into a tile laid out as a 128-byte-swizzled TMA box
// sequence: 64-column boxes of 128 rows x 128 bytes, box kb at
// tile + kb * 16 KB, and in row r the 16-byte chunk j at position j ^ (r % 8)
// (the layout CU_TENSOR_MAP_SWIZZLE_128B reads; a warp's 32 rows then spread
// over the eight 16-byte bank groups).  `v` are fp32 bit patterns.
template <bool BF>
__device__ __forceinline__ void stage_row_chunk_sw128(uint32_t tile, int r, int c, const uint32_t* v, float scale) {
  const uint32_t rowp = tile + static_cast<uint32_t>((c >> 1) * (kBM * 128) + r * 128);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int j = 4 * (c & 1) + q;
    const uint32_t* u = v + 8 * q;
    sts_v4(rowp + static_cast<uint32_t>((j ^ (r & 7)) << 4),
           pack2<BF>(__uint_as_float(u[0]) * scale, __uint_as_float(u[1]) * scale),
           pack2<BF>(__uint_as_float(u[2]) * scale, __uint_as_float(u[3]) * scale),
           pack2<BF>(__uint_as_float(u[4]) * scale, __uint_as_float(u[5]) * scale),
           pack2<BF>(__uint_as_float(u[6]) * scale, __uint_as_float(u[7]) * scale));
  }
}

template <typename T>
struct DT;
template <>
struct DT<__nv_bfloat16> {
  static constexpr bool bf16 = true;
};
template <>
struct DT<__half> {
  static constexpr bool bf16 = false;
};

}  // namespace ta
