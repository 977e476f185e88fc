// Backward attention kernels for sm_103a (tcgen05 + TMA), standard and
// piecewise.
//
// Three kernels, each one CTA per 128-row tile, 320 threads:
//   warps 0-7  element-wise softmax gradient; TMEM lane = row (warp % 4
//              selects the 32-lane quarter), and warp / 4 selects which half
//              of the tile's 128 columns the thread handles;
//   warp 8     TMA producer;
//   warp 9     TMEM allocator and MMA issuer (the whole warp; one elected
//              lane issues each K-loop of MMAs as a single asm block).
//
//  * attn_bwd_dkdv_std_kernel: key-stationary.  The CTA keeps a 128-key tile
//    of K and V in shared memory and walks the query tiles that see it.  Per
//    query tile: S^T = K Q^T and dP^T = V dO^T (tcgen05, into TMEM); thread j
//    (key row j) recomputes P^T = exp2(S^T * c - L * log2 e) and
//    dS^T = P^T o (dP^T - delta), writes both back into TMEM as 16-bit
//    operands; then dV += P^T dO and dK += dS^T Q read them straight from
//    TMEM.  dK is scaled by sm_scale at the end.  Standard mode, and the
//    piecewise mode at D = 64.
//  * attn_bwd_dq_std_kernel: query-stationary.  Per key tile: S = Q K^T,
//    dP = dO V^T, dS = P o (dP - delta), dQ += dS K; dQ * sm_scale at the
//    end; it also forms delta.  Standard mode, and the piecewise mode at
//    D = 64.
//  * attn_bwd_dq_kernel: the same for the piecewise mode at D = 128, with Q1,
//    Q2 and dO resident in shared memory.  (The piecewise key side at D = 128
//    runs in bwd_pw_steps.cu with 64-query steps: TMEM cannot hold all three
//    accumulators beside a 128-query tile's S^T and dP^T.)
//
// Page sources: "Triton fused attention tutorial, updated with JVP support",
// _attn_bwd / _attn_bwd_dkdv / _attn_bwd_dq (pT = exp2(qkT - m), dv += pT do,
// dpT = v do^T, dsT = pT (dpT - Di), dk += dsT q, dq += ds k, dk *= sm_scale)
// with the comment thread's fix (non-causal tiles run over the full range);
// "FlagAttention piecewise.py", _bwd_kv_kernel / _bwd_q_kernel (p = exp2(s *
// qk_scale - L * log2e), ds split by piecewise_mask into ds1 -> (dq1, dk1),
// ds2 -> (dq2, dk2), both scaled by sm_scale).
//
// Departures from the pages, all result-preserving: P^T and dS^T stay in
// TMEM as MMA operands; piecewise tiles that are entirely near or entirely
// far run one score MMA and one gradient MMA instead of two, and a tile
// that straddles w runs its two score products in turn in one buffer.
#include <type_traits>

#include "bwd_common.cuh"
#include "common.cuh"
#include "launch.h"

namespace ta {

enum : int { kNearB = 1, kFarB = 2 };
constexpr int kBwdThreads = 320;
constexpr int kWarpProducer = 8;
constexpr int kWarpMma = 9;
constexpr int kRowWarps = 8;  // arrivals on the per-tile softmax barriers

__device__ __forceinline__ int pw_class_b(int q0, int k0, int P_SEQ, int w) {
  const long long lo = (long long)q0 + P_SEQ - k0 - w;  // min over (i, j) of i + P_SEQ - j - w is lo - (kBN-1)
  // i in [q0, q0 + kBM), j in [k0, k0 + kBN): far iff i + P_SEQ - j - w >= 0
  if (lo - (kBN - 1) >= 0) return kFarB;
  if (lo + (kBM - 1) < 0) return kNearB;
  return kNearB | kFarB;
}



// d (+)= X Y: X is 128 x 128 16-bit in TMEM whose K-steps 0-3 sit at columns
// x + [0, 32) and K-steps 4-7 at x + [64, 96) (the two column halves); Y is a
// 128-row x D tile in smem read as an MN-major B operand (rows = K).
template <int D, int HS = 64>  // HS: TMEM column offset of the second half's K-steps
__device__ __forceinline__ void mma_tY(uint32_t d_tmem, uint32_t x_tmem, uint32_t y_smem, uint32_t idesc,
                                       bool accumulate) {
  const uint64_t dy = sdesc_sw128(y_smem, kBM * 128, 1024);
  uint32_t a[8];
  uint64_t b[8];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    a[kk] = x_tmem + (kk & 3) * 8 + (kk >> 2) * HS;
    b[kk] = dy + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<8>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}


// ======================================================================
//                         dQ (query-stationary)
// ======================================================================
// Half of <dO_r, O_r>, the elements [half * D / 2, (half + 1) * D / 2) of row
// r, summed in fp32: dO from the calling thread's TMEM lane (the row as
// tile_row_to_tmem stores it, two 16-bit elements per column from column
// a_tmem), O from its K-major 128-byte-swizzled tile in shared memory.
template <typename T, int D>
__device__ __forceinline__ float row_dot_half_tmem(uint32_t a_tmem, const uint8_t* b, int r, int half) {
  constexpr int NC = D / 4;  // columns of half a row
  uint32_t x[NC];
  if constexpr (NC == 32) {
    tmem_ld_x32(a_tmem + half * NC, x);
    tmem_ld_wait(x);
  } else {
    static_assert(NC == 16, "D = 64 or 128");
    tmem_ld_x16(a_tmem + half * NC, x);
    tmem_ld_wait(x);
  }
  float acc = 0.f;
#pragma unroll
  for (int c8 = 0; c8 < D / 16; ++c8) {
    const int gc = half * (D / 16) + c8;  // 16-byte chunk of the row
    const uint4 y = *reinterpret_cast<const uint4*>(b + (gc >> 3) * (kBM * 128) + r * 128 + (((gc & 7) ^ (r & 7)) * 16));
    const uint4 xv = make_uint4(x[4 * c8], x[4 * c8 + 1], x[4 * c8 + 2], x[4 * c8 + 3]);
    const T* xp = reinterpret_cast<const T*>(&xv);
    const T* yp = reinterpret_cast<const T*>(&y);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(static_cast<float>(xp[i]), static_cast<float>(yp[i]), acc);
  }
  return acc;
}

// d = A B^T over D with A (128 rows x D, 16-bit) in TMEM, 8 packed columns
// per K-step from a_tmem, and B a 128-row x D K-major swizzled tile in smem.
template <int D>
__device__ __forceinline__ void mma_tB(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem, uint32_t idesc) {
  const uint64_t db0 = sdesc_sw128(b_smem, 16, 1024);
  uint32_t a[D / 16];
  uint64_t b[D / 16];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    a[kk] = a_tmem + kk * 8;
    b[kk] = db0 + static_cast<uint64_t>(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
  }
  mma_ts_n<D / 16>(d_tmem, a, b, idesc, 0u);
}


// The same with dO from its K-major 128-byte-swizzled tile in shared memory.
template <typename T, int D>
__device__ __forceinline__ float row_dot_half_smem(const uint8_t* a, const uint8_t* b, int r, int half) {
  float acc = 0.f;
#pragma unroll
  for (int c8 = 0; c8 < D / 16; ++c8) {
    const int gc = half * (D / 16) + c8;  // 16-byte chunk of the row
    const int off = (gc >> 3) * (kBM * 128) + r * 128 + (((gc & 7) ^ (r & 7)) * 16);
    const uint4 x = *reinterpret_cast<const uint4*>(a + off);
    const uint4 y = *reinterpret_cast<const uint4*>(b + off);
    const T* xp = reinterpret_cast<const T*>(&x);
    const T* yp = reinterpret_cast<const T*>(&y);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc = fmaf(static_cast<float>(xp[i]), static_cast<float>(yp[i]), acc);
  }
  return acc;
}

template <int MODE, int D>
struct DqCfg {
  static constexpr int BLK = kBM * 128;
  static constexpr int TILE = (D / 64) * BLK;
  static constexpr int NRES = (MODE == kStd) ? 2 : 3;  // Q, dO | Q1, Q2, dO
  static constexpr int NKT = (MODE == kStd) ? 2 : 3;   // K, V | K1, K2, V
  static constexpr int STAGE = NKT * TILE;
  static constexpr int RESERVE = 2048;
  static constexpr int ST_FIT = (kSmemMax - RESERVE - (NRES + 1) * TILE) / STAGE;
  static constexpr int STAGES = ST_FIT > 4 ? 4 : ST_FIT;
  static constexpr int OFF_O = NRES * TILE + STAGES * STAGE;  // the O tile (delta), after the ring
  static constexpr int SMEM = OFF_O + TILE + 1024;
  static constexpr uint32_t COL_A = 0, COL_B = 128, COL_DQ = 256, COL_DQ2 = 256 + D;
  static_assert(STAGES >= 1, "tile does not fit in shared memory");
  static_assert(SMEM + RESERVE <= kSmemMax, "shared memory overflow");
  static_assert(COL_DQ2 + (MODE == kPiecewise ? D : 0) <= 512, "TMEM overflow");
};

template <typename T, int MODE, int D>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_q2, const __grid_constant__ CUtensorMap tm_k2,
                       const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dq2,
                       const __grid_constant__ CUtensorMap tm_o, const BwdArgs args) {
  using C = DqCfg<MODE, D>;
  constexpr bool BF = DT<T>::bf16;
  constexpr int STAGES = C::STAGES;
  constexpr bool PW = (MODE == kPiecewise);

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_kv[STAGES], bar_kvempty[STAGES];
  __shared__ __align__(8) uint64_t bar_s, bar_dp, bar_consumed, bar_ds, bar_done;
  __shared__ __align__(8) uint64_t bar_o;  // delta: the O tile landed
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_q_tiles = (args.M + kBM - 1) / kBM;
  int bh, rank;
  if (!grouped_tile(blockIdx.x, args.BH, num_q_tiles, kGroupHeads, &bh, &rank)) return;
  const int qt = num_q_tiles - 1 - rank;  // heaviest causal tiles first
  const int q0 = qt * kBM;
  const int nkv = kv_tiles_for(q0, args.M, args.N, args.P_SEQ, args.causal);
  const bool make_delta = args.delta_out != nullptr;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sQ2 = base + C::TILE;
  uint8_t* sDO = base + (C::NRES - 1) * C::TILE;
  uint8_t* sStages = base + C::NRES * C::TILE;
  uint8_t* sO = base + C::OFF_O;
  auto sK = [&](int st) { return sStages + st * C::STAGE; };
  auto sK2 = [&](int st) { return sStages + st * C::STAGE + C::TILE; };
  auto sV = [&](int st) { return sStages + st * C::STAGE + (C::NKT - 1) * C::TILE; };

  WaitCtl ctl{args.err, args.timeout_ns, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bar_kv[s], 1);
      mbar_init(&bar_kvempty[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_consumed, kRowWarps);
    mbar_init(&bar_ds, kRowWarps);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nkv > 0) {
      bool o_issued = false;
      mbar_expect_tx(&bar_q, C::NRES * C::TILE);
      load_tile_b<D>(sQ, &tm_q, &bar_q, q0, bh);
      if constexpr (PW) load_tile_b<D>(sQ2, &tm_q2, &bar_q, q0, bh);
      load_tile_b<D>(sDO, &tm_do, &bar_q, q0, bh);
      int issued = 0;
      for (int t = 0; t < nkv; ++t) {
        const int st = t % STAGES;
        if (t >= STAGES && !mbar_wait(&bar_kvempty[st], ((t / STAGES) - 1) & 1, ctl, kErrTimeoutMma)) break;
        const int k0 = t * kBN;
        int cls = kNearB;
        if constexpr (PW) cls = pw_class_b(q0, k0, args.P_SEQ, args.w);
        const int nk = ((cls & kNearB) ? 1 : 0) + ((cls & kFarB) ? 1 : 0);
        mbar_expect_tx(&bar_kv[st], (nk + 1) * C::TILE);
        if (cls & kNearB) load_tile_b<D>(sK(st), &tm_k, &bar_kv[st], k0, bh);
        if (cls & kFarB) load_tile_b<D>(sK2(st), &tm_k2, &bar_kv[st], k0, bh);
        load_tile_b<D>(sV(st), &tm_v, &bar_kv[st], k0, bh);
        issued = t + 1;
        if (t == 0 && make_delta) {  // O for delta, behind the first K/V tile
          mbar_expect_tx(&bar_o, C::TILE);
          load_tile_b<D>(sO, &tm_o, &bar_o, q0, bh);
          o_issued = true;
        }
      }
      int zero = 0;
      WaitCtl drain{args.err, args.timeout_ns, reinterpret_cast<volatile int*>(&zero)};
      mbar_wait(&bar_q, 0, drain, kErrTimeoutTma);
      if (o_issued) mbar_wait(&bar_o, 0, drain, kErrTimeoutTma);
      for (int t = issued - STAGES > 0 ? issued - STAGES : 0; t < issued; ++t)
        mbar_wait(&bar_kv[t % STAGES], (t / STAGES) & 1, drain, kErrTimeoutTma);
    }
  } else if (warp == kWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (nkv > 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBM, kBN, BF, false, false);
      constexpr uint32_t idesc_g = idesc_f16(kBM, D, BF, false, true);
      bool ok = warp_wait(&bar_q, 0, ctl, kErrTimeoutTma);
      bool acc1 = false, acc2 = false;
      int nstr = 0;
      for (int t = 0; ok && t < nkv; ++t) {
        const int st = t % STAGES;
        if (!(ok = warp_wait(&bar_kv[st], (t / STAGES) & 1, ctl, kErrTimeoutTma))) break;
        tc_fence_after();
        int cls = kNearB;
        if constexpr (PW) cls = pw_class_b(q0, t * kBN, args.P_SEQ, args.w);
        if (cls == kNearB) {
          mma_abT<D>(tmem + C::COL_A, smem_u32(sQ), smem_u32(sK(st)), idesc_s);
        } else if (cls == kFarB) {
          mma_abT<D>(tmem + C::COL_A, smem_u32(sQ2), smem_u32(sK2(st)), idesc_s);
        } else {
          mma_abT<D>(tmem + C::COL_A, smem_u32(sQ), smem_u32(sK(st)), idesc_s);
          mma_abT<D>(tmem + C::COL_B, smem_u32(sQ2), smem_u32(sK2(st)), idesc_s);
        }
        commit_el(&bar_s);
        if (cls == (kNearB | kFarB)) {
          if (!(ok = warp_wait(&bar_consumed, nstr & 1, ctl, kErrTimeoutSoftmax))) break;
          tc_fence_after();
          ++nstr;
        }
        mma_abT<D>(tmem + C::COL_B, smem_u32(sDO), smem_u32(sV(st)), idesc_s);  // dP = dO V^T
        commit_el(&bar_dp);
        if (!(ok = warp_wait(&bar_ds, t & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        if constexpr (!PW) {
          mma_tY<D>(tmem + C::COL_DQ, tmem + C::COL_B, smem_u32(sK(st)), idesc_g, t > 0);  // dQ += dS K
        } else {
          if (cls == kNearB) {
            mma_tY<D>(tmem + C::COL_DQ, tmem + C::COL_B, smem_u32(sK(st)), idesc_g, acc1);
            acc1 = true;
          } else if (cls == kFarB) {
            mma_tY<D>(tmem + C::COL_DQ2, tmem + C::COL_B, smem_u32(sK2(st)), idesc_g, acc2);
            acc2 = true;
          } else {
            mma_tY<D>(tmem + C::COL_DQ, tmem + C::COL_B, smem_u32(sK(st)), idesc_g, acc1);
            mma_tY<D>(tmem + C::COL_DQ2, tmem + C::COL_A + 32, smem_u32(sK2(st)), idesc_g, acc2);
            acc1 = acc2 = true;
          }
        }
        commit_el(&bar_kvempty[st]);
      }
      if (ok) commit_el(&bar_done);
    }
  } else {
    // --------------------------------------------- query-row softmax gradient
    const int hc = warp >> 2;
    const int cb = 64 * hc;
    const int row = q0 + (threadIdx.x & 127);
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool in_m = row < args.M;
    const size_t g = static_cast<size_t>(bh) * args.M + (in_m ? row : 0);
    const float neg_L2 = in_m ? -args.lse[g] * kLog2e : -INFINITY;
    float dlt = (in_m && !make_delta) ? args.delta[g] : 0.f;
    bool ok = true;
    if (make_delta) {
      // delta of this tile's rows, each softmax group summing half of every
      // row from the resident dO tile and the O tile, while S(0) and dP(0)
      // are computed.  Rows past M and columns past the stored D read as
      // zeros; a tile that sees no key has O = 0 and keeps delta = 0.
      const int r = threadIdx.x & 127;
      float half = 0.f;
      if (nkv > 0) {
        ok = warp_wait(&bar_q, 0, ctl, kErrTimeoutTma) && warp_wait(&bar_o, 0, ctl, kErrTimeoutTma);
        if (ok) half = row_dot_half_smem<T, D>(sDO, sO, r, hc);
      }
      // the groups swap halves through the O tile once both have read it
      float* halves = reinterpret_cast<float*>(sO);
      named_bar_sync(1, kRowWarps * 32);
      halves[hc * kBM + r] = half;
      named_bar_sync(1, kRowWarps * 32);
      dlt = halves[r] + halves[kBM + r];
      if (hc == 0 && in_m) args.delta_out[g] = dlt;
    }
    bool touched1 = false, touched2 = false;
    for (int t = 0; ok && t < nkv; ++t) {
      const int k0 = t * kBN;
      if (!(ok = warp_wait(&bar_s, t & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      int cls = kNearB;
      if constexpr (PW) cls = pw_class_b(q0, k0, args.P_SEQ, args.w);
      touched1 |= (cls & kNearB) != 0;
      touched2 |= (cls & kFarB) != 0;
      const uint32_t s_col = C::COL_A;
      uint32_t s[64];
      tmem_ld_x32(lane_addr + s_col + cb, TB_CHUNK(s, 0));
      tmem_ld_x32(lane_addr + s_col + cb + 32, TB_CHUNK(s, 1));
      tmem_ld_wait(TB_CHUNK(s, 0));
      tmem_ld_wait(TB_CHUNK(s, 1));
      // far iff key k0 + c satisfies row + P_SEQ - (k0 + c) >= w, i.e. c <= pwl
      const long long pwl = (long long)row + args.P_SEQ - k0 - args.w;
      if (cls == (kNearB | kFarB)) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t s2[32];
          tmem_ld_x32(lane_addr + C::COL_B + cb + 32 * c, s2);
          tmem_ld_wait(s2);
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (cb + 32 * c + e <= pwl) s[32 * c + e] = s2[e];
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_consumed);
      }
      float p[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) p[c] = ex2(fmaf(__uint_as_float(s[c]), args.scale_log2, neg_L2));
      if ((args.causal && k0 + kBN - 1 > q0 + args.P_SEQ) || k0 + kBN > args.N) {
        int lim = args.N - 1 - k0;  // keys past N are padding
        if (args.causal) lim = min(lim, row + args.P_SEQ - k0);
        lim -= cb;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c > lim) p[c] = 0.f;
      }
      if (!(ok = warp_wait(&bar_dp, t & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dp[32];
        tmem_ld_x32(lane_addr + C::COL_B + cb + 32 * c, dp);
        tmem_ld_wait(dp);
        uint32_t pk1[16];
        if (cls == (kNearB | kFarB)) {
          uint32_t pk2[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = 32 * c + 2 * e;
            const float ds0 = p[c0] * (__uint_as_float(dp[2 * e]) - dlt);
            const float ds1 = p[c0 + 1] * (__uint_as_float(dp[2 * e + 1]) - dlt);
            const bool f0 = cb + c0 <= pwl, f1 = cb + c0 + 1 <= pwl;
            pk1[e] = pack2<BF>(f0 ? 0.f : ds0, f1 ? 0.f : ds1);
            pk2[e] = pack2<BF>(f0 ? ds0 : 0.f, f1 ? ds1 : 0.f);
          }
          tmem_st_x16(lane_addr + s_col + cb + 32 + 16 * c, pk2);
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = 32 * c + 2 * e;
            pk1[e] = pack2<BF>(p[c0] * (__uint_as_float(dp[2 * e]) - dlt),
                               p[c0 + 1] * (__uint_as_float(dp[2 * e + 1]) - dlt));
          }
        }
        tmem_st_x16(lane_addr + C::COL_B + cb + 16 * c, pk1);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ds);
    }
    if (nkv > 0 && ok) ok = warp_wait(&bar_done, 0, ctl, kErrTimeoutMma);
    tc_fence_after();
    const bool live = ok && nkv > 0;
    (void)g;
    (void)in_m;
    // dQ (dQ1, dQ2), rounded, is staged over the resident Q / Q2 tiles (free:
    // every MMA has finished) in the output maps' swizzled box layout and
    // written by TMA stores, which clip rows past M and columns past D.  An
    // output no key tile touched is zero.
    auto stage_out = [&](int slot, uint32_t col, bool touched) {
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = hc * (D / 64) + cc;  // this thread's 32-column chunks of the row
        uint32_t v[32];
        if (live && touched) {
          tmem_ld_x32(lane_addr + col + 32 * c, v);
          tmem_ld_wait(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        stage_row_chunk_sw128<BF>(smem_u32(base + slot * C::TILE), threadIdx.x & 127, c, v, args.sm_scale);
      }
    };
    stage_out(0, C::COL_DQ, !PW || touched1);
    if constexpr (PW) stage_out(1, C::COL_DQ2, touched2);
    fence_proxy_async_smem();
    named_bar_sync(1, kRowWarps * 32);
    if (warp == 0 && lane == 0 && q0 < args.M) {
#pragma unroll
      for (int kb = 0; kb < D / 64; ++kb) {
        tma_store_3d(&tm_dq, base + kb * (kBM * 128), kb * 64, q0, bh);
        if constexpr (PW) tma_store_3d(&tm_dq2, base + C::TILE + kb * (kBM * 128), kb * 64, q0, bh);
      }
      tma_store_commit_and_wait_read();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}


// d (+)= X Y over the K-steps of chunk group g only (X, Y as in mma_tY); the
// first MMA accumulates iff `accumulate`.  Whole converged warp.
template <int G>
__device__ __forceinline__ void mma_tY_g(uint32_t d_tmem, uint32_t x_tmem, uint32_t y_smem, uint32_t idesc,
                                         bool accumulate) {
  const uint64_t dy = sdesc_sw128(y_smem, kBM * 128, 1024);
  uint32_t a[4];
  uint64_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int kk = chunk_kstep(G, i);
    a[i] = x_tmem + (kk & 3) * 8 + (kk >> 2) * 64;
    b[i] = dy + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<4>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}


// ======================================================================
//      dQ, standard mode: Q and dO in TMEM, three-or-more-deep K/V ring
// ======================================================================
// Q and dO are the A operands of S = Q K^T and dP = dO V^T for every key
// tile, so they live in TMEM (two 16-bit elements per column) and those MMAs
// read only K or V from shared memory.  Q and dO arrive by TMA in the last
// slot of the K/V ring; the softmax warps copy them into TMEM, after which the
// slot joins the ring.  The softmax warps also release the S buffer as soon
// as they have loaded S(t), so S(t + 1) is computed while they work on t:
//   S(0) dP(0) | S(t+1) | dQ(t) dP(t+1) | ...
// When args.delta_out is set the kernel also forms the backward preprocess
// delta = rowsum(dO o O) of its query tile ("Triton fused attention tutorial,
// updated with JVP support", _attn_bwd_preprocess): O arrives after the first
// K/V tile, in a slot of its own and on a barrier of its own, and each
// softmax group sums half of every row's columns (dO from TMEM) while the
// first score MMAs run.  The sum is used here and written to delta_out for
// the dK/dV pass, which then runs after this one.
//
// Piecewise mode (PW, D = 64: TMEM has room for Q2 and dQ2 beside the rest):
// Q1, Q2 and dO are the resident A operands and each ring slot holds K1, K2
// and V, of which a key tile loads the K its class needs.  A tile whose keys
// straddle the distance w gets both score products in turn in the S buffer:
// S(q1, k1), read by the softmax warps, then S(q2, k2), merged by distance
// ("FlagAttention piecewise.py", _bwd_q_kernel).  Its dS goes to dQ1 through
// the near part and to dQ2 through the far part, which the softmax warps
// write beside the near part in the columns dP has vacated.
template <int D, bool PW = false>
struct DqStdCfg {
  static constexpr int BLK = kBM * 128;
  static constexpr int TILE = (D / 64) * BLK;
  static constexpr int NKT = PW ? 3 : 2;  // K, V | K1, K2, V
  static constexpr int STAGE = NKT * TILE;
  static constexpr int ST_FIT = (kSmemMax - 2048 - TILE) / STAGE;
  static constexpr int STAGES = ST_FIT > 4 ? 4 : ST_FIT;
  static constexpr int OFF_O = STAGES * STAGE;  // the O tile (delta), after the ring
  static constexpr int SMEM = OFF_O + TILE + 1024;
  static constexpr uint32_t COL_A = 0, COL_B = 128, COL_DQ = 256;
  static constexpr uint32_t COL_QT = 256 + D, COL_DOT = 256 + D + D / 2;
  static constexpr uint32_t COL_DQ2 = 256 + 2 * D, COL_Q2T = 256 + 3 * D;  // piecewise
  static_assert(!PW || D == 64, "piecewise mode at D = 64 only");
  static_assert(STAGES >= 3, "K/V ring too shallow");
  static_assert(SMEM + 2048 <= kSmemMax, "shared memory overflow");
  static_assert(COL_DOT + D / 2 <= 512 && (!PW || COL_Q2T + D / 2 <= 512), "TMEM overflow");
};

template <typename T, int D, bool PW>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dq_std_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                           const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_o,
                           const __grid_constant__ CUtensorMap tm_q2, const __grid_constant__ CUtensorMap tm_k2,
                           const __grid_constant__ CUtensorMap tm_dq2, const BwdArgs args) {
  using C = DqStdCfg<D, PW>;
  constexpr bool BF = DT<T>::bf16;
  constexpr int STAGES = C::STAGES;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q, bar_qfree, bar_kv[STAGES], bar_kvempty[STAGES];
  __shared__ __align__(8) uint64_t bar_s, bar_consumed, bar_dp, bar_ds[2], bar_done, bar_o;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_q_tiles = (args.M + kBM - 1) / kBM;
  int bh, rank;
  if (!grouped_tile(blockIdx.x, args.BH, num_q_tiles, kGroupHeads, &bh, &rank)) return;
  const int qt = num_q_tiles - 1 - rank;  // heaviest causal tiles first
  const int q0 = qt * kBM;
  const int nkv = kv_tiles_for(q0, args.M, args.N, args.P_SEQ, args.causal);
  const bool make_delta = args.delta_out != nullptr;

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto sK = [&](int st) { return base + st * C::STAGE; };
  auto sK2 = [&](int st) { return base + st * C::STAGE + C::TILE; };  // piecewise
  auto sV = [&](int st) { return base + st * C::STAGE + (C::NKT - 1) * C::TILE; };
  uint8_t* sQ = sK(STAGES - 1);  // Q (Q1, Q2) and dO transit through the last ring slot
  uint8_t* sQ2 = sK2(STAGES - 1);
  uint8_t* sDO = sV(STAGES - 1);
  uint8_t* sO = base + C::OFF_O;
  // piecewise: which score products key tile t needs (kNearB | kFarB bits)
  auto cls_of = [&](int t) { return PW ? pw_class_b(q0, t * kBN, args.P_SEQ, args.w) : kNearB; };

  WaitCtl ctl{args.err, args.timeout_ns, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    mbar_init(&bar_qfree, kRowWarps);
    for (int st = 0; st < STAGES; ++st) {
      mbar_init(&bar_kv[st], 1);
      mbar_init(&bar_kvempty[st], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_consumed, kRowWarps);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_ds[0], kRowWarps);
    mbar_init(&bar_ds[1], kRowWarps);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kWarpProducer) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nkv > 0) {
      mbar_expect_tx(&bar_q, (PW ? 3 : 2) * C::TILE);
      load_tile_b<D>(sQ, &tm_q, &bar_q, q0, bh);
      if constexpr (PW) load_tile_b<D>(sQ2, &tm_q2, &bar_q, q0, bh);
      load_tile_b<D>(sDO, &tm_do, &bar_q, q0, bh);
      int issued = 0;
      bool o_issued = false;
      for (int t = 0; t < nkv; ++t) {
        const int st = t % STAGES;
        if (t >= STAGES) {
          if (!mbar_wait(&bar_kvempty[st], ((t / STAGES) - 1) & 1, ctl, kErrTimeoutMma)) break;
        } else if (st == STAGES - 1) {  // the slot still holds Q and dO until they are in TMEM
          if (!mbar_wait(&bar_qfree, 0, ctl, kErrTimeoutSoftmax)) break;
        }
        const int cls = cls_of(t);
        mbar_expect_tx(&bar_kv[st], (((cls & kNearB) ? 1 : 0) + ((cls & kFarB) ? 1 : 0) + 1) * C::TILE);
        if (cls & kNearB) load_tile_b<D>(sK(st), &tm_k, &bar_kv[st], t * kBN, bh);
        if (PW && (cls & kFarB)) load_tile_b<D>(sK2(st), &tm_k2, &bar_kv[st], t * kBN, bh);
        load_tile_b<D>(sV(st), &tm_v, &bar_kv[st], t * kBN, bh);
        issued = t + 1;
        if (t == 0 && make_delta) {  // O for delta, behind the first K/V tile
          mbar_expect_tx(&bar_o, C::TILE);
          load_tile_b<D>(sO, &tm_o, &bar_o, q0, bh);
          o_issued = true;
        }
      }
      int zero = 0;
      WaitCtl drain{args.err, args.timeout_ns, reinterpret_cast<volatile int*>(&zero)};
      mbar_wait(&bar_q, 0, drain, kErrTimeoutTma);
      if (o_issued) mbar_wait(&bar_o, 0, drain, kErrTimeoutTma);
      for (int t = issued - STAGES > 0 ? issued - STAGES : 0; t < issued; ++t)
        mbar_wait(&bar_kv[t % STAGES], (t / STAGES) & 1, drain, kErrTimeoutTma);
    }
  } else if (warp == kWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (nkv > 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBM, kBN, BF, false, false);
      constexpr uint32_t idesc_g = idesc_f16(kBM, D, BF, false, true);
      // the first (or only) score product of key tile t: S = Q K^T (piecewise:
      // S(q1, k1) if any of the tile is near, else S(q2, k2))
      auto issue_s = [&](int t, int st) {
        if (!PW || (cls_of(t) & kNearB)) {
          mma_tB<D>(tmem + C::COL_A, tmem + C::COL_QT, smem_u32(sK(st)), idesc_s);
        } else if constexpr (PW) {
          mma_tB<D>(tmem + C::COL_A, tmem + C::COL_Q2T, smem_u32(sK2(st)), idesc_s);
        }
        commit_el(&bar_s);
      };
      int ncons = 0;  // phases of bar_consumed waited for (piecewise: two on a tile that straddles w)
      bool acc1 = false, acc2 = false;  // piecewise: dQ1, dQ2 hold a product
      bool ok = warp_wait(&bar_qfree, 0, ctl, kErrTimeoutSoftmax) && warp_wait(&bar_kv[0], 0, ctl, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        mma_tB<D>(tmem + C::COL_B, tmem + C::COL_DOT, smem_u32(sV(0)), idesc_s);  // dP = dO V^T
        commit_el(&bar_dp);
      }
      for (int t = 0; ok && t < nkv; ++t) {
        const int st = t % STAGES;
        const int st1 = (t + 1) % STAGES;
        const bool next = t + 1 < nkv;
        const int cls = cls_of(t);
        if constexpr (PW) {
          if (cls == (kNearB | kFarB)) {  // S(q2, k2) once the softmax warps hold S(q1, k1)
            if (!(ok = warp_wait(&bar_consumed, ncons & 1, ctl, kErrTimeoutSoftmax))) break;
            ++ncons;
            tc_fence_after();
            mma_tB<D>(tmem + C::COL_A, tmem + C::COL_Q2T, smem_u32(sK2(st)), idesc_s);
            commit_el(&bar_s);
          }
        }
        if (next) {
          if (!(ok = warp_wait(&bar_consumed, ncons & 1, ctl, kErrTimeoutSoftmax))) break;
          ++ncons;
          if (!(ok = warp_wait(&bar_kv[st1], ((t + 1) / STAGES) & 1, ctl, kErrTimeoutTma))) break;
          tc_fence_after();
          issue_s(t + 1, st1);
        }
        // dQ += dS K, chunk group 0 as soon as the softmax warps have formed it
        // (piecewise: dQ1 += dS_near K1, dQ2 += dS_far K2, the far part beside
        // the near one when the tile straddles w)
        if (!(ok = warp_wait(&bar_ds[0], t & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        if constexpr (!PW) {
          mma_tY_g<0>(tmem + C::COL_DQ, tmem + C::COL_B, smem_u32(sK(st)), idesc_g, t > 0);
        } else {
          if (cls & kNearB) mma_tY_g<0>(tmem + C::COL_DQ, tmem + C::COL_B, smem_u32(sK(st)), idesc_g, acc1);
          if (cls & kFarB)
            mma_tY_g<0>(tmem + C::COL_DQ2, tmem + C::COL_B + (cls == kFarB ? 0u : 32u), smem_u32(sK2(st)), idesc_g,
                        acc2);
        }
        if (!(ok = warp_wait(&bar_ds[1], t & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        if constexpr (!PW) {
          mma_tY_g<1>(tmem + C::COL_DQ, tmem + C::COL_B, smem_u32(sK(st)), idesc_g, true);
        } else {
          if (cls & kNearB) mma_tY_g<1>(tmem + C::COL_DQ, tmem + C::COL_B, smem_u32(sK(st)), idesc_g, true);
          if (cls & kFarB)
            mma_tY_g<1>(tmem + C::COL_DQ2, tmem + C::COL_B + (cls == kFarB ? 0u : 32u), smem_u32(sK2(st)), idesc_g,
                        true);
          acc1 |= (cls & kNearB) != 0;
          acc2 |= (cls & kFarB) != 0;
        }
        commit_el(&bar_kvempty[st]);
        if (next) {
          mma_tB<D>(tmem + C::COL_B, tmem + C::COL_DOT, smem_u32(sV(st1)), idesc_s);
          commit_el(&bar_dp);
        }
      }
      if (ok) commit_el(&bar_done);
    }
  } else {
    // --------------------------------------------- query-row softmax gradient
    const int hc = warp >> 2;  // key half of the tile: columns [64 hc, 64 hc + 64)
    const int cb = 64 * hc;
    const int r = threadIdx.x & 127;
    const int row = q0 + r;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const bool in_m = row < args.M;
    const size_t g = static_cast<size_t>(bh) * args.M + (in_m ? row : 0);
    const float neg_L2 = in_m ? -args.lse[g] * kLog2e : -INFINITY;
    float dlt = (in_m && !make_delta) ? args.delta[g] : 0.f;
    bool ok = true;
    if (nkv > 0) {  // group 0 copies Q (Q1 and Q2), group 1 copies dO into TMEM
      ok = warp_wait(&bar_q, 0, ctl, kErrTimeoutTma);
      if (ok) {
        tile_row_to_tmem<D>(hc == 0 ? sQ : sDO, r, lane_addr + (hc == 0 ? C::COL_QT : C::COL_DOT));
        if constexpr (PW) {
          if (hc == 0) tile_row_to_tmem<D>(sQ2, r, lane_addr + C::COL_Q2T);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_qfree);
      }
    }
    if (make_delta) {
      // This group's half of delta while S(0) and dP(0) are computed: dO is
      // in TMEM once all eight warps have arrived on bar_qfree.  Rows past M
      // and columns past the stored D read as zeros; a tile that sees no key
      // has O = 0 and keeps delta = 0.
      float half = 0.f;
      if (nkv > 0 && ok) {
        ok = warp_wait(&bar_qfree, 0, ctl, kErrTimeoutSoftmax) && warp_wait(&bar_o, 0, ctl, kErrTimeoutTma);
        if (ok) {
          tc_fence_after();
          half = row_dot_half_tmem<T, D>(lane_addr + C::COL_DOT, sO, r, hc);
        }
      }
      // the groups swap halves through the O tile once both have read it
      float* halves = reinterpret_cast<float*>(sO);
      named_bar_sync(1, kRowWarps * 32);
      halves[hc * kBM + r] = half;
      named_bar_sync(1, kRowWarps * 32);
      dlt = halves[r] + halves[kBM + r];
      if (hc == 0 && in_m) args.delta_out[g] = dlt;
    }
    int sph = 0;  // phases of bar_s seen (piecewise: two on a tile that straddles w)
    bool touched1 = false, touched2 = false;  // piecewise: some key tile fed dQ1 / dQ2
    for (int t = 0; ok && t < nkv; ++t) {
      const int k0 = t * kBN;
      const int cls = cls_of(t);
      if (!(ok = warp_wait(&bar_s, sph & 1, ctl, kErrTimeoutMma))) break;
      ++sph;
      tc_fence_after();
      uint32_t sv[64];
      tmem_ld_x32(lane_addr + C::COL_A + cb, TB_CHUNK(sv, 0));
      tmem_ld_x32(lane_addr + C::COL_A + cb + 32, TB_CHUNK(sv, 1));
      tmem_ld_wait(TB_CHUNK(sv, 0));
      tmem_ld_wait(TB_CHUNK(sv, 1));
      // piecewise: key column j of the tile is far iff j <= pwl
      const long long pwl = PW ? (long long)row + args.P_SEQ - k0 - args.w : 0;
      if constexpr (PW) {
        touched1 |= (cls & kNearB) != 0;
        touched2 |= (cls & kFarB) != 0;
        if (cls == (kNearB | kFarB)) {  // S(q1, k1) is held: take S(q2, k2) where far
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_consumed);
          if (!(ok = warp_wait(&bar_s, sph & 1, ctl, kErrTimeoutMma))) break;
          ++sph;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t s2[32];
            tmem_ld_x32(lane_addr + C::COL_A + cb + 32 * c, s2);
            tmem_ld_wait(s2);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (cb + 32 * c + e <= pwl) sv[32 * c + e] = s2[e];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_consumed);  // S buffer free for S(t + 1)
      float p[64];
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 y = ffma2(make_float2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])),
                               make_float2(args.scale_log2, args.scale_log2), make_float2(neg_L2, neg_L2));
        p[c] = ex2(y.x);
        p[c + 1] = ex2(y.y);
      }
      if ((args.causal && k0 + kBN - 1 > q0 + args.P_SEQ) || k0 + kBN > args.N) {
        int lim = args.N - 1 - k0;  // keys past N are padding
        if (args.causal) lim = min(lim, row + args.P_SEQ - k0);
        lim -= cb;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c > lim) p[c] = 0.f;
      }
      if (!(ok = warp_wait(&bar_dp, t & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      if (PW && cls == (kNearB | kFarB)) {
        // dS split by distance: the near part over dP as usual, the far part
        // 32 columns further (chunk 0's once dP's chunk 1 has been read)
        uint32_t far0[16];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t dp[32];
          tmem_ld_x32(lane_addr + C::COL_B + cb + 32 * c, dp);
          tmem_ld_wait(dp);
          uint32_t nk[16], fk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c0 = 32 * c + 2 * e;
            const float2 ds = fmul2(make_float2(p[c0], p[c0 + 1]),
                                    fadd2(make_float2(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])),
                                          make_float2(-dlt, -dlt)));
            const bool f0 = cb + c0 <= pwl, f1 = cb + c0 + 1 <= pwl;
            nk[e] = pack2<BF>(f0 ? 0.f : ds.x, f1 ? 0.f : ds.y);
            fk[e] = pack2<BF>(f0 ? ds.x : 0.f, f1 ? ds.y : 0.f);
          }
          tmem_st_x16(lane_addr + C::COL_B + cb + 16 * c, nk);
          if (c == 0) {
#pragma unroll
            for (int e = 0; e < 16; ++e) far0[e] = fk[e];
            continue;
          }
          tmem_st_x16(lane_addr + C::COL_B + cb + 32, far0);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_ds[0]);
          tmem_st_x16(lane_addr + C::COL_B + cb + 48, fk);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_ds[1]);
        }
        continue;
      }
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t dp[32];
        tmem_ld_x32(lane_addr + C::COL_B + cb + 32 * c, dp);
        tmem_ld_wait(dp);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int c0 = 32 * c + 2 * e;
          const float2 ds = fmul2(make_float2(p[c0], p[c0 + 1]),
                                  fadd2(make_float2(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])),
                                        make_float2(-dlt, -dlt)));
          pk[e] = pack2<BF>(ds.x, ds.y);
        }
        tmem_st_x16(lane_addr + C::COL_B + cb + 16 * c, pk);  // dS (16-bit) over dP
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_ds[c]);  // chunk group c of dS is in place
      }
    }
    if (nkv > 0 && ok) ok = warp_wait(&bar_done, 0, ctl, kErrTimeoutMma);
    tc_fence_after();
    // dQ (x sm_scale), rounded, is staged over the ring's first K slot (free:
    // every MMA has finished) in the output map's swizzled box layout and
    // written by TMA stores, which clip rows past M and columns past D.
    (void)g;
    const bool live = ok && nkv > 0;
    // (piecewise: dQ1 over the first slot's K1, dQ2 over its K2; an output no
    // key tile fed is zero)
    auto stage_out = [&](uint8_t* tile, uint32_t col, bool fed) {
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = hc * (D / 64) + cc;  // this thread's 32-column chunks of the row
        uint32_t v[32];
        if (live && fed) {
          tmem_ld_x32(lane_addr + col + 32 * c, v);
          tmem_ld_wait(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        stage_row_chunk_sw128<BF>(smem_u32(tile), r, c, v, args.sm_scale);
      }
    };
    stage_out(sK(0), C::COL_DQ, !PW || touched1);
    if constexpr (PW) stage_out(sK2(0), C::COL_DQ2, touched2);
    fence_proxy_async_smem();
    named_bar_sync(1, kRowWarps * 32);
    if (warp == 0 && lane == 0 && q0 < args.M) {
#pragma unroll
      for (int kb = 0; kb < D / 64; ++kb) {
        tma_store_3d(&tm_dq, sK(0) + kb * (kBM * 128), kb * 64, q0, bh);
        if constexpr (PW) tma_store_3d(&tm_dq2, sK2(0) + kb * (kBM * 128), kb * 64, q0, bh);
      }
      tma_store_commit_and_wait_read();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

// ======================================================================
//        dK, dV, standard mode: score MMA one query tile ahead
// ======================================================================
// The softmax warps load S^T(u) into registers and release the score buffer
// at once (bar_consumed), so S^T(u + 1) is computed while they work on u;
// they write P^T and dS^T (16-bit, interleaved 16 + 16 packed columns per
// 32-column chunk) over dP^T, where dV and dK read them:
//   S^T(0) dP^T(0) | S^T(u+1) | dV(u) dK(u) dP^T(u+1) | ...
// That needs Q(u + 1) a whole tile earlier than a plain ring provides, so Q
// has its own ring (3 deep at D = 128) and dO a separate one (2 deep), and the
// per-query L and delta are loaded by the softmax warps themselves, a tile
// ahead, into a small double buffer instead of riding with the Q stages.
//
// Every byte of shared memory the kernel uses lives in the dynamic region
// (no static __shared__), in this order from the first 1024-byte boundary:
// K, V, the Q ring, the dO ring (128-byte swizzled tiles), L and delta
// (double-buffered, see below), then the mbarriers and flags.  The tiles
// leave too little room for a full 1024-byte alignment allowance, so the
// kernel checks the actual padding against PAD at run time and reports
// kErrSmemLayout instead of running if it does not fit.
//
// Piecewise mode (PW, D = 64): K1, K2 and V stationary, each Q ring slot
// holds Q1 and Q2 (loaded as the query tile's class needs), and TMEM has the
// room for dK2 beside dV and dK1 and for the far part of dS^T of a query tile
// that straddles w (Q2 is its B operand), written densely in the last 64
// columns.  Such a tile computes S^T(k1, q1), then, once the softmax warps
// hold it, S^T(k2, q2) in the same buffer, merged per element by distance
// ("FlagAttention piecewise.py", _bwd_kv_kernel).  Its dS phase is a separate
// instance of the code, so the other tiles run the standard one.
template <int D, bool PW = false>
struct DkdvStdCfg {
  static constexpr int BLK = kBM * 128;
  static constexpr int TILE = (D / 64) * BLK;
  static constexpr int NKT = PW ? 3 : 2;  // stationary K, V | K1, K2, V
  static constexpr int NQT = PW ? 2 : 1;  // tiles of a Q ring slot: Q | Q1, Q2
  static constexpr int QST = PW ? 3 : (D == 128) ? 3 : 4;  // Q ring depth
  static constexpr int OST = PW ? 3 : (D == 128) ? 2 : 4;  // dO ring depth
  static constexpr int LD_OFF = (NKT + NQT * QST + OST) * TILE;  // L / delta: [buffer][half][L, delta][64] floats
  static constexpr int LD_BYTES = 2 * 2 * 2 * 64 * 4;
  static constexpr int BAR_OFF = LD_OFF + LD_BYTES;
  static constexpr int BAR_BYTES = 256;
  static constexpr int USED = BAR_OFF + BAR_BYTES;
  static constexpr int PAD = (kSmemMax - USED) < 1023 ? (kSmemMax - USED) : 1023;  // alignment allowance
  static constexpr int SMEM = USED + PAD;
  static constexpr uint32_t COL_A = 0, COL_B = 128, COL_DV = 256, COL_DK = 256 + D;
  static constexpr uint32_t COL_DK2 = 256 + 2 * D, COL_DSF = 256 + 3 * D;  // piecewise
  static_assert(!PW || D == 64, "piecewise mode at D = 64 only");
  static_assert(PAD >= 0 && SMEM <= kSmemMax, "tiles do not fit in shared memory");
  static_assert(BAR_BYTES >= 8 * (1 + 2 * QST + 2 * OST + 6 + 4) + 8, "barrier area too small");
  static_assert(COL_DK + D <= 512 && (!PW || COL_DSF + 64 <= 512), "TMEM overflow");
};

// d (+)= X Y over the K-steps of chunk group G, X with dense K-steps: step kk
// at x + 8 kk; Y as in mma_tY_il_g.  Whole converged warp.
template <int G>
__device__ __forceinline__ void mma_tY_dense_g(uint32_t d_tmem, uint32_t x_tmem, uint32_t y_smem, uint32_t idesc,
                                               bool accumulate) {
  const uint64_t dy = sdesc_sw128(y_smem, kBM * 128, 1024);
  uint32_t a[4];
  uint64_t b[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int kk = chunk_kstep(G, i);
    a[i] = x_tmem + kk * 8;
    b[i] = dy + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<4>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}

// d (+)= X Y with X's K-steps interleaved: step kk at x + (kk / 2) * 32 +
// (kk % 2) * 8 (16 packed columns in each 32-column chunk); Y as in mma_tY.
template <int D>
__device__ __forceinline__ void mma_tY_il(uint32_t d_tmem, uint32_t x_tmem, uint32_t y_smem, uint32_t idesc,
                                          bool accumulate) {
  const uint64_t dy = sdesc_sw128(y_smem, kBM * 128, 1024);
  uint32_t a[8];
  uint64_t b[8];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    a[kk] = x_tmem + (kk >> 1) * 32 + (kk & 1) * 8;
    b[kk] = dy + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<8>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}

template <typename T, int D, bool PW>
__global__ void __launch_bounds__(kBwdThreads, 1)
    attn_bwd_dkdv_std_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                             const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                             const __grid_constant__ CUtensorMap tm_q2, const __grid_constant__ CUtensorMap tm_k2,
                             const __grid_constant__ CUtensorMap tm_dk2, const BwdArgs args) {
  using C = DkdvStdCfg<D, PW>;
  constexpr bool BF = DT<T>::bf16;
  constexpr int QST = C::QST, OST = C::OST;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (base - smem_raw > C::PAD) {  // uniform across the CTA: nothing has been touched yet
    if (threadIdx.x == 0 && args.err) atomicOr(args.err, kErrSmemLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::BAR_OFF);
  uint64_t& bar_kv = bars[0];
  uint64_t* bar_qf = bars + 1;
  uint64_t* bar_qe = bar_qf + QST;
  uint64_t* bar_of = bar_qe + QST;
  uint64_t* bar_oe = bar_of + OST;
  uint64_t& bar_s = bar_oe[OST];
  uint64_t& bar_consumed = bar_oe[OST + 1];
  uint64_t& bar_dp = bar_oe[OST + 2];
  uint64_t* bar_ds = bar_oe + OST + 3;  // [chunk group]
  uint64_t& bar_done = bar_oe[OST + 5];
  uint64_t* bar_pub = bar_oe + OST + 6;  // [buffer * 2 + half]: L / delta of a tile stored
  uint32_t& tmem_slot = *reinterpret_cast<uint32_t*>(bar_pub + 4);
  int& abort_flag = *(reinterpret_cast<int*>(bar_pub + 4) + 1);
  float* sLD = reinterpret_cast<float*>(base + C::LD_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int bh, kt;  // key tiles with the most query tiles (the first ones, causal) first
  if (!grouped_tile(blockIdx.x, args.BH, (args.N + kBN - 1) / kBN, kGroupHeads, &bh, &kt)) return;
  const int k0 = kt * kBN;
  const int num_q_tiles = (args.M + kBM - 1) / kBM;
  const int i0 = first_q_tile_for(k0, args.P_SEQ, args.causal);
  const int nq = num_q_tiles > i0 ? num_q_tiles - i0 : 0;

  uint8_t* sK = base;             // K (piecewise: K1)
  uint8_t* sK2 = base + C::TILE;  // piecewise
  uint8_t* sV = base + (C::NKT - 1) * C::TILE;
  auto sQ = [&](int i) { return base + (C::NKT + C::NQT * i) * C::TILE; };       // Q (Q1)
  auto sQ2 = [&](int i) { return base + (C::NKT + C::NQT * i + 1) * C::TILE; };  // piecewise
  auto sDO = [&](int i) { return base + (C::NKT + C::NQT * QST + i) * C::TILE; };
  // piecewise: which score products query tile u needs (kNearB | kFarB bits)
  auto cls_of = [&](int u) { return PW ? pw_class_b((i0 + u) * kBM, k0, args.P_SEQ, args.w) : kNearB; };

  WaitCtl ctl{args.err, args.timeout_ns, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_kv, 1);
    for (int i = 0; i < QST; ++i) {
      mbar_init(&bar_qf[i], 1);
      mbar_init(&bar_qe[i], 1);
    }
    for (int i = 0; i < OST; ++i) {
      mbar_init(&bar_of[i], 1);
      mbar_init(&bar_oe[i], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_consumed, kRowWarps);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_ds[0], kRowWarps);
    mbar_init(&bar_ds[1], kRowWarps);
    mbar_init(&bar_done, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&bar_pub[i], kRowWarps / 2);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kWarpProducer) {
    // ---------------------- producer: lane 0 K, V and the Q ring; lane 1 the dO ring
    if (lane < 2 && nq > 0) {
      const bool is_q = (lane == 0);
      const int depth = is_q ? QST : OST;
      uint64_t* full = is_q ? bar_qf : bar_of;
      uint64_t* empty = is_q ? bar_qe : bar_oe;
      const CUtensorMap* map = is_q ? &tm_q : &tm_do;
      if (is_q) {
        mbar_expect_tx(&bar_kv, C::NKT * C::TILE);
        load_tile_b<D>(sK, &tm_k, &bar_kv, k0, bh);
        if constexpr (PW) load_tile_b<D>(sK2, &tm_k2, &bar_kv, k0, bh);
        load_tile_b<D>(sV, &tm_v, &bar_kv, k0, bh);
      }
      int issued = 0;
      for (int u = 0; u < nq; ++u) {
        const int st = u % depth;
        if (u >= depth && !mbar_wait(&empty[st], ((u / depth) - 1) & 1, ctl, kErrTimeoutMma)) break;
        if (PW && is_q) {  // Q1 if any of the tile is near, Q2 if any is far
          const int cls = cls_of(u);
          mbar_expect_tx(&full[st], (((cls & kNearB) ? 1 : 0) + ((cls & kFarB) ? 1 : 0)) * C::TILE);
          if (cls & kNearB) load_tile_b<D>(sQ(st), &tm_q, &full[st], (i0 + u) * kBM, bh);
          if (cls & kFarB) load_tile_b<D>(sQ2(st), &tm_q2, &full[st], (i0 + u) * kBM, bh);
        } else {
          mbar_expect_tx(&full[st], C::TILE);
          load_tile_b<D>(is_q ? sQ(st) : sDO(st), map, &full[st], (i0 + u) * kBM, bh);
        }
        issued = u + 1;
      }
      int zero = 0;
      WaitCtl drain{args.err, args.timeout_ns, reinterpret_cast<volatile int*>(&zero)};
      if (is_q) mbar_wait(&bar_kv, 0, drain, kErrTimeoutTma);
      for (int u = issued - depth > 0 ? issued - depth : 0; u < issued; ++u)
        mbar_wait(&full[u % depth], (u / depth) & 1, drain, kErrTimeoutTma);
    }
  } else if (warp == kWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (nq > 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBN, kBM, BF, false, false);  // M = keys, N = queries
      constexpr uint32_t idesc_g = idesc_f16(kBN, D, BF, false, true);     // M = keys, N = D
      // the first (or only) score product of query tile u: S^T = K Q^T
      // (piecewise: S^T(k1, q1) if any of the tile is near, else S^T(k2, q2))
      auto issue_s = [&](int u, int sq) {
        if (!PW || (cls_of(u) & kNearB)) {
          mma_abT<D>(tmem + C::COL_A, smem_u32(sK), smem_u32(sQ(sq)), idesc_s);
        } else if constexpr (PW) {
          mma_abT<D>(tmem + C::COL_A, smem_u32(sK2), smem_u32(sQ2(sq)), idesc_s);
        }
        commit_el(&bar_s);
      };
      int ncons = 0;  // phases of bar_consumed waited for (piecewise: two on a tile that straddles w)
      bool acc1 = false, acc2 = false;  // piecewise: dK1, dK2 hold a product
      bool ok = warp_wait(&bar_kv, 0, ctl, kErrTimeoutTma) && warp_wait(&bar_qf[0], 0, ctl, kErrTimeoutTma) &&
                warp_wait(&bar_of[0], 0, ctl, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        mma_abT<D>(tmem + C::COL_B, smem_u32(sV), smem_u32(sDO(0)), idesc_s);  // dP^T = V dO^T
        commit_el(&bar_dp);
      }
      for (int u = 0; ok && u < nq; ++u) {
        const int sq = u % QST, so = u % OST;
        const int sq1 = (u + 1) % QST, so1 = (u + 1) % OST;
        const bool next = u + 1 < nq;
        const int cls = cls_of(u);
        if constexpr (PW) {
          if (cls == (kNearB | kFarB)) {  // S^T(k2, q2) once the softmax warps hold S^T(k1, q1)
            if (!(ok = warp_wait(&bar_consumed, ncons & 1, ctl, kErrTimeoutSoftmax))) break;
            ++ncons;
            tc_fence_after();
            mma_abT<D>(tmem + C::COL_A, smem_u32(sK2), smem_u32(sQ2(sq)), idesc_s);
            commit_el(&bar_s);
          }
        }
        if (next) {
          if (!(ok = warp_wait(&bar_consumed, ncons & 1, ctl, kErrTimeoutSoftmax))) break;
          ++ncons;
          if (!(ok = warp_wait(&bar_qf[sq1], ((u + 1) / QST) & 1, ctl, kErrTimeoutTma))) break;
          tc_fence_after();
          issue_s(u + 1, sq1);
        }
        // dV += P^T dO and dK += dS^T Q, chunk group 0 as soon as the softmax
        // warps have formed it (piecewise: dK1 += dS_near^T Q1, dK2 += dS_far^T
        // Q2; the far part sits in its own columns when the tile straddles w)
        if (!(ok = warp_wait(&bar_ds[0], u & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        mma_tY_il_g<0>(tmem + C::COL_DV, tmem + C::COL_B, smem_u32(sDO(so)), idesc_g, u > 0);
        if constexpr (!PW) {
          mma_tY_il_g<0>(tmem + C::COL_DK, tmem + C::COL_B + 16, smem_u32(sQ(sq)), idesc_g, u > 0);
        } else {
          if (cls == kFarB) {
            mma_tY_il_g<0>(tmem + C::COL_DK2, tmem + C::COL_B + 16, smem_u32(sQ2(sq)), idesc_g, acc2);
          } else {
            mma_tY_il_g<0>(tmem + C::COL_DK, tmem + C::COL_B + 16, smem_u32(sQ(sq)), idesc_g, acc1);
            if (cls & kFarB) mma_tY_dense_g<0>(tmem + C::COL_DK2, tmem + C::COL_DSF, smem_u32(sQ2(sq)), idesc_g, acc2);
          }
        }
        if (!(ok = warp_wait(&bar_ds[1], u & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        mma_tY_il_g<1>(tmem + C::COL_DV, tmem + C::COL_B, smem_u32(sDO(so)), idesc_g, true);
        commit_el(&bar_oe[so]);
        if constexpr (!PW) {
          mma_tY_il_g<1>(tmem + C::COL_DK, tmem + C::COL_B + 16, smem_u32(sQ(sq)), idesc_g, true);
        } else {
          if (cls == kFarB) {
            mma_tY_il_g<1>(tmem + C::COL_DK2, tmem + C::COL_B + 16, smem_u32(sQ2(sq)), idesc_g, true);
          } else {
            mma_tY_il_g<1>(tmem + C::COL_DK, tmem + C::COL_B + 16, smem_u32(sQ(sq)), idesc_g, true);
            if (cls & kFarB) mma_tY_dense_g<1>(tmem + C::COL_DK2, tmem + C::COL_DSF, smem_u32(sQ2(sq)), idesc_g, true);
          }
          acc1 |= (cls & kNearB) != 0;
          acc2 |= (cls & kFarB) != 0;
        }
        commit_el(&bar_qe[sq]);
        if (next) {
          if (!(ok = warp_wait(&bar_of[so1], ((u + 1) / OST) & 1, ctl, kErrTimeoutTma))) break;
          tc_fence_after();
          mma_abT<D>(tmem + C::COL_B, smem_u32(sV), smem_u32(sDO(so1)), idesc_s);
          commit_el(&bar_dp);
        }
      }
      if (ok) commit_el(&bar_done);
    }
  } else {
    // ------------------------------------------- key-row softmax gradient
    const int hc = warp >> 2;                // query half of the tile: columns [64 hc, 64 hc + 64)
    const int cb = 64 * hc;
    const int j = k0 + (threadIdx.x & 127);  // this thread's key
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    // L and delta of the half's 64 queries: the half's 128 threads each load
    // one of the 128 values (coalesced) a tile ahead, store it once they are
    // done with the current tile and publish the buffer on bar_pub; the
    // reads are then shared-memory broadcasts.  Queries past M read L = +inf
    // (P = 0) and delta = 0.
    const int ld_arr = (threadIdx.x & 127) >> 6;  // 0: L, 1: delta
    const int ld_col = threadIdx.x & 63;
    auto ld_fetch = [&](int u) -> float {
      const int q = (i0 + u) * kBM + cb + ld_col;
      if (q >= args.M) return ld_arr ? 0.f : INFINITY;
      return __ldg((ld_arr ? args.delta : args.lse) + static_cast<size_t>(bh) * args.M + q);
    };
    auto ld_slot = [&](int u) { return sLD + ((u & 1) * 2 + hc) * 128; };
    if (nq > 0) {
      ld_slot(0)[ld_arr * 64 + ld_col] = ld_fetch(0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pub[hc]);
    }
    bool ok = true;
    int sph = 0;  // phases of bar_s seen (piecewise: two on a tile that straddles w)
    bool touched1 = false, touched2 = false;  // piecewise: some query tile fed dK1 / dK2
    for (int u = 0; u < nq; ++u) {
      const int q0 = (i0 + u) * kBM;
      const int qb = q0 + cb;  // first query of this thread's columns
      const int cls = cls_of(u);
      const float pre = (u + 1 < nq) ? ld_fetch(u + 1) : 0.f;
      if (!(ok = warp_wait(&bar_s, sph & 1, ctl, kErrTimeoutMma))) break;
      ++sph;
      tc_fence_after();
      // 16-lane shapes: in each 16-lane group g of its warp, thread t holds
      // keys (t / 4) and (t / 4 + 8) at the query pairs 8 jj + 2 m, +1
      // (m = t % 4) of the half, so it needs 16 of the half's L and delta
      // values instead of 64.  sv[32 g + 4 jj + e], e = {(k, q), (k, q + 1),
      // (k + 8, q), (k + 8, q + 1)}.
      uint32_t sv[64];
      tmem_ld_16x256b_x8(lane_addr + C::COL_A + cb, TB_CHUNK(sv, 0));
      tmem_ld_16x256b_x8(lane_addr + (16u << 16) + C::COL_A + cb, TB_CHUNK(sv, 1));
      tmem_ld_wait(TB_CHUNK(sv, 0));
      tmem_ld_wait(TB_CHUNK(sv, 1));
      // piecewise: element (g, jj, e) (key k0 + 32 (warp % 4) + lane / 4 + 16 g
      // + 8 (e / 2), query qb + 2 m + 8 jj + e % 2) is far, its distance
      // query + P_SEQ - key at least w, iff 8 jj + (e & 1) >= fl + 16 g + 8 (e >> 1)
      int fl = 0;
      if constexpr (PW) {
        const long long f = (long long)args.w - args.P_SEQ - qb - 2 * (lane & 3) + k0 + 32 * (warp & 3) + (lane >> 2);
        fl = f < -128 ? -128 : (f > 128 ? 128 : static_cast<int>(f));
        touched1 |= (cls & kNearB) != 0;
        touched2 |= (cls & kFarB) != 0;
        if (cls == (kNearB | kFarB)) {  // S^T(k1, q1) is held: take S^T(k2, q2) where far
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_consumed);
          if (!(ok = warp_wait(&bar_s, sph & 1, ctl, kErrTimeoutMma))) break;
          ++sph;
          tc_fence_after();
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t s2[32];
            tmem_ld_16x256b_x8(lane_addr + (static_cast<uint32_t>(16 * g) << 16) + C::COL_A + cb, s2);
            tmem_ld_wait(s2);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
#pragma unroll
              for (int e = 0; e < 4; ++e)
                if (8 * jj + (e & 1) >= fl + 16 * g + 8 * (e >> 1)) sv[32 * g + 4 * jj + e] = s2[4 * jj + e];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_consumed);  // score buffer free for S^T(u + 1)
      if (!(ok = warp_wait(&bar_pub[(u & 1) * 2 + hc], (u >> 1) & 1, ctl, kErrTimeoutSoftmax))) break;
      const int m = lane & 3;
      const float* sL = ld_slot(u) + 2 * m;
      const float* sD = sL + 64;
      const float2 sc2 = make_float2(args.scale_log2, args.scale_log2);
      float p[64];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float2 l2 = *reinterpret_cast<const float2*>(sL + 8 * jj);
        const float2 nl = fmul2(l2, make_float2(-kLog2e, -kLog2e));
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int i = 32 * g + 4 * jj;
          const float2 y0 = ffma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), sc2, nl);
          const float2 y1 = ffma2(make_float2(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])), sc2, nl);
          p[i + 0] = ex2(y0.x);
          p[i + 1] = ex2(y0.y);
          p[i + 2] = ex2(y1.x);
          p[i + 3] = ex2(y1.y);
        }
      }
      if (args.causal && k0 + kBN - 1 > q0 + args.P_SEQ) {  // key k visible from q iff q >= k - P_SEQ
        // element (g, jj, e) is masked iff 8 jj + (e & 1) < lo + 16 g + 8 (e >> 1)
        const int lo = k0 + 32 * (warp & 3) + (lane >> 2) - args.P_SEQ - qb - 2 * m;
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
          for (int jj = 0; jj < 8; ++jj)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (8 * jj + (e & 1) < lo + 16 * g + 8 * (e >> 1)) p[32 * g + 4 * jj + e] = 0.f;
      }
      if (!(ok = warp_wait(&bar_dp, u & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      // P^T and dS^T of the tile (SPLIT: a piecewise tile that straddles w,
      // whose dS^T is split by distance), compiled apart so that the other
      // tiles run the standard code
      auto write_chunks = [&](auto split_tag) {
        constexpr bool SPLIT = decltype(split_tag)::value;
  #pragma unroll
        for (int c = 0; c < 2; ++c) {
          // chunk c (32 queries): read dP^T, write P^T and dS^T (16 packed
          // columns each, pair 4 jq + m) back into the same 32 columns
          uint32_t dp[32];  // [g][16]
          tmem_ld_16x256b_x4(lane_addr + C::COL_B + cb + 32 * c, TB_CHUNK16(dp, 0));
          tmem_ld_16x256b_x4(lane_addr + (16u << 16) + C::COL_B + cb + 32 * c, TB_CHUNK16(dp, 1));
          tmem_ld_wait(TB_CHUNK16(dp, 0));
          tmem_ld_wait(TB_CHUNK16(dp, 1));
          float2 nd2[4];  // -delta of the thread's query pairs
  #pragma unroll
          for (int jq = 0; jq < 4; ++jq) {
            const float2 d2 = *reinterpret_cast<const float2*>(sD + 8 * (4 * c + jq));
            nd2[jq] = make_float2(-d2.x, -d2.y);
          }
  #pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t pp[8], pd[8];
            uint32_t pf[8];  // SPLIT: the far part of dS^T (pd keeps the near part)
  #pragma unroll
            for (int jq = 0; jq < 4; ++jq) {
              const int i = 32 * g + 4 * (4 * c + jq);
              const int di = 16 * g + 4 * jq;
              pp[2 * jq] = pack2<BF>(p[i], p[i + 1]);
              pp[2 * jq + 1] = pack2<BF>(p[i + 2], p[i + 3]);
              const float2 s0 = fmul2(make_float2(p[i], p[i + 1]),
                                      fadd2(make_float2(__uint_as_float(dp[di]), __uint_as_float(dp[di + 1])), nd2[jq]));
              const float2 s1 = fmul2(make_float2(p[i + 2], p[i + 3]),
                                      fadd2(make_float2(__uint_as_float(dp[di + 2]), __uint_as_float(dp[di + 3])), nd2[jq]));
              if constexpr (SPLIT) {
                const int jj = 4 * c + jq;
                const bool f0 = 8 * jj >= fl + 16 * g, f1 = 8 * jj + 1 >= fl + 16 * g;
                const bool f2 = 8 * jj >= fl + 16 * g + 8, f3 = 8 * jj + 1 >= fl + 16 * g + 8;
                pd[2 * jq] = pack2<BF>(f0 ? 0.f : s0.x, f1 ? 0.f : s0.y);
                pd[2 * jq + 1] = pack2<BF>(f2 ? 0.f : s1.x, f3 ? 0.f : s1.y);
                pf[2 * jq] = pack2<BF>(f0 ? s0.x : 0.f, f1 ? s0.y : 0.f);
                pf[2 * jq + 1] = pack2<BF>(f2 ? s1.x : 0.f, f3 ? s1.y : 0.f);
              } else {
                pd[2 * jq] = pack2<BF>(s0.x, s0.y);
                pd[2 * jq + 1] = pack2<BF>(s1.x, s1.y);
              }
            }
            const uint32_t ga = lane_addr + (static_cast<uint32_t>(16 * g) << 16) + C::COL_B + cb + 32 * c;
            tmem_st_16x128b_x4(ga, pp);
            tmem_st_16x128b_x4(ga + 16, pd);
            if constexpr (SPLIT)
              tmem_st_16x128b_x4(lane_addr + (static_cast<uint32_t>(16 * g) << 16) + C::COL_DSF + (cb >> 1) + 16 * c,
                                 pf);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_ds[c]);  // chunk group c of P^T / dS^T is in place
        }
      };
      if (PW && cls == (kNearB | kFarB)) write_chunks(std::true_type{});
      else write_chunks(std::false_type{});
      if (u + 1 < nq) {  // every warp of the half is past tile u - 1, the buffer's previous tile
        ld_slot(u + 1)[ld_arr * 64 + ld_col] = pre;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_pub[((u + 1) & 1) * 2 + hc]);
      }
    }
    // ------------------------------------------------------------ epilogue
    if (nq > 0 && ok) ok = warp_wait(&bar_done, 0, ctl, kErrTimeoutMma);
    tc_fence_after();
    // dV and dK (x sm_scale), rounded, are staged over the K and V tiles
    // (free: every MMA has finished) in the output maps' swizzled box layout
    // and written by TMA stores, which clip rows past N and columns past D.
    (void)j;
    const int r = threadIdx.x & 127;  // this thread's key within the tile
    const bool live = ok && nq > 0;
    // (piecewise: dK2 over K2; an output no query tile fed is zero)
#pragma unroll
    for (int a = 0; a < (PW ? 3 : 2); ++a) {  // 0: dV over K, 1: dK over V, 2: dK2 over K2
      const bool fed = !PW || a == 0 || (a == 1 ? touched1 : touched2);
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = hc * (D / 64) + cc;  // this thread's 32-column chunks of the row
        uint32_t v[32];
        if (live && fed) {
          tmem_ld_x32(lane_addr + (a == 0 ? C::COL_DV : a == 1 ? C::COL_DK : C::COL_DK2) + 32 * c, v);
          tmem_ld_wait(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        stage_row_chunk_sw128<BF>(smem_u32(a == 0 ? sK : a == 1 ? sV : sK2), r, c, v, a ? args.sm_scale : 1.f);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, kRowWarps * 32);
    if (warp == 0 && lane == 0 && k0 < args.N) {
#pragma unroll
      for (int kb = 0; kb < D / 64; ++kb) {
        tma_store_3d(&tm_dv, sK + kb * (kBM * 128), kb * 64, k0, bh);
        tma_store_3d(&tm_dk, sV + kb * (kBM * 128), kb * 64, k0, bh);
        if constexpr (PW) tma_store_3d(&tm_dk2, sK2 + kb * (kBM * 128), kb * 64, k0, bh);
      }
      tma_store_commit_and_wait_read();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side
template <typename T, int MODE, int D>
static cudaError_t launch_dq_t(const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  using C = DqCfg<MODE, D>;
  auto kern = attn_bwd_dq_kernel<T, MODE, D>;
  static std::atomic<bool> attr[kMaxDevices];
  cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
  if (e_attr != cudaSuccess) return e_attr;
  const long long blocks = static_cast<long long>(a.BH) * ((a.M + kBM - 1) / kBM);
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(blocks), kBwdThreads, C::SMEM, s>>>(m.q, m.k, m.v, m.dO, m.q2, m.k2, m.dq, m.dq2,
                                                                    a.delta_out ? m.o : m.q, a);
  return cudaGetLastError();
}

template <typename T, int D, bool PW = false>
static cudaError_t launch_dkdv_std_t(const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  using C = DkdvStdCfg<D, PW>;
  auto kern = attn_bwd_dkdv_std_kernel<T, D, PW>;
  static std::atomic<bool> attr[kMaxDevices];
  cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
  if (e_attr != cudaSuccess) return e_attr;
  const long long blocks = static_cast<long long>(a.BH) * ((a.N + kBN - 1) / kBN);
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(blocks), kBwdThreads, C::SMEM, s>>>(m.q, m.k, m.v, m.dO, m.dk, m.dv,
                                                                    PW ? m.q2 : m.q, PW ? m.k2 : m.k,
                                                                    PW ? m.dk2 : m.dk, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(int mode, bool bf16, int D, const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  if (mode == kStd && D == 64) return bf16 ? launch_dkdv_std_t<__nv_bfloat16, 64>(m, a, s) : launch_dkdv_std_t<__half, 64>(m, a, s);
  if (mode == kStd && D == 128) return bf16 ? launch_dkdv_std_t<__nv_bfloat16, 128>(m, a, s) : launch_dkdv_std_t<__half, 128>(m, a, s);
  if (mode == kPiecewise && D == 64)  // the standard kernel's structure with K2, Q2 and dK2
    return bf16 ? launch_dkdv_std_t<__nv_bfloat16, 64, true>(m, a, s) : launch_dkdv_std_t<__half, 64, true>(m, a, s);
  // piecewise D = 128: the one-pass kernel of bwd_pw_steps.cu (launch_bwd_pw_steps)
  return cudaErrorNotSupported;
}

template <typename T, int D, bool PW = false>
static cudaError_t launch_dq_std_t(const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  using C = DqStdCfg<D, PW>;
  auto kern = attn_bwd_dq_std_kernel<T, D, PW>;
  static std::atomic<bool> attr[kMaxDevices];
  cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
  if (e_attr != cudaSuccess) return e_attr;
  const long long blocks = static_cast<long long>(a.BH) * ((a.M + kBM - 1) / kBM);
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(blocks), kBwdThreads, C::SMEM, s>>>(m.q, m.k, m.v, m.dO, m.dq,
                                                                    a.delta_out ? m.o : m.q, PW ? m.q2 : m.q,
                                                                    PW ? m.k2 : m.k, PW ? m.dq2 : m.dq, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dq(int mode, bool bf16, int D, const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  if (mode == kStd && D == 64) return bf16 ? launch_dq_std_t<__nv_bfloat16, 64>(m, a, s) : launch_dq_std_t<__half, 64>(m, a, s);
  if (mode == kStd && D == 128) return bf16 ? launch_dq_std_t<__nv_bfloat16, 128>(m, a, s) : launch_dq_std_t<__half, 128>(m, a, s);
  if (mode == kPiecewise && D == 64)  // the standard kernel's structure with Q2 and dQ2 in TMEM
    return bf16 ? launch_dq_std_t<__nv_bfloat16, 64, true>(m, a, s) : launch_dq_std_t<__half, 64, true>(m, a, s);
  if (mode == kPiecewise && D == 128) return bf16 ? launch_dq_t<__nv_bfloat16, kPiecewise, 128>(m, a, s) : launch_dq_t<__half, kPiecewise, 128>(m, a, s);
  return cudaErrorNotSupported;
}

}  // namespace ta

TA_GUARD_ACCESSOR(bwd)
