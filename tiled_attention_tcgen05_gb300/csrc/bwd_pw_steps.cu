// Piecewise backward, key side, in ONE pass at D = 128 (sm_103a, tcgen05 +
// TMA): dV, dK1 and dK2 of a 128-key tile.  "FlagAttention piecewise.py",
// _bwd_kv_kernel: with P = exp(S - L), S_ij = sm_scale q2_i . k2_j where the
// signed distance i + N - M - j >= w (far) and sm_scale q1_i . k1_j otherwise
// (near), dP = dO V^T and dS = P o (dP - delta):
//   dV = P^T dO,  dK1 = sm_scale dS_near^T Q1,  dK2 = sm_scale dS_far^T Q2.
//
// The key-stationary kernel of bwd.cu streams 128-query tiles; at D = 128
// TMEM cannot hold S^T, dP^T and the three accumulators of such a tile
// (a two-pass split would repeat the score and softmax work).  Here the
// queries stream in 64-row steps, as in the backward of the JVP: S^T and
// dP^T take 64 columns each and the accumulators dV, dK1, dK2 128 each, 512
// in all.
//
// One CTA per (head, key tile), 320 threads:
//   warps 0-7  element-wise phase; warp % 4 selects the 32-lane quarter
//              (keys) and warp / 4 the half of the step's 64 queries;
//   warp 8     TMA producer: K1, K2, V once, then Q1, Q2, dO per step (two
//              stages) with the step's L * log2(e) and delta;
//   warp 9     TMEM allocator and MMA issuer.
// TMEM: S buffer [0, 64), dP buffer [64, 128), dV [128, 256), dK1 [256, 384),
// dK2 [384, 512).  The 16-bit MMA operands are written back in place, a
// thread packing its 32 columns into 16 (K-step kk of 16 queries at column
// 32 (kk / 2) + 8 (kk % 2)): P^T into the S buffer, dS^T (the near part, or
// all of it when the step is wholly far) into the dP buffer, and on a step
// that straddles the distance w the far part of dS^T into the S buffer's
// other 16 columns of each 32-column slice.  Such a step computes S(q1, k1)
// into the S buffer and S(q2, k2) into the dP buffer; dP^T follows once the
// element-wise warps have read S(q2, k2).
#include "bwd_common.cuh"
#include "common.cuh"
#include "launch.h"

namespace ta {

namespace {

constexpr int kPsThreads = 320;
constexpr int kPsWarpProducer = 8;
constexpr int kPsWarpMma = 9;
constexpr int kPsRowWarps = 8;
constexpr int kPsR = 64;  // queries of a streamed step

enum : int { kPsNear = 1, kPsFar = 2 };

template <int D>
struct PwStepCfg {
  static constexpr int XBLK = kBM * 128;  // one 64-column block of a 128-row tile (bytes)
  static constexpr int YBLK = kPsR * 128; // one 64-column block of a 64-row tile
  static constexpr int XT = (D / 64) * XBLK;
  static constexpr int YT = (D / 64) * YBLK;
  static constexpr int STAGE = 3 * YT;  // Q1, Q2, dO of one step
  static constexpr int STATIC_RESERVE = 4 * 1024;
  static constexpr int FIT = (kSmemMax - STATIC_RESERVE - 1024 - 3 * XT) / STAGE;
  static constexpr int STAGES = FIT > 3 ? 3 : FIT;
  static constexpr int SMEM = 3 * XT + STAGES * STAGE + 1024;
  static constexpr uint32_t COL_S = 0, COL_DP = 64, COL_DV = 128, COL_DK1 = 128 + D, COL_DK2 = 128 + 2 * D;
  static_assert(STAGES >= 2, "two stages of streamed steps must fit");
  static_assert(COL_DK2 + D <= 512, "TMEM overflow");
};

// Which score products the step [r0, r0 + 64) needs against keys
// [k0, k0 + 128): far iff i + P_SEQ - j >= w.
__device__ __forceinline__ int pw_step_class(int r0, int k0, int P_SEQ, int w) {
  const long long lo = (long long)r0 + P_SEQ - (k0 + kBN - 1) - w;  // smallest i + P_SEQ - j - w
  const long long hi = (long long)r0 + kPsR - 1 + P_SEQ - k0 - w;   // largest
  if (lo >= 0) return kPsFar;
  if (hi < 0) return kPsNear;
  return kPsNear | kPsFar;
}

template <int D>
__device__ __forceinline__ void ps_load(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row0, int bh,
                                        int blk) {
#pragma unroll
  for (int kb = 0; kb < D / 64; ++kb) tma_load_3d(dst + kb * blk, map, bar, kb * 64, row0, bh);
}

// d = X Y^T over D: X a 128-row tile, Y a 64-row tile, both K-major with
// 128-byte swizzle in 64-column blocks.
template <int D>
__device__ __forceinline__ void ps_mma_xyT(uint32_t d_tmem, uint32_t x_smem, uint32_t y_smem, uint32_t idesc) {
  const uint64_t dx0 = sdesc_sw128(x_smem, 16, 1024);
  const uint64_t dy0 = sdesc_sw128(y_smem, 16, 1024);
  uint64_t dx[D / 16], dy[D / 16];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    dx[kk] = dx0 + static_cast<uint64_t>(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
    dy[kk] = dy0 + static_cast<uint64_t>(((kk >> 2) * (kPsR * 128) + (kk & 3) * 32) >> 4);
  }
  mma_ss_n<D / 16>(d_tmem, dx, dy, idesc, 0u);
}

// d (+)= A Y: A a 128 x 64 16-bit operand packed in TMEM (K-step kk at
// a + 32 (kk / 2) + 8 (kk % 2)); Y a 64-row x D tile read as an MN-major B
// operand (its rows are the K dimension).
template <int D>
__device__ __forceinline__ void ps_mma_aY(uint32_t d_tmem, uint32_t a_tmem, uint32_t y_smem, uint32_t idesc,
                                          bool acc) {
  const uint64_t dy = sdesc_sw128(y_smem, kPsR * 128, 1024);
  uint32_t a[4];
  uint64_t b[4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    a[kk] = a_tmem + 32 * (kk >> 1) + 8 * (kk & 1);
    b[kk] = dy + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<4>(d_tmem, a, b, idesc, acc ? 1u : 0u);
}

template <bool BF>
__device__ __forceinline__ void ps_pack16(const float* x, uint32_t (&o)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = pack2<BF>(x[2 * e], x[2 * e + 1]);
}

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kPsThreads, 1)
    attn_bwd_pw_steps_kernel(const __grid_constant__ CUtensorMap tm_k1, const __grid_constant__ CUtensorMap tm_k2,
                             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q1,
                             const __grid_constant__ CUtensorMap tm_q2, const __grid_constant__ CUtensorMap tm_do,
                             const __grid_constant__ CUtensorMap tm_dv, const __grid_constant__ CUtensorMap tm_dk1,
                             const __grid_constant__ CUtensorMap tm_dk2, const BwdArgs args) {
  using C = PwStepCfg<D>;
  constexpr bool BF = DT<T>::bf16;
  constexpr int STAGES = C::STAGES;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_x, bar_y[STAGES], bar_yempty[STAGES];
  __shared__ __align__(8) uint64_t bar_s, bar_dp, bar_p, bar_ds, bar_consumed, bar_done;
  __shared__ __align__(16) float sRow[STAGES][2][kPsR];  // per streamed query: L * log2(e), delta
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ntiles = (args.N + kBN - 1) / kBN;
  int bh, kt;  // key tiles with the most queries (the first ones, causal) first
  if (!grouped_tile(blockIdx.x, args.BH, ntiles, kGroupHeads, &bh, &kt)) return;
  const int k0 = kt * kBN;
  const int first_q = args.causal ? max(0, k0 - args.P_SEQ) : 0;
  const int u0 = first_q / kPsR;
  const int tot = (args.M + kPsR - 1) / kPsR;
  const int nu = tot > u0 ? tot - u0 : 0;
  auto cls_of = [&](int u) { return pw_step_class((u0 + u) * kPsR, k0, args.P_SEQ, args.w); };

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto sX = [&](int i) { return base + i * C::XT; };  // K1, K2, V
  auto sY = [&](int st, int i) { return base + 3 * C::XT + st * C::STAGE + i * C::YT; };  // Q1, Q2, dO

  WaitCtl ctl{args.err, args.timeout_ns, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_x, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bar_y[s], 2);  // TMA bytes + the row constants
      mbar_init(&bar_yempty[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_p, kPsRowWarps);
    mbar_init(&bar_ds, kPsRowWarps);
    mbar_init(&bar_consumed, kPsRowWarps);
    mbar_init(&bar_done, 1);
    fence_mbar_init();
  }
  if (warp == kPsWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kPsWarpProducer) {
    // ------------------------------------------------------------ producer
    if (nu > 0) {
      if (lane == 0) {
        mbar_expect_tx(&bar_x, 3 * C::XT);
        ps_load<D>(sX(0), &tm_k1, &bar_x, k0, bh, C::XBLK);
        ps_load<D>(sX(1), &tm_k2, &bar_x, k0, bh, C::XBLK);
        ps_load<D>(sX(2), &tm_v, &bar_x, k0, bh, C::XBLK);
      }
      int issued = 0;
      for (int u = 0; u < nu; ++u) {
        const int st = u % STAGES;
        if (u >= STAGES && !warp_wait(&bar_yempty[st], ((u / STAGES) - 1) & 1, ctl, kErrTimeoutMma)) break;
        const int r0 = (u0 + u) * kPsR;
        if (lane == 0) {
          mbar_expect_tx(&bar_y[st], 3 * C::YT);
          ps_load<D>(sY(st, 0), &tm_q1, &bar_y[st], r0, bh, C::YBLK);
          ps_load<D>(sY(st, 1), &tm_q2, &bar_y[st], r0, bh, C::YBLK);
          ps_load<D>(sY(st, 2), &tm_do, &bar_y[st], r0, bh, C::YBLK);
        }
#pragma unroll
        for (int e = 0; e < kPsR / 32; ++e) {
          const int q = r0 + lane + 32 * e;
          const bool in = q < args.M;
          const size_t g = static_cast<size_t>(bh) * args.M + (in ? q : 0);
          sRow[st][0][lane + 32 * e] = in ? args.lse[g] * kLog2e : INFINITY;  // padding queries: P = 0
          sRow[st][1][lane + 32 * e] = in ? args.delta[g] : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_y[st]);
        issued = u + 1;
      }
      if (lane == 0) {  // never leave a TMA write in flight behind an early exit
        int zero = 0;
        WaitCtl drain{args.err, args.timeout_ns, reinterpret_cast<volatile int*>(&zero)};
        mbar_wait(&bar_x, 0, drain, kErrTimeoutTma);
        for (int u = issued - STAGES > 0 ? issued - STAGES : 0; u < issued; ++u)
          mbar_wait(&bar_y[u % STAGES], (u / STAGES) & 1, drain, kErrTimeoutTma);
      }
    }
  } else if (warp == kPsWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (nu > 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBM, kPsR, BF, false, false);  // M = keys, N = queries
      constexpr uint32_t idesc_g = idesc_f16(kBM, D, BF, false, true);      // M = keys, N = D
      const uint32_t xk1 = smem_u32(sX(0)), xk2 = smem_u32(sX(1)), xv = smem_u32(sX(2));
      auto ys = [&](int st, int i) { return smem_u32(sY(st, i)); };
      // S^T of step u: the near product (or the far one when the step is
      // wholly far) into the S buffer; a straddling step's far product into
      // the dP buffer
      auto scores_s = [&](int u, int st) {
        const int cls = cls_of(u);
        if (cls == kPsFar) ps_mma_xyT<D>(tmem + C::COL_S, xk2, ys(st, 1), idesc_s);
        else ps_mma_xyT<D>(tmem + C::COL_S, xk1, ys(st, 0), idesc_s);
        if (cls == (kPsNear | kPsFar)) ps_mma_xyT<D>(tmem + C::COL_DP, xk2, ys(st, 1), idesc_s);
        commit_el(&bar_s);
      };
      auto scores_dp = [&](int st) {  // dP^T = V dO^T
        ps_mma_xyT<D>(tmem + C::COL_DP, xv, ys(st, 2), idesc_s);
        commit_el(&bar_dp);
      };
      bool ok = warp_wait(&bar_x, 0, ctl, kErrTimeoutTma) && warp_wait(&bar_y[0], 0, ctl, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        scores_s(0, 0);
        if (cls_of(0) != (kPsNear | kPsFar)) scores_dp(0);
      }
      bool acc1 = false, acc2 = false;
      int nboth = 0;  // straddling steps so far (phases of bar_consumed)
      for (int u = 0; ok && u < nu; ++u) {
        const int st = u % STAGES, st1 = (u + 1) % STAGES;
        const bool more = u + 1 < nu;
        const int cls = cls_of(u);
        const int cls1 = more ? cls_of(u + 1) : 0;
        if (cls == (kPsNear | kPsFar)) {  // dP^T once S(q2, k2) has left the dP buffer
          if (!(ok = warp_wait(&bar_consumed, nboth & 1, ctl, kErrTimeoutSoftmax))) break;
          tc_fence_after();
          ++nboth;
          scores_dp(st);
        }
        if (!(ok = warp_wait(&bar_p, u & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        ps_mma_aY<D>(tmem + C::COL_DV, tmem + C::COL_S, ys(st, 2), idesc_g, u > 0);  // dV += P^T dO
        // The next step's scores go out under this step's dS phase when
        // neither step needs the S buffer's other columns or the dP buffer.
        const bool early = more && cls != (kPsNear | kPsFar) && cls1 != (kPsNear | kPsFar);
        if (early) {
          if (!(ok = warp_wait(&bar_y[st1], ((u + 1) / STAGES) & 1, ctl, kErrTimeoutTma))) break;
          tc_fence_after();
          scores_s(u + 1, st1);
        }
        if (!(ok = warp_wait(&bar_ds, u & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        if (cls & kPsNear) {
          ps_mma_aY<D>(tmem + C::COL_DK1, tmem + C::COL_DP, ys(st, 0), idesc_g, acc1);  // dK1 += dS_near^T Q1
          acc1 = true;
        }
        if (cls & kPsFar) {
          const uint32_t src = (cls == kPsFar) ? C::COL_DP : C::COL_S + 16;
          ps_mma_aY<D>(tmem + C::COL_DK2, tmem + src, ys(st, 1), idesc_g, acc2);  // dK2 += dS_far^T Q2
          acc2 = true;
        }
        commit_el(&bar_yempty[st]);
        if (more) {
          if (!early) {
            if (!(ok = warp_wait(&bar_y[st1], ((u + 1) / STAGES) & 1, ctl, kErrTimeoutTma))) break;
            tc_fence_after();
            scores_s(u + 1, st1);
          }
          if (cls1 != (kPsNear | kPsFar)) scores_dp(st1);
        }
      }
      if (ok) commit_el(&bar_done);
    }
  } else {
    // ------------------------------------------------- element-wise phase
    const int h = warp >> 2;                 // half of the step's 64 queries
    const int row = (warp & 3) * 32 + lane;  // TMEM lane: this thread's key within the tile
    const int j = k0 + row;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    bool ok = true;
    bool touched1 = false, touched2 = false;
    for (int u = 0; u < nu; ++u) {
      const int st = u % STAGES;
      const int r0 = (u0 + u) * kPsR;
      const int c0 = r0 + 32 * h;  // query of this thread's column 0
      const int cls = cls_of(u);
      touched1 |= (cls & kPsNear) != 0;
      touched2 |= (cls & kPsFar) != 0;
      if (!(ok = warp_wait(&bar_y[st], (u / STAGES) & 1, ctl, kErrTimeoutTma))) break;
      if (!(ok = warp_wait(&bar_s, u & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld_x32(lane_addr + C::COL_S + 32 * h, sr);
      tmem_ld_wait(sr);
      // far iff query c0 + e is at distance >= w from key j: e >= fl
      const int fl = j + args.w - args.P_SEQ - c0;
      if (cls == (kPsNear | kPsFar)) {
        uint32_t s2[32];
        tmem_ld_x32(lane_addr + C::COL_DP + 32 * h, s2);
        tmem_ld_wait(s2);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e >= fl) sr[e] = s2[e];
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_consumed);  // the dP buffer may take dP^T
      }
      float p[32];
      const float4* L4 = reinterpret_cast<const float4*>(&sRow[st][0][32 * h]);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 l4 = L4[c4];
        p[4 * c4 + 0] = ex2(fmaf(__uint_as_float(sr[4 * c4 + 0]), args.scale_log2, -l4.x));
        p[4 * c4 + 1] = ex2(fmaf(__uint_as_float(sr[4 * c4 + 1]), args.scale_log2, -l4.y));
        p[4 * c4 + 2] = ex2(fmaf(__uint_as_float(sr[4 * c4 + 2]), args.scale_log2, -l4.z));
        p[4 * c4 + 3] = ex2(fmaf(__uint_as_float(sr[4 * c4 + 3]), args.scale_log2, -l4.w));
      }
      if (args.causal) {  // key j is visible from query c0 + e iff e >= j - P_SEQ - c0
        const int lo = j - args.P_SEQ - c0;
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e < lo) p[e] = 0.f;
      }
      // P^T for dV, as soon as it exists
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk[8];
        ps_pack16<BF>(&p[16 * cc], pk);
        tmem_st_x8(lane_addr + C::COL_S + 32 * h + 8 * cc, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p);
      if (!(ok = warp_wait(&bar_dp, u & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      uint32_t dpr[32];
      tmem_ld_x32(lane_addr + C::COL_DP + 32 * h, dpr);
      tmem_ld_wait(dpr);
      const float4* D4 = reinterpret_cast<const float4*>(&sRow[st][1][32 * h]);
      float ds[32];
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4) {
        const float4 d4 = D4[c4];
        ds[4 * c4 + 0] = p[4 * c4 + 0] * (__uint_as_float(dpr[4 * c4 + 0]) - d4.x);
        ds[4 * c4 + 1] = p[4 * c4 + 1] * (__uint_as_float(dpr[4 * c4 + 1]) - d4.y);
        ds[4 * c4 + 2] = p[4 * c4 + 2] * (__uint_as_float(dpr[4 * c4 + 2]) - d4.z);
        ds[4 * c4 + 3] = p[4 * c4 + 3] * (__uint_as_float(dpr[4 * c4 + 3]) - d4.w);
      }
      if (cls == (kPsNear | kPsFar)) {  // near part into the dP buffer, far part beside P^T
        float dn[32], df[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const bool far = e >= fl;
          dn[e] = far ? 0.f : ds[e];
          df[e] = far ? ds[e] : 0.f;
        }
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pn[8], pf[8];
          ps_pack16<BF>(&dn[16 * cc], pn);
          ps_pack16<BF>(&df[16 * cc], pf);
          tmem_st_x8(lane_addr + C::COL_DP + 32 * h + 8 * cc, pn);
          tmem_st_x8(lane_addr + C::COL_S + 16 + 32 * h + 8 * cc, pf);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[8];
          ps_pack16<BF>(&ds[16 * cc], pk);
          tmem_st_x8(lane_addr + C::COL_DP + 32 * h + 8 * cc, pk);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ds);
    }
    // ------------------------------------------------------------ epilogue
    if (nu > 0 && ok) ok = warp_wait(&bar_done, 0, ctl, kErrTimeoutMma);
    tc_fence_after();
    const bool live = ok && nu > 0;
    // dV, dK1 and dK2 (x sm_scale), rounded, are staged over the K1, K2 and
    // V tiles (free: every MMA has finished) in the output maps' swizzled box
    // layout and written by TMA stores, which clip rows past N and columns
    // past D.  An output that no step touched is zero.
    auto stage_out = [&](int slot, uint32_t col, bool touched, float scale) {
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = h * (D / 64) + cc;  // this thread's 32-column chunks of the row
        uint32_t v[32];
        if (live && touched) {
          tmem_ld_x32(lane_addr + col + 32 * c, v);
          tmem_ld_wait(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        stage_row_chunk_sw128<BF>(smem_u32(sX(slot)), row, c, v, scale);
      }
    };
    stage_out(0, C::COL_DV, true, 1.f);
    stage_out(1, C::COL_DK1, touched1, args.sm_scale);
    stage_out(2, C::COL_DK2, touched2, args.sm_scale);
    fence_proxy_async_smem();
    named_bar_sync(1, kPsRowWarps * 32);
    if (warp == 0 && lane == 0 && k0 < args.N) {
#pragma unroll
      for (int kb = 0; kb < D / 64; ++kb) {
        tma_store_3d(&tm_dv, sX(0) + kb * C::XBLK, kb * 64, k0, bh);
        tma_store_3d(&tm_dk1, sX(1) + kb * C::XBLK, kb * 64, k0, bh);
        tma_store_3d(&tm_dk2, sX(2) + kb * C::XBLK, kb * 64, k0, bh);
      }
      tma_store_commit_and_wait_read();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kPsWarpMma) tmem_dealloc(tmem, 512);
}

bool bwd_pw_steps_supported(int D) { return D == 128; }

template <typename T>
static cudaError_t launch_pw_steps_t(const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  using C = PwStepCfg<128>;
  auto kern = attn_bwd_pw_steps_kernel<T, 128>;
  static std::atomic<bool> attr[kMaxDevices];
  cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
  if (e_attr != cudaSuccess) return e_attr;
  const long long blocks = static_cast<long long>(a.BH) * ((a.N + kBN - 1) / kBN);
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  if (blocks == 0) return cudaSuccess;
  kern<<<static_cast<unsigned>(blocks), kPsThreads, C::SMEM, s>>>(m.k, m.k2, m.v, m.q64, m.q264, m.dO64, m.dv,
                                                                  m.dk, m.dk2, a);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pw_steps(bool bf16, const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  return bf16 ? launch_pw_steps_t<__nv_bfloat16>(m, a, s) : launch_pw_steps_t<__half>(m, a, s);
}

}  // namespace ta

TA_GUARD_ACCESSOR(bwd_pw_steps)
