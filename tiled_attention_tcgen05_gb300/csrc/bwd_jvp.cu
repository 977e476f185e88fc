// Backward of the forward-mode JVP for sm_103a (tcgen05 + TMA): the
// gradients of <dO, O> + <dtO, tO> with respect to q, k and v, where O and
// tO are the outputs of the JVP forward of "Triton fused attention tutorial,
// updated with JVP support" (_attn_fwd_inner with ENABLE_JVP and the _attn_fwd
// JVP epilogue).  The page stops at the forward; this is the chain rule taken
// back through its steps.  Per (query i, key j), with P = exp(S - L),
// T = sm_scale (tq k^T + q tk^T), mu = tL = rowsum(P o T) and two per-query
// constants eps = <dtO, O> and delta2 = <dO, O> + <dtO, tO>:
//   dtP = dtO V^T,            dPa = dO V^T + dtO tV^T,
//   dT  = P o (dtP - eps),    dS  = P o (dPa - delta2) + (T - mu) o dT,
//   tP  = P o (T - mu),
//   dQ = sm_scale (dS K + dT tK),  dK = sm_scale (dS^T Q + dT^T tQ),
//   dV = P^T dO + tP^T dtO.
// The tangents' own gradients are the plain backward with dO replaced by
// dtO (tO is linear in the tangents): dtq = sm_scale dT K, dtk = sm_scale
// dT^T Q, dtv = P^T dtO.  These kernels accumulate them too (TANG) where
// TMEM has room: dtK and dtV at D <= 64, dtQ at every D; otherwise the plain
// backward's key-stationary kernel computes dtK and dtV.
//
// Two kernels from one template, each one CTA per 128-row stationary tile,
// 320 threads:
//   KEYS = true  (dK, dV): stationary K, tK, V, tV; streamed 64-query steps
//                of Q, tQ, dO, dtO; TMEM lane = key.
//   KEYS = false (dQ):     stationary Q, tQ, dO, dtO; streamed 64-key steps
//                of K, tK, V, tV; TMEM lane = query.
//   warps 0-7  element-wise phase; warp % 4 selects the 32-lane quarter and
//              warp / 4 the half of the step's 64 columns;
//   warp 8     TMA producer (and, for KEYS, the per-query constants);
//   warp 9     TMEM allocator and MMA issuer (the whole warp; one elected
//              lane issues each K-loop of MMAs as a single asm block).
//
// TMEM (512 columns): four fp32 score buffers of 64 columns (S, T, dtP, dPa)
// and the fp32 accumulators from column 256 (dV, dK[, dtV, dtK] or
// dQ[, dtQ]).  The 16-bit MMA operands are written back in place: a thread
// packs its 32 columns into the first 16 columns of its own 32-column slice,
// so K-step kk (16 streamed rows) of an operand sits at column
// 32 (kk / 2) + 8 (kk % 2) of its buffer.
// Operands: P and tP (KEYS only) in the S and T buffers, dS and dT in the
// dtP and dPa buffers.  The next step's S and T go into their buffers as
// soon as those are free, under the current step's element-wise work.
#include "bwd_common.cuh"
#include "common.cuh"
#include "launch.h"

namespace ta {

constexpr int kJvpThreads = 320;
constexpr int kJvpWarpProducer = 8;
constexpr int kJvpWarpMma = 9;
constexpr int kJvpRowWarps = 8;
constexpr int kJR = 64;  // rows of a streamed step

template <int D>
struct JvpBwdCfg {
  static constexpr int XBLK = kBM * 128;  // one 64-column block of a 128-row tile (bytes)
  static constexpr int YBLK = kJR * 128;  // one 64-column block of a 64-row tile
  static constexpr int XT = (D / 64) * XBLK;
  static constexpr int YT = (D / 64) * YBLK;
  static constexpr int STAGE = 4 * YT;
  static constexpr int STATIC_RESERVE = 8 * 1024;  // barriers and the per-stage query constants
  static constexpr int FIT = (kSmemMax - STATIC_RESERVE - 1024 - 4 * XT) / STAGE;
  static constexpr int STAGES = FIT > 4 ? 4 : FIT;
  static constexpr int SMEM = 4 * XT + STAGES * STAGE + 1024;
  static constexpr uint32_t COL_S = 0, COL_T = 64, COL_DTP = 128, COL_DPA = 192, COL_ACC = 256;
  static_assert(STAGES >= 1, "tiles do not fit in shared memory");
  static_assert(COL_ACC + 2 * D <= 512, "TMEM overflow");
};

// The tangents' gradients fit beside the others: dV, dK, dtV, dtK (4 D
// accumulator columns) in the key-stationary kernel, dQ, dtQ (2 D) in the
// query-stationary one.
template <int D, bool KEYS>
constexpr bool jvp_tangents_fit() { return 256 + (KEYS ? 4 : 2) * D <= 512; }

template <int D>
__device__ __forceinline__ void jvp_load(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row0, int bh,
                                         int blk) {
#pragma unroll
  for (int kb = 0; kb < D / 64; ++kb) tma_load_3d(dst + kb * blk, map, bar, kb * 64, row0, bh);
}

// d (+)= X Y^T over D: X a 128-row tile, Y a 64-row tile, both K-major with
// 128-byte swizzle in 64-column blocks.
template <int D>
__device__ __forceinline__ void mma_xyT(uint32_t d_tmem, uint32_t x_smem, uint32_t y_smem, uint32_t idesc,
                                        uint32_t acc) {
  const uint64_t dx0 = sdesc_sw128(x_smem, 16, 1024);
  const uint64_t dy0 = sdesc_sw128(y_smem, 16, 1024);
  uint64_t dx[D / 16], dy[D / 16];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    dx[kk] = dx0 + static_cast<uint64_t>(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
    dy[kk] = dy0 + static_cast<uint64_t>(((kk >> 2) * (kJR * 128) + (kk & 3) * 32) >> 4);
  }
  mma_ss_n<D / 16>(d_tmem, dx, dy, idesc, acc);
}

// d (+)= A Y: A is a 128 x 64 16-bit operand in TMEM (K-step kk at column
// a + 32 (kk / 2) + 8 (kk % 2)); Y a 64-row x D tile read as an MN-major B
// operand (its rows are the K dimension).
template <int D>
__device__ __forceinline__ void mma_aY(uint32_t d_tmem, uint32_t a_tmem, uint32_t y_smem, uint32_t idesc,
                                       uint32_t acc) {
  const uint64_t dy = sdesc_sw128(y_smem, kJR * 128, 1024);
  uint32_t a[4];
  uint64_t b[4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    a[kk] = a_tmem + 32 * (kk >> 1) + 8 * (kk & 1);
    b[kk] = dy + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<4>(d_tmem, a, b, idesc, acc);
}

template <bool BF>
__device__ __forceinline__ void pack16(const float* x, uint32_t (&o)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = pack2<BF>(x[2 * e], x[2 * e + 1]);
}

template <typename T, bool KEYS, int D, bool TANG>
__global__ void __launch_bounds__(kJvpThreads, 1)
    attn_bwd_jvp_kernel(const __grid_constant__ CUtensorMap tx0, const __grid_constant__ CUtensorMap tx1,
                        const __grid_constant__ CUtensorMap tx2, const __grid_constant__ CUtensorMap tx3,
                        const __grid_constant__ CUtensorMap ty0, const __grid_constant__ CUtensorMap ty1,
                        const __grid_constant__ CUtensorMap ty2, const __grid_constant__ CUtensorMap ty3,
                        const __grid_constant__ CUtensorMap tz0, const __grid_constant__ CUtensorMap tz1,
                        const __grid_constant__ CUtensorMap tz2, const __grid_constant__ CUtensorMap tz3,
                        const BwdArgs args) {
  using C = JvpBwdCfg<D>;
  constexpr bool BF = DT<T>::bf16;
  constexpr int STAGES = C::STAGES;
  static_assert(!TANG || jvp_tangents_fit<D, KEYS>(), "no TMEM room for the tangents' gradients");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_x, bar_y[STAGES], bar_yempty[STAGES];
  __shared__ __align__(8) uint64_t bar_s, bar_dp, bar_p, bar_sfree, bar_ops, bar_done;
  // KEYS: per streamed query, L log2(e), mu, eps, delta2
  __shared__ __align__(16) float sRow[KEYS ? STAGES : 1][4][kJR];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int x_len = KEYS ? args.N : args.M;  // rows of the stationary tensors
  const int ntiles = (x_len + kBM - 1) / kBM;
  int bh, rank;
  if (!grouped_tile(blockIdx.x, args.BH, ntiles, kGroupHeads, &bh, &rank)) return;
  const int xt = KEYS ? rank : ntiles - 1 - rank;  // heaviest causal tiles first
  const int x0 = xt * kBM;
  // streamed steps u0 .. u0 + nu - 1 (64 rows each)
  int u0 = 0, nu = 0;
  if constexpr (KEYS) {
    const int first_q = args.causal ? max(0, x0 - args.P_SEQ) : 0;
    u0 = first_q / kJR;
    const int tot = (args.M + kJR - 1) / kJR;
    nu = tot > u0 ? tot - u0 : 0;
  } else {
    int last_k = args.N - 1;
    if (args.causal) last_k = min(last_k, x0 + kBM - 1 + args.P_SEQ);
    nu = last_k < 0 ? 0 : last_k / kJR + 1;
  }

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto sX = [&](int i) { return base + i * C::XT; };
  auto sY = [&](int st, int i) { return base + 4 * C::XT + st * C::STAGE + i * C::YT; };

  WaitCtl ctl{args.err, args.timeout_ns, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_x, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bar_y[s], KEYS ? 2 : 1);  // TMA bytes (+ the query constants)
      mbar_init(&bar_yempty[s], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_dp, 1);
    mbar_init(&bar_p, kJvpRowWarps);
    mbar_init(&bar_sfree, kJvpRowWarps);
    mbar_init(&bar_ops, kJvpRowWarps);
    mbar_init(&bar_done, 1);
    fence_mbar_init();
  }
  if (warp == kJvpWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kJvpWarpProducer) {
    // ------------------------------------------------------------ producer
    if (nu > 0) {
      if (lane == 0) {
        mbar_expect_tx(&bar_x, 4 * C::XT);
        jvp_load<D>(sX(0), &tx0, &bar_x, x0, bh, C::XBLK);
        jvp_load<D>(sX(1), &tx1, &bar_x, x0, bh, C::XBLK);
        jvp_load<D>(sX(2), &tx2, &bar_x, x0, bh, C::XBLK);
        jvp_load<D>(sX(3), &tx3, &bar_x, x0, bh, C::XBLK);
      }
      int issued = 0;
      for (int u = 0; u < nu; ++u) {
        const int st = u % STAGES;
        if (u >= STAGES) {
          if (!warp_wait(&bar_yempty[st], ((u / STAGES) - 1) & 1, ctl, kErrTimeoutMma)) break;
        }
        const int r0 = (u0 + u) * kJR;
        if (lane == 0) {
          mbar_expect_tx(&bar_y[st], 4 * C::YT);
          jvp_load<D>(sY(st, 0), &ty0, &bar_y[st], r0, bh, C::YBLK);
          jvp_load<D>(sY(st, 1), &ty1, &bar_y[st], r0, bh, C::YBLK);
          jvp_load<D>(sY(st, 2), &ty2, &bar_y[st], r0, bh, C::YBLK);
          jvp_load<D>(sY(st, 3), &ty3, &bar_y[st], r0, bh, C::YBLK);
        }
        if constexpr (KEYS) {
#pragma unroll
          for (int e = 0; e < kJR / 32; ++e) {
            const int q = r0 + lane + 32 * e;
            const bool in = q < args.M;
            const size_t g = static_cast<size_t>(bh) * args.M + (in ? q : 0);
            sRow[st][0][lane + 32 * e] = in ? args.lse[g] * kLog2e : INFINITY;  // padding queries: P = 0
            sRow[st][1][lane + 32 * e] = in ? args.mu[g] : 0.f;
            sRow[st][2][lane + 32 * e] = in ? args.eps[g] : 0.f;
            sRow[st][3][lane + 32 * e] = in ? args.delta[g] : 0.f;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_y[st]);
        }
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
  } else if (warp == kJvpWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (nu > 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBM, kJR, BF, false, false);  // M = stationary, N = streamed
      constexpr uint32_t idesc_g = idesc_f16(kBM, D, BF, false, true);     // M = stationary, N = D
      const uint32_t xs0 = smem_u32(sX(0)), xs1 = smem_u32(sX(1)), xs2 = smem_u32(sX(2)), xs3 = smem_u32(sX(3));
      bool ok = warp_wait(&bar_x, 0, ctl, kErrTimeoutTma);
      auto ys = [&](int st, int i) { return smem_u32(sY(st, i)); };
      // S = X0 Y0^T; T = X1 Y0^T + X0 Y1^T (K Q^T, tK Q^T + K tQ^T, or Q K^T, tQ K^T + Q tK^T)
      auto scores_st = [&](int st) {
        mma_xyT<D>(tmem + C::COL_S, xs0, ys(st, 0), idesc_s, 0u);
        mma_xyT<D>(tmem + C::COL_T, xs1, ys(st, 0), idesc_s, 0u);
        mma_xyT<D>(tmem + C::COL_T, xs0, ys(st, 1), idesc_s, 1u);
        commit_el(&bar_s);
      };
      // dtP = V dtO^T (or dtO V^T); dPa = V dO^T + tV dtO^T (or dO V^T + dtO tV^T)
      auto scores_dp = [&](int st) {
        if constexpr (KEYS) mma_xyT<D>(tmem + C::COL_DTP, xs2, ys(st, 3), idesc_s, 0u);
        else mma_xyT<D>(tmem + C::COL_DTP, xs3, ys(st, 2), idesc_s, 0u);
        mma_xyT<D>(tmem + C::COL_DPA, xs2, ys(st, 2), idesc_s, 0u);
        mma_xyT<D>(tmem + C::COL_DPA, xs3, ys(st, 3), idesc_s, 1u);
        commit_el(&bar_dp);
      };
      // With two or more stages the next step's S and T are issued as soon as
      // their buffers are free (after dV's MMAs read P and tP, or once the dQ
      // kernel's threads hold S and T in registers), so they run under the
      // element-wise phase; with one stage its data arrives only after the
      // current step's last MMA.
      constexpr bool kEarly = STAGES >= 2;
      if (ok) ok = warp_wait(&bar_y[0], 0, ctl, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        scores_st(0);
        scores_dp(0);
      }
      for (int u = 0; ok && u < nu; ++u) {
        const int st = u % STAGES, st1 = (u + 1) % STAGES;
        const bool more = u + 1 < nu;
        const uint32_t first = u > 0 ? 1u : 0u;
        if constexpr (KEYS) {
          if (!(ok = warp_wait(&bar_p, u & 1, ctl, kErrTimeoutSoftmax))) break;
          tc_fence_after();
          mma_aY<D>(tmem + C::COL_ACC, tmem + C::COL_S, ys(st, 2), idesc_g, first);  // dV += P^T dO
          mma_aY<D>(tmem + C::COL_ACC, tmem + C::COL_T, ys(st, 3), idesc_g, 1u);     // dV += tP^T dtO
          if constexpr (TANG) mma_aY<D>(tmem + C::COL_ACC + 2 * D, tmem + C::COL_S, ys(st, 3), idesc_g, first);  // dtV
        } else if constexpr (kEarly) {
          if (!(ok = warp_wait(&bar_sfree, u & 1, ctl, kErrTimeoutSoftmax))) break;
          tc_fence_after();
        }
        if (kEarly && more) {
          if (!(ok = warp_wait(&bar_y[st1], ((u + 1) / STAGES) & 1, ctl, kErrTimeoutTma))) break;
          tc_fence_after();
          scores_st(st1);
        }
        if (!(ok = warp_wait(&bar_ops, u & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        // dS and dT sit in the dtP and dPa buffers
        if constexpr (KEYS) {
          mma_aY<D>(tmem + C::COL_ACC + D, tmem + C::COL_DTP, ys(st, 0), idesc_g, first);  // dK += dS^T Q
          mma_aY<D>(tmem + C::COL_ACC + D, tmem + C::COL_DPA, ys(st, 1), idesc_g, 1u);     // dK += dT^T tQ
          if constexpr (TANG) mma_aY<D>(tmem + C::COL_ACC + 3 * D, tmem + C::COL_DPA, ys(st, 0), idesc_g, first);  // dtK
        } else {
          mma_aY<D>(tmem + C::COL_ACC, tmem + C::COL_DTP, ys(st, 0), idesc_g, first);  // dQ += dS K
          mma_aY<D>(tmem + C::COL_ACC, tmem + C::COL_DPA, ys(st, 1), idesc_g, 1u);     // dQ += dT tK
          if constexpr (TANG) mma_aY<D>(tmem + C::COL_ACC + D, tmem + C::COL_DPA, ys(st, 0), idesc_g, first);  // dtQ
        }
        commit_el(&bar_yempty[st]);
        if (more) {
          if (!kEarly) {
            if (!(ok = warp_wait(&bar_y[st1], ((u + 1) / STAGES) & 1, ctl, kErrTimeoutTma))) break;
            tc_fence_after();
            scores_st(st1);
          }
          scores_dp(st1);
        }
      }
      if (ok) commit_el(&bar_done);
    }
  } else {
    // ------------------------------------------------- element-wise phase
    const int h = warp >> 2;                  // half of the step's 64 columns
    const int row = (warp & 3) * 32 + lane;   // TMEM lane
    const int xr = x0 + row;                  // this thread's key (KEYS) or query
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float rLc = 0.f, rMu = 0.f, rEps = 0.f, rDel = 0.f;  // the dQ kernel's per-query constants
    if constexpr (!KEYS) {
      const bool in = xr < args.M;
      const size_t g = static_cast<size_t>(bh) * args.M + (in ? xr : 0);
      rLc = in ? args.lse[g] * kLog2e : INFINITY;
      rMu = in ? args.mu[g] : 0.f;
      rEps = in ? args.eps[g] : 0.f;
      rDel = in ? args.delta[g] : 0.f;
    }
    bool ok = true;
    for (int u = 0; u < nu; ++u) {
      const int st = u % STAGES;
      const int r0 = (u0 + u) * kJR;  // first streamed row of the step
      const int c0 = r0 + 32 * h;     // streamed row of this thread's column 0
      if constexpr (KEYS) {
        if (!(ok = warp_wait(&bar_y[st], (u / STAGES) & 1, ctl, kErrTimeoutTma))) break;
      }
      if (!(ok = warp_wait(&bar_s, u & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      uint32_t sr[32], tr[32];
      tmem_ld_x32(lane_addr + C::COL_S + 32 * h, sr);
      tmem_ld_x32(lane_addr + C::COL_T + 32 * h, tr);
      tmem_ld_wait(sr);
      tmem_ld_wait(tr);
      if constexpr (!KEYS) {  // S and T are in registers: their buffers may take the next step's
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_sfree);
      }
      float p[32], tm[32];  // P and T - mu of the thread's 32 columns
      if constexpr (KEYS) {
        const float4* L4 = reinterpret_cast<const float4*>(&sRow[st][0][32 * h]);
        const float4* M4 = reinterpret_cast<const float4*>(&sRow[st][1][32 * h]);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 l4 = L4[c4], m4 = M4[c4];
          const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, mv[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            p[4 * c4 + e] = ex2(fmaf(__uint_as_float(sr[4 * c4 + e]), args.scale_log2, -lv[e]));
            tm[4 * c4 + e] = fmaf(__uint_as_float(tr[4 * c4 + e]), args.sm_scale, -mv[e]);
          }
        }
        // causal: key xr is visible from query c0 + e iff e >= xr - P_SEQ - c0
        if (args.causal) {
          const int lo = xr - args.P_SEQ - c0;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e < lo) p[e] = 0.f;
        }
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          p[e] = ex2(fmaf(__uint_as_float(sr[e]), args.scale_log2, -rLc));
          tm[e] = fmaf(__uint_as_float(tr[e]), args.sm_scale, -rMu);
        }
        // key c0 + e exists and (causal) is visible from query xr
        int hi = args.N - 1 - c0;
        if (args.causal) hi = min(hi, xr + args.P_SEQ - c0);
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (e > hi) p[e] = 0.f;
      }
      if constexpr (KEYS) {  // P^T and tP^T for dV, as soon as they exist
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float tp[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) tp[e] = p[16 * cc + e] * tm[16 * cc + e];
          uint32_t pk[8], tk[8];
          pack16<BF>(&p[16 * cc], pk);
          pack16<BF>(tp, tk);
          tmem_st_x8(lane_addr + C::COL_S + 32 * h + 8 * cc, pk);
          tmem_st_x8(lane_addr + C::COL_T + 32 * h + 8 * cc, tk);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_p);
      }
      if (!(ok = warp_wait(&bar_dp, u & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dtp[16], dpa[16];
        tmem_ld_x16(lane_addr + C::COL_DTP + 32 * h + 16 * cc, dtp);
        tmem_ld_x16(lane_addr + C::COL_DPA + 32 * h + 16 * cc, dpa);
        tmem_ld_wait(dtp);
        tmem_ld_wait(dpa);
        float dT[16], dS[16];
        if constexpr (KEYS) {
          const float4* E4 = reinterpret_cast<const float4*>(&sRow[st][2][32 * h + 16 * cc]);
          const float4* D4 = reinterpret_cast<const float4*>(&sRow[st][3][32 * h + 16 * cc]);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const float4 e4 = E4[c4], d4 = D4[c4];
            const float ev[4] = {e4.x, e4.y, e4.z, e4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = 4 * c4 + e, k = 16 * cc + i;
              dT[i] = p[k] * (__uint_as_float(dtp[i]) - ev[e]);
              dS[i] = fmaf(tm[k], dT[i], p[k] * (__uint_as_float(dpa[i]) - dv[e]));
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int k = 16 * cc + i;
            dT[i] = p[k] * (__uint_as_float(dtp[i]) - rEps);
            dS[i] = fmaf(tm[k], dT[i], p[k] * (__uint_as_float(dpa[i]) - rDel));
          }
        }
        uint32_t pks[8], pkt[8];
        pack16<BF>(dS, pks);
        pack16<BF>(dT, pkt);
        tmem_st_x8(lane_addr + C::COL_DTP + 32 * h + 8 * cc, pks);
        tmem_st_x8(lane_addr + C::COL_DPA + 32 * h + 8 * cc, pkt);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_ops);
    }
    // ------------------------------------------------------------ epilogue
    if (nu > 0 && ok) ok = warp_wait(&bar_done, 0, ctl, kErrTimeoutMma);
    tc_fence_after();
    const bool live = ok && nu > 0;
    // The outputs (KEYS: dV, dK, then dtV, dtK; else dQ, then dtQ), rounded,
    // are staged over the stationary tiles (free: every MMA has finished) in
    // the output maps' swizzled box layout and written by TMA stores, which
    // clip rows past the tensor and columns past D.
    auto stage_out = [&](int slot, uint32_t col, float scale) {
#pragma unroll
      for (int cc = 0; cc < D / 64; ++cc) {
        const int c = h * (D / 64) + cc;  // this thread's 32-column chunks of the row
        uint32_t v[32];
        if (live) {
          tmem_ld_x32(lane_addr + col + 32 * c, v);
          tmem_ld_wait(v);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        stage_row_chunk_sw128<BF>(smem_u32(sX(slot)), row, c, v, scale);
      }
    };
    constexpr int NOUT = KEYS ? (TANG ? 4 : 2) : (TANG ? 2 : 1);
    if constexpr (KEYS) {
      stage_out(0, C::COL_ACC, 1.f);
      stage_out(1, C::COL_ACC + D, args.sm_scale);
      if constexpr (TANG) {
        stage_out(2, C::COL_ACC + 2 * D, 1.f);
        stage_out(3, C::COL_ACC + 3 * D, args.sm_scale);
      }
    } else {
      stage_out(0, C::COL_ACC, args.sm_scale);
      if constexpr (TANG) stage_out(1, C::COL_ACC + D, args.sm_scale);
    }
    fence_proxy_async_smem();
    named_bar_sync(1, kJvpRowWarps * 32);
    if (warp == 0 && lane == 0 && x0 < x_len) {
      const CUtensorMap* outs[4] = {&tz0, &tz1, &tz2, &tz3};
#pragma unroll
      for (int o = 0; o < NOUT; ++o)
#pragma unroll
        for (int kb = 0; kb < D / 64; ++kb) tma_store_3d(outs[o], sX(o) + kb * C::XBLK, kb * 64, x0, bh);
      tma_store_commit_and_wait_read();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kJvpWarpMma) tmem_dealloc(tmem, 512);
}

template <typename T, bool KEYS, int D>
static cudaError_t launch_jvp_bwd_t(const JvpBwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  using C = JvpBwdCfg<D>;
  auto kern = attn_bwd_jvp_kernel<T, KEYS, D, jvp_tangents_fit<D, KEYS>()>;
  static std::atomic<bool> attr[kMaxDevices];
  cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
  if (e_attr != cudaSuccess) return e_attr;
  const int rows = KEYS ? a.N : a.M;
  const long long blocks = static_cast<long long>(a.BH) * ((rows + kBM - 1) / kBM);
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  if (blocks == 0) return cudaSuccess;
  if constexpr (KEYS) {
    kern<<<static_cast<unsigned>(blocks), kJvpThreads, C::SMEM, s>>>(m.k128, m.tk128, m.v128, m.tv128, m.q64,
                                                                      m.tq64, m.do64, m.dto64, m.dv, m.dk, m.dtv,
                                                                      m.dtk, a);
  } else {
    kern<<<static_cast<unsigned>(blocks), kJvpThreads, C::SMEM, s>>>(m.q128, m.tq128, m.do128, m.dto128, m.k64,
                                                                      m.tk64, m.v64, m.tv64, m.dq, m.dtq, m.dq,
                                                                      m.dq, a);
  }
  return cudaGetLastError();
}

bool bwd_jvp_has_tangents(bool keys, int D) {
  if (keys) return D == 64 ? jvp_tangents_fit<64, true>() : jvp_tangents_fit<128, true>();
  return D == 64 ? jvp_tangents_fit<64, false>() : jvp_tangents_fit<128, false>();
}

cudaError_t launch_bwd_jvp(bool keys, bool bf16, int D, const JvpBwdMaps& m, const BwdArgs& a, cudaStream_t s) {
#define TA_JVP_BWD(K_, D_) \
  if (keys == K_ && D == D_)   \
    return bf16 ? launch_jvp_bwd_t<__nv_bfloat16, K_, D_>(m, a, s) : launch_jvp_bwd_t<__half, K_, D_>(m, a, s);
  TA_JVP_BWD(true, 64)
  TA_JVP_BWD(true, 128)
  TA_JVP_BWD(false, 64)
  TA_JVP_BWD(false, 128)
#undef TA_JVP_BWD
  return cudaErrorNotSupported;
}

}  // namespace ta

TA_GUARD_ACCESSOR(bwd_jvp)
