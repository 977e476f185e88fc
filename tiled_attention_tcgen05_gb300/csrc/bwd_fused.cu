// Fused attention backward for sm_103a (tcgen05 + TMA): dK, dV and dQ from one
// key-stationary pass, five matmuls per (key, query) pair.
//
// Page sources: "Triton fused attention tutorial, updated with JVP support",
// _attn_bwd (one program computes dK/dV of its key block and dQ of its query
// block), _attn_bwd_dkdv (pT = exp2(qkT - m), dv += pT do, dpT = v do^T,
// dsT = pT (dpT - Di), dk += dsT q), _attn_bwd_dq (dq += ds k, dq *= ln 2
// with its pre-scaled k: here dq *= sm_scale) and the comment thread's fix
// (non-causal tiles run over the full range).
//
// The pages' dQ pass recomputes S and dP for every (query, key) block pair
// that the dK/dV pass has already formed.  Here the key-stationary CTA also
// forms the pair's dQ contribution, dQ^T += K^T dS^T over its 128 keys, and
// adds it into an fp32 accumulator in global memory; a small pass then
// scales the sum by sm_scale and rounds it to the element type.  A pair
// therefore costs five matmuls (S^T, dP^T, dV, dK, dQ^T) instead of seven
// (S^T, dP^T, dV, dK and S, dP, dQ again).
//
// One CTA per 128-key tile walks its queries in steps of 64.  TMEM (512
// columns) holds, per step, S^T (64 fp32 columns), dP^T (64, overwritten in
// place by P^T and dS^T in 16 bits), dQ^T (64: 128 feature lanes x 64
// queries) and, for the whole CTA, V as the A operand of dP^T (64 packed
// columns), dV and dK (128 each).  64-query steps are what make room for a
// dQ^T buffer of its own beside S^T and dP^T; with 128-query steps those
// alone fill TMEM with dV and dK.
//
// 448 threads:
//   warps 0-7   key-row softmax gradient: TMEM lane = key, warp / 4 selects
//               which 32 of the step's 64 queries the thread handles; P^T and
//               dS^T go back into TMEM for dV and dK, dS^T also into shared
//               memory (double-buffered) for the dQ^T MMA;
//   warps 8-11  dQ drain: TMEM lane = feature d; each reads its 32 lanes of
//               dQ^T (64 values a thread) and adds them to the accumulator
//               with warp-coalesced red.global.add.f32 (one 128-byte line per
//               instruction);
//   warp 12     TMA producer (lane 0: K, V and the Q ring; lane 1: dO ring);
//   warp 13     TMEM allocator and MMA issuer.
// MMA order for step s:
//   S^T(s + 1) | dK(s) dV(s) | dP^T(s + 1) | dQ^T(s)
// S^T(s + 1) starts as soon as the softmax warps hold S^T(s) in registers,
// and dQ^T(s) runs while they form dS(s + 1).
//
// The accumulator is summed with atomics, so dQ's fp32 summation order (and
// possibly its last bit after rounding) varies from run to run.
#include "bwd_common.cuh"
#include "common.cuh"
#include "launch.h"

namespace ta {

namespace {

constexpr int kQS = 64;  // queries per streamed step
constexpr int kFThreads = 448;
constexpr int kFRowWarps = 8;  // softmax warps 0-7
constexpr int kFDrain0 = 8;    // drain warps 8-11
constexpr int kFDrainWarps = 4;
constexpr int kFWarpProducer = 12;
constexpr int kFWarpMma = 13;

template <int D>
struct FusedCfg {
  static constexpr int BLK = kBN * 128;    // one 64-column block of a 128-row tile (16 KB)
  static constexpr int SBLK = kQS * 128;   // one 64-column block of a 64-row step tile (8 KB)
  static constexpr int TILE_K = (D / 64) * BLK;
  static constexpr int TILE_S = (D / 64) * SBLK;
  static constexpr int DS_BYTES = kBN * 128;  // dS^T of a step: 128 key rows x 64 queries
  static constexpr int QST = 4;  // Q ring depth (steps)
  static constexpr int OST = 4;  // dO ring depth
  static constexpr int V_OFF = TILE_K;
  static constexpr int DS_OFF = 2 * TILE_K;  // two dS^T buffers
  static constexpr int Q_OFF = DS_OFF + 2 * DS_BYTES;
  static constexpr int O_OFF = Q_OFF + QST * TILE_S;
  static constexpr int LD_OFF = O_OFF + OST * TILE_S;  // L / delta: [buffer][group][L, delta][32] floats
  static constexpr int LD_BYTES = 2 * 2 * 2 * 32 * 4;
  static constexpr int BAR_OFF = LD_OFF + LD_BYTES;
  static constexpr int NBARS = 2 + 2 * QST + 2 * OST + 13 + 4;
  static constexpr int BAR_BYTES = 8 * NBARS + 8;
  static constexpr int USED = BAR_OFF + BAR_BYTES;
  static constexpr int PAD = (kSmemMax - USED) < 1023 ? (kSmemMax - USED) : 1023;  // alignment allowance
  static constexpr int SMEM = USED + PAD;
  static constexpr uint32_t COL_S = 0, COL_P = 64, COL_Q = 128, COL_V = 192, COL_DV = 256, COL_DK = 256 + D;
  static_assert(D == 128, "the fused backward is built for D = 128");
  static_assert(PAD >= 0 && SMEM <= kSmemMax, "tiles do not fit in shared memory");
  static_assert(COL_DK + D <= 512, "TMEM overflow");
};

__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// A 64-row step tile (D columns, two 64-column blocks 8 KB apart).
template <int D>
__device__ __forceinline__ void load_step(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row0, int bh) {
#pragma unroll
  for (int kb = 0; kb < D / 64; ++kb) tma_load_3d(dst + kb * (kQS * 128), map, bar, kb * 64, row0, bh);
}

// S^T = K Q^T over D: A = K (128 rows, K-major), B = Q of the step (64 rows,
// K-major); M = 128 keys, N = 64 queries.
template <int D>
__device__ __forceinline__ void mma_sT(uint32_t d_tmem, uint32_t k_smem, uint32_t q_smem, uint32_t idesc) {
  const uint64_t da = sdesc_sw128(k_smem, 16, 1024);
  const uint64_t db = sdesc_sw128(q_smem, 16, 1024);
  uint64_t a[D / 16], b[D / 16];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    a[kk] = da + static_cast<uint64_t>(((kk >> 2) * (kBN * 128) + (kk & 3) * 32) >> 4);
    b[kk] = db + static_cast<uint64_t>(((kk >> 2) * (kQS * 128) + (kk & 3) * 32) >> 4);
  }
  mma_ss_n<D / 16>(d_tmem, a, b, idesc, 0u);
}

// dP^T = V dO^T over D: A = V in TMEM (8 packed columns per K-step), B = dO
// of the step (64 rows, K-major).
template <int D>
__device__ __forceinline__ void mma_dpT(uint32_t d_tmem, uint32_t v_tmem, uint32_t o_smem, uint32_t idesc) {
  const uint64_t db = sdesc_sw128(o_smem, 16, 1024);
  uint32_t a[D / 16];
  uint64_t b[D / 16];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    a[kk] = v_tmem + 8 * kk;
    b[kk] = db + static_cast<uint64_t>(((kk >> 2) * (kQS * 128) + (kk & 3) * 32) >> 4);
  }
  mma_ts_n<D / 16>(d_tmem, a, b, idesc, 0u);
}

// d (+)= X Y over the two K-steps (16 queries each) of query group G (the
// step's queries 32 G .. 32 G + 31): X = P^T or dS^T in TMEM, group G's 16
// packed columns at x + 32 G (K-step 2 G + i at + 8 i); Y = dO or Q of the
// step read MN-major (K = query rows, N = D in two 64-column blocks 8 KB
// apart).  The first MMA accumulates iff `accumulate`.
template <int G>
__device__ __forceinline__ void mma_grad(uint32_t d_tmem, uint32_t x_tmem, uint32_t y_smem, uint32_t idesc,
                                         bool accumulate) {
  const uint64_t dy = sdesc_sw128(y_smem, kQS * 128, 1024);
  uint32_t a[2];
  uint64_t b[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int kk = 2 * G + i;
    a[i] = x_tmem + 32 * G + 8 * i;
    b[i] = dy + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<2>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}

// dQ^T = K^T dS^T over the tile's 128 keys: A = K read MN-major (M = feature
// d in two 64-column blocks 16 KB apart, K = key), B = dS^T of the step read
// MN-major (K = key, N = the step's 64 queries in one 128-byte row); a K-step
// of 16 keys advances 16 rows (2048 bytes) in both.
__device__ __forceinline__ void mma_dqT(uint32_t d_tmem, uint32_t k_smem, uint32_t ds_smem, uint32_t idesc) {
  const uint64_t da = sdesc_sw128(k_smem, kBN * 128, 1024);
  const uint64_t db = sdesc_sw128(ds_smem, kBN * 128, 1024);
  uint64_t a[8], b[8];
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint64_t off = static_cast<uint64_t>((kk * 16 * 128) >> 4);
    a[kk] = da + off;
    b[kk] = db + off;
  }
  mma_ss_n<8>(d_tmem, a, b, idesc, 0u);
}

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kFThreads, 1)
    attn_bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                          const BwdArgs args) {
  using C = FusedCfg<D>;
  constexpr bool BF = DT<T>::bf16;
  constexpr int QST = C::QST, OST = C::OST;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (base - smem_raw > C::PAD) {  // uniform across the CTA: nothing has been touched yet
    if (threadIdx.x == 0 && args.err) atomicOr(args.err, kErrSmemLayout);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::BAR_OFF);
  uint64_t& bar_kv = bars[0];        // K and V in shared memory
  uint64_t& bar_vt = bars[1];        // V copied into TMEM
  uint64_t* bar_qf = bars + 2;
  uint64_t* bar_qe = bar_qf + QST;
  uint64_t* bar_of = bar_qe + QST;
  uint64_t* bar_oe = bar_of + OST;
  uint64_t* bt = bar_oe + OST;       // per-step barriers
  uint64_t& bar_s = bt[0];           // S^T(s) in TMEM
  uint64_t& bar_consumed = bt[1];    // softmax holds S^T(s): its columns are free
  uint64_t& bar_dp = bt[2];          // dP^T(s) in TMEM
  uint64_t* bar_ds = bt + 3;         // [query group]: P^T / dS^T(s) in TMEM
  uint64_t* bar_dss = bt + 5;        // [buffer]: dS^T(s) in shared memory
  uint64_t* bar_dq = bt + 7;         // [buffer]: dQ^T(s) in TMEM (and every earlier MMA done)
  uint64_t& bar_drained = bt[9];     // drain warps hold dQ^T(s): its columns are free
  uint64_t& bar_done = bt[10];       // every MMA done
  uint64_t* bar_pub = bt + 13;       // [buffer * 2 + group]: L / delta of a step stored
  uint32_t& tmem_slot = *reinterpret_cast<uint32_t*>(bars + C::NBARS);
  int& abort_flag = *(reinterpret_cast<int*>(bars + C::NBARS) + 1);
  float* sLD = reinterpret_cast<float*>(base + C::LD_OFF);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int bh, kt;  // key tiles with the most queries (the first ones, causal) first
  if (!grouped_tile(blockIdx.x, args.BH, (args.N + kBN - 1) / kBN, kGroupHeads, &bh, &kt)) return;
  const int k0 = kt * kBN;
  const int num_steps = (args.M + kQS - 1) / kQS;
  int s0 = 0;  // first step that sees one of the tile's keys
  if (args.causal && k0 - args.P_SEQ > 0) s0 = (k0 - args.P_SEQ) / kQS;
  const int ns = num_steps > s0 ? num_steps - s0 : 0;

  uint8_t* sK = base;
  uint8_t* sV = base + C::V_OFF;
  auto sDS = [&](int b) { return base + C::DS_OFF + b * C::DS_BYTES; };
  auto sQ = [&](int i) { return base + C::Q_OFF + i * C::TILE_S; };
  auto sDO = [&](int i) { return base + C::O_OFF + i * C::TILE_S; };

  WaitCtl ctl{args.err, args.timeout_ns, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_kv, 1);
    mbar_init(&bar_vt, 4);
    for (int i = 0; i < QST; ++i) {
      mbar_init(&bar_qf[i], 1);
      mbar_init(&bar_qe[i], 1);
    }
    for (int i = 0; i < OST; ++i) {
      mbar_init(&bar_of[i], 1);
      mbar_init(&bar_oe[i], 1);
    }
    mbar_init(&bar_s, 1);
    mbar_init(&bar_consumed, kFRowWarps);
    mbar_init(&bar_dp, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_ds[i], kFRowWarps / 2);
      mbar_init(&bar_dss[i], kFRowWarps);
      mbar_init(&bar_dq[i], 1);
    }
    mbar_init(&bar_drained, kFDrainWarps);
    mbar_init(&bar_done, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&bar_pub[i], kFRowWarps / 2);
    fence_mbar_init();
  }
  if (warp == kFWarpMma) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == kFWarpProducer) {
    // ---------------------- producer: lane 0 K, V and the Q ring; lane 1 the dO ring
    if (lane < 2 && ns > 0) {
      const bool is_q = (lane == 0);
      const int depth = is_q ? QST : OST;
      uint64_t* full = is_q ? bar_qf : bar_of;
      uint64_t* empty = is_q ? bar_qe : bar_oe;
      const CUtensorMap* map = is_q ? &tm_q : &tm_do;
      if (is_q) {
        mbar_expect_tx(&bar_kv, 2 * C::TILE_K);
        load_tile_b<D>(sK, &tm_k, &bar_kv, k0, bh);
        load_tile_b<D>(sV, &tm_v, &bar_kv, k0, bh);
      }
      int issued = 0;
      for (int s = 0; s < ns; ++s) {
        const int st = s % depth;
        if (s >= depth && !mbar_wait(&empty[st], ((s / depth) - 1) & 1, ctl, kErrTimeoutMma)) break;
        mbar_expect_tx(&full[st], C::TILE_S);
        load_step<D>(is_q ? sQ(st) : sDO(st), map, &full[st], (s0 + s) * kQS, bh);
        issued = s + 1;
      }
      int zero = 0;
      WaitCtl drain{args.err, args.timeout_ns, reinterpret_cast<volatile int*>(&zero)};
      if (is_q) mbar_wait(&bar_kv, 0, drain, kErrTimeoutTma);
      for (int s = issued - depth > 0 ? issued - depth : 0; s < issued; ++s)
        mbar_wait(&full[s % depth], (s / depth) & 1, drain, kErrTimeoutTma);
    }
  } else if (warp == kFWarpMma) {
    // ----------------------------------------------------------------- MMA
    if (ns > 0) {
      constexpr uint32_t idesc_s = idesc_f16(kBN, kQS, BF, false, false);  // M = keys, N = queries
      constexpr uint32_t idesc_g = idesc_f16(kBN, D, BF, false, true);     // M = keys, N = D
      constexpr uint32_t idesc_q = idesc_f16(D, kQS, BF, true, true);      // M = D, N = queries
      bool ok = warp_wait(&bar_kv, 0, ctl, kErrTimeoutTma) && warp_wait(&bar_qf[0], 0, ctl, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        mma_sT<D>(tmem + C::COL_S, smem_u32(sK), smem_u32(sQ(0)), idesc_s);  // S^T = K Q^T
        commit_el(&bar_s);
      }
      ok = ok && warp_wait(&bar_vt, 0, ctl, kErrTimeoutSoftmax) && warp_wait(&bar_of[0], 0, ctl, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        mma_dpT<D>(tmem + C::COL_P, tmem + C::COL_V, smem_u32(sDO(0)), idesc_s);  // dP^T = V dO^T
        commit_el(&bar_dp);
      }
      for (int s = 0; ok && s < ns; ++s) {
        const int sq = s % QST, so = s % OST;
        if (s + 1 < ns) {  // S^T(s + 1) once the softmax warps hold S^T(s)
          if (!(ok = warp_wait(&bar_consumed, s & 1, ctl, kErrTimeoutSoftmax))) break;
          if (!(ok = warp_wait(&bar_qf[(s + 1) % QST], ((s + 1) / QST) & 1, ctl, kErrTimeoutTma))) break;
          tc_fence_after();
          mma_sT<D>(tmem + C::COL_S, smem_u32(sK), smem_u32(sQ((s + 1) % QST)), idesc_s);
          commit_el(&bar_s);
        }
        // dK += dS^T Q and dV += P^T dO, query group 0 as soon as its softmax
        // warps have formed it
        if (!(ok = warp_wait(&bar_ds[0], s & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        mma_grad<0>(tmem + C::COL_DK, tmem + C::COL_P + 16, smem_u32(sQ(sq)), idesc_g, s > 0);
        mma_grad<0>(tmem + C::COL_DV, tmem + C::COL_P, smem_u32(sDO(so)), idesc_g, s > 0);
        if (!(ok = warp_wait(&bar_ds[1], s & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        mma_grad<1>(tmem + C::COL_DK, tmem + C::COL_P + 16, smem_u32(sQ(sq)), idesc_g, true);
        commit_el(&bar_qe[sq]);
        mma_grad<1>(tmem + C::COL_DV, tmem + C::COL_P, smem_u32(sDO(so)), idesc_g, true);
        commit_el(&bar_oe[so]);
        if (s + 1 < ns) {  // dP^T(s + 1), its columns freed by dK(s), dV(s)
          const int so1 = (s + 1) % OST;
          if (!(ok = warp_wait(&bar_of[so1], ((s + 1) / OST) & 1, ctl, kErrTimeoutTma))) break;
          tc_fence_after();
          mma_dpT<D>(tmem + C::COL_P, tmem + C::COL_V, smem_u32(sDO(so1)), idesc_s);
          commit_el(&bar_dp);
        }
        // dQ^T(s): the drain holds dQ^T(s - 1), dS^T(s) is in shared memory
        if (s >= 1 && !(ok = warp_wait(&bar_drained, (s - 1) & 1, ctl, kErrTimeoutOther))) break;
        if (!(ok = warp_wait(&bar_dss[s & 1], (s >> 1) & 1, ctl, kErrTimeoutSoftmax))) break;
        tc_fence_after();
        mma_dqT(tmem + C::COL_Q, smem_u32(sK), smem_u32(sDS(s & 1)), idesc_q);
        commit_el(&bar_dq[s & 1]);
      }
      if (ok) commit_el(&bar_done);
    }
  } else if (warp >= kFDrain0 && warp < kFDrain0 + kFDrainWarps) {
    // ----------------------------------------------------------- dQ drain
    // Lane quadrant (warp % 4) holds features d = 32 (warp % 4) + lane; the
    // 64 columns are the step's queries.  A warp's 32 lanes cover 32
    // consecutive floats of one accumulator row: one 128-byte line per red.
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float* acc = args.dq_acc + static_cast<size_t>(bh) * args.M * D + (warp & 3) * 32 + lane;
    for (int s = 0; s < ns; ++s) {
      if (!warp_wait(&bar_dq[s & 1], (s >> 1) & 1, ctl, kErrTimeoutMma)) break;
      tc_fence_after();
      uint32_t v[64];
      tmem_ld_x32(lane_addr + C::COL_Q, TB_CHUNK(v, 0));
      tmem_ld_x32(lane_addr + C::COL_Q + 32, TB_CHUNK(v, 1));
      tmem_ld_wait(TB_CHUNK(v, 0));
      tmem_ld_wait(TB_CHUNK(v, 1));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_drained);  // dQ^T's columns are free for step s + 1
      const int q0 = (s0 + s) * kQS;
      float* row = acc + static_cast<size_t>(q0) * D;
      const int nrow = args.M - q0;  // rows of the step that exist
      if (!TA_CHECK(q0 >= 0 && q0 < args.M && bh < args.BH)) continue;
#pragma unroll
      for (int jr = 0; jr < kQS; ++jr)
        if (jr < nrow) red_add_f32(row + static_cast<size_t>(jr) * D, __uint_as_float(v[jr]));
    }
  } else if (warp < kFRowWarps) {
    // ------------------------------------------- key-row softmax gradient
    const int hc = warp >> 2;                // query group: the step's queries [32 hc, 32 hc + 32)
    const int j = k0 + (threadIdx.x & 127);  // this thread's key (epilogue row)
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const int m = lane & 3;
    // dS^T in shared memory: key row kr (= 32 (warp % 4) + 16 g + lane / 4,
    // and + 8), 16-byte chunk 4 hc + jq of the row swizzled with
    // (kr % 8) = lane / 4, bytes 4 m.. of the chunk.
    const uint32_t ds_row = ((warp & 3) * 32 + (lane >> 2)) * 128 + (m << 2);
    const int swz = lane >> 2;
    // V into TMEM (A operand of dP^T): group 0's 128 threads copy one row each.
    bool ok = true;
    if (hc == 0 && ns > 0) {
      ok = warp_wait(&bar_kv, 0, ctl, kErrTimeoutTma);
      if (ok) {
        tile_row_to_tmem<D>(sV, (warp & 3) * 32 + lane, lane_addr + C::COL_V);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_vt);
      }
    }
    // L and delta of the group's 32 queries: warp 0 of the group loads L,
    // warp 1 delta (one value a lane, coalesced) a step ahead, stores it once
    // the group is done with the current step and publishes the buffer on
    // bar_pub; the reads are then shared-memory broadcasts.  Queries past M
    // read L = +inf (P = 0) and delta = 0.
    const int ld_arr = warp & 3;  // 0: L, 1: delta, 2-3: nothing to load
    auto ld_fetch = [&](int s) -> float {
      if (ld_arr > 1) return 0.f;
      const int q = (s0 + s) * kQS + 32 * hc + lane;
      if (q >= args.M) return ld_arr ? 0.f : INFINITY;
      return __ldg((ld_arr ? args.delta : args.lse) + static_cast<size_t>(bh) * args.M + q);
    };
    auto ld_slot = [&](int s) { return sLD + ((s & 1) * 2 + hc) * 64; };
    if (ns > 0 && ok) {
      if (ld_arr <= 1) ld_slot(0)[ld_arr * 32 + lane] = ld_fetch(0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_pub[hc]);
    }
    for (int s = 0; ok && s < ns; ++s) {
      const int q0 = (s0 + s) * kQS;
      const int qb = q0 + 32 * hc;  // first query of this thread's columns
      const float pre = (s + 1 < ns) ? ld_fetch(s + 1) : 0.f;
      if (!(ok = warp_wait(&bar_s, s & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      // 16-lane shapes: in each 16-lane group g of its warp, thread t holds
      // keys (t / 4) and (t / 4 + 8) at the query pairs 8 jq + 2 m, +1
      // (m = t % 4) of the group.  sv[16 g + 4 jq + e], e = {(k, q), (k, q + 1),
      // (k + 8, q), (k + 8, q + 1)}.
      uint32_t sv[32];
      tmem_ld_16x256b_x4(lane_addr + C::COL_S + 32 * hc, TB_CHUNK16(sv, 0));
      tmem_ld_16x256b_x4(lane_addr + (16u << 16) + C::COL_S + 32 * hc, TB_CHUNK16(sv, 1));
      tmem_ld_wait(TB_CHUNK16(sv, 0));
      tmem_ld_wait(TB_CHUNK16(sv, 1));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_consumed);  // S^T's columns free for S^T(s + 1)
      if (!(ok = warp_wait(&bar_pub[(s & 1) * 2 + hc], (s >> 1) & 1, ctl, kErrTimeoutSoftmax))) break;
      const float* sL = ld_slot(s) + 2 * m;
      const float* sD = sL + 32;
      const float2 sc2 = make_float2(args.scale_log2, args.scale_log2);
      float p[32];
#pragma unroll
      for (int jq = 0; jq < 4; ++jq) {
        const float2 l2 = *reinterpret_cast<const float2*>(sL + 8 * jq);
        const float2 nl = fmul2(l2, make_float2(-kLog2e, -kLog2e));
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          const int i = 16 * g + 4 * jq;
          const float2 y0 = ffma2(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), sc2, nl);
          const float2 y1 = ffma2(make_float2(__uint_as_float(sv[i + 2]), __uint_as_float(sv[i + 3])), sc2, nl);
          p[i + 0] = ex2(y0.x);
          p[i + 1] = ex2(y0.y);
          p[i + 2] = ex2(y1.x);
          p[i + 3] = ex2(y1.y);
        }
      }
      if (args.causal && k0 + kBN - 1 > qb + args.P_SEQ) {  // key k visible from q iff q >= k - P_SEQ
        // element (g, jq, e) is masked iff 8 jq + (e & 1) < lo + 16 g + 8 (e >> 1)
        const int lo = k0 + 32 * (warp & 3) + (lane >> 2) - args.P_SEQ - qb - 2 * m;
#pragma unroll
        for (int g = 0; g < 2; ++g)
#pragma unroll
          for (int jq = 0; jq < 4; ++jq)
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (8 * jq + (e & 1) < lo + 16 * g + 8 * (e >> 1)) p[16 * g + 4 * jq + e] = 0.f;
      }
      if (!(ok = warp_wait(&bar_dp, s & 1, ctl, kErrTimeoutMma))) break;
      // dS^T buffer s % 2 was last read by dQ^T(s - 2)
      if (s >= 2 && !(ok = warp_wait(&bar_dq[s & 1], ((s >> 1) - 1) & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      // read dP^T, write P^T and dS^T (16 packed columns each, pair 4 jq + m)
      // back into the group's 32 columns, and dS^T into shared memory
      uint32_t dp[32];  // [g][16]
      tmem_ld_16x256b_x4(lane_addr + C::COL_P + 32 * hc, TB_CHUNK16(dp, 0));
      tmem_ld_16x256b_x4(lane_addr + (16u << 16) + C::COL_P + 32 * hc, TB_CHUNK16(dp, 1));
      tmem_ld_wait(TB_CHUNK16(dp, 0));
      tmem_ld_wait(TB_CHUNK16(dp, 1));
      float2 nd2[4];  // -delta of the thread's query pairs
#pragma unroll
      for (int jq = 0; jq < 4; ++jq) {
        const float2 d2 = *reinterpret_cast<const float2*>(sD + 8 * jq);
        nd2[jq] = make_float2(-d2.x, -d2.y);
      }
      const uint32_t dsb = smem_u32(sDS(s & 1)) + ds_row;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint32_t pp[8], pd[8];
#pragma unroll
        for (int jq = 0; jq < 4; ++jq) {
          const int i = 16 * g + 4 * jq;
          pp[2 * jq] = pack2<BF>(p[i], p[i + 1]);
          pp[2 * jq + 1] = pack2<BF>(p[i + 2], p[i + 3]);
          const float2 s0v = fmul2(make_float2(p[i], p[i + 1]),
                                   fadd2(make_float2(__uint_as_float(dp[i]), __uint_as_float(dp[i + 1])), nd2[jq]));
          const float2 s1v = fmul2(make_float2(p[i + 2], p[i + 3]),
                                   fadd2(make_float2(__uint_as_float(dp[i + 2]), __uint_as_float(dp[i + 3])), nd2[jq]));
          pd[2 * jq] = pack2<BF>(s0v.x, s0v.y);
          pd[2 * jq + 1] = pack2<BF>(s1v.x, s1v.y);
        }
        const uint32_t ga = lane_addr + (static_cast<uint32_t>(16 * g) << 16) + C::COL_P + 32 * hc;
        tmem_st_16x128b_x4(ga, pp);
        tmem_st_16x128b_x4(ga + 16, pd);
#pragma unroll
        for (int jq = 0; jq < 4; ++jq) {
          const uint32_t a = dsb + g * (16 * 128) + (((4 * hc + jq) ^ swz) << 4);
          sts_b32(a, pd[2 * jq]);
          sts_b32(a + 8 * 128, pd[2 * jq + 1]);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_smem();  // dS^T stores -> visible to the dQ^T MMA
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bar_ds[hc]);    // the group's P^T / dS^T are in place
        mbar_arrive(&bar_dss[s & 1]);
      }
      if (s + 1 < ns) {  // every warp of the group is past step s - 1, the buffer's previous step
        if (ld_arr <= 1) ld_slot(s + 1)[ld_arr * 32 + lane] = pre;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar_pub[((s + 1) & 1) * 2 + hc]);
      }
    }
    // ------------------------------------------------------------ epilogue
    if (ns > 0 && ok) ok = warp_wait(&bar_done, 0, ctl, kErrTimeoutMma);
    tc_fence_after();
    const bool st_row = j < args.N;
    const size_t off = (static_cast<size_t>(bh) * args.N + (st_row ? j : 0)) * args.dg;
    T* dvp = reinterpret_cast<T*>(args.dv) + off;
    T* dkp = reinterpret_cast<T*>(args.dk) + off;
    const int dc = hc * (D / 2);
    if (ok && ns > 0) {
      epilogue_half<T, D>(lane_addr + C::COL_DV, dvp, dc, st_row, true, 1.f, args.dg);
      epilogue_half<T, D>(lane_addr + C::COL_DK, dkp, dc, st_row, true, args.sm_scale, args.dg);
    } else if (st_row) {
      zero_half<T, D>(dvp, dc, args.dg);
      zero_half<T, D>(dkp, dc, args.dg);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kFWarpMma) tmem_dealloc(tmem, 512);
}

template <typename T, int D>
static cudaError_t launch_fused_t(const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  using C = FusedCfg<D>;
  auto kern = attn_bwd_fused_kernel<T, D>;
  static std::atomic<bool> attr[kMaxDevices];
  cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
  if (e_attr != cudaSuccess) return e_attr;
  const long long blocks = static_cast<long long>(a.BH) * ((a.N + kBN - 1) / kBN);
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(blocks), kFThreads, C::SMEM, s>>>(m.q, m.k, m.v, m.dO, a);
  return cudaGetLastError();
}

bool bwd_fused_supported(int D) { return D == 128; }

int bwd_fused_step_rows() { return kQS; }

cudaError_t launch_bwd_fused(bool bf16, int D, const BwdMaps& m, const BwdArgs& a, cudaStream_t s) {
  if (D == 128) return bf16 ? launch_fused_t<__nv_bfloat16, 128>(m, a, s) : launch_fused_t<__half, 128>(m, a, s);
  return cudaErrorNotSupported;
}

}  // namespace ta

TA_GUARD_ACCESSOR(bwd_fused)
