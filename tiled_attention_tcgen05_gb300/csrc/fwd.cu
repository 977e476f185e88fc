// Forward attention kernels for sm_103a: TMA-fed K/V ring, tcgen05 MMAs with
// TMEM accumulators, one softmax thread per query row.
//
// One CTA owns one 128-row query tile of one (batch, head) and walks the key
// tiles the causal / ragged schedule allows.  Warp roles (192 threads):
//   warps 0-3  softmax + correction + epilogue; thread r owns query row r,
//              which is TMEM lane r (tcgen05.ld 32x32b shape), so row max and
//              row sum need no shuffles;
//   warp 4     TMA producer (Q once, then a STAGES-deep ring of K/V tiles);
//   warp 5     TMEM allocator and MMA issuer (the whole warp; one elected lane
//              issues each K-loop of MMAs as a single asm block).
// Per key tile t:  S = Q K_t^T (tcgen05.mma, A and B from shared memory) ->
// softmax writes P (16-bit, packed two per TMEM column) over S -> O += P V_t
// with P read straight from TMEM.  The standard and piecewise modes
// double-buffer S so the next QK^T overlaps the current softmax; a piecewise
// tile that needs both score products puts S(q2, k2) in a third buffer.
//
// Page sources: "Triton fused attention tutorial, updated with JVP support",
// _attn_fwd / _attn_fwd_inner (online exp2 softmax with running max and sum,
// acc = acc * alpha + P V, epilogue M = m + log2 l, O = acc / l; JVP branch:
// t_qk = t_q k^T + q t_k^T, p_tqk = p * t_qk * sm_scale, mu, g_acc, p_tv_acc
// and t_O = g_acc / l - (mu / l) O + p_tv_acc / l); "FlagAttention
// piecewise.py", _fwd_kernel (piecewise_mask choosing q2 k2^T or q1 k1^T,
// causal mask P_SEQ + i >= j, empty rows O = 0, L = -inf, natural-log L).
//
// Departures from the pages' design, all result-preserving: P lives in TMEM
// instead of registers/shared memory; the running maximum is raised lazily
// (only when it grows by more than 2^8), so O is rescaled rarely; the
// tangent accumulators g_acc and p_tv_acc are one TMEM accumulator U; and
// piecewise tiles whose keys are all near (or all far) run one QK^T MMA
// instead of two.
#include <cstdio>

#include "cluster.cuh"
#include "common.cuh"
#include "launch.h"

namespace ta {

template <int MODE, int D>
struct FwdCfg {
  static constexpr int KB = D / 64;       // 64-column (128-byte) swizzle blocks per row
  static constexpr int BLK = kBM * 128;   // bytes of one 128-row x 64-column block
  static constexpr int TILE = KB * BLK;   // bytes of one 128 x D tile
  static constexpr int NQ = (MODE == kStd) ? 1 : 2;   // resident query-like tiles
  static constexpr int NKT = (MODE == kStd) ? 1 : 2;  // key-like tiles per stage
  static constexpr int NVT = (MODE == kJvp) ? 2 : 1;  // value-like tiles per stage
  static constexpr int STAGE = (NKT + NVT) * TILE;
  static constexpr int RESERVE = 2048;    // alignment slack + static shared memory
  static constexpr int ST_FIT = (kSmemMax - RESERVE - NQ * TILE) / STAGE;
  static constexpr int STAGES = ST_FIT > 4 ? 4 : ST_FIT;
  // Two S buffers let QK^T(t + 1) run before P V(t); that needs a second
  // K/V stage (tile t + 1's keys arrive while tile t's values are in use).
  // The JVP at D = 64 (JVP2) double-buffers S and keeps T in a buffer of its
  // own: S0 | S1 | T | O | U fill the 512 columns.  P goes over the first 64
  // columns of its S buffer and P o T over the other 64, so T's columns are
  // free once the softmax has read T, and T(t + 1) is computed while the
  // softmax still works on tile t.  At D = 128 the JVP keeps one S buffer
  // (S | T | O | U) and writes P o T over T.
  static constexpr bool JVP2 = (MODE == kJvp && D == 64);
  static constexpr int NBUF = ((MODE == kJvp && !JVP2) || STAGES < 2) ? 1 : 2;
  static constexpr int SMEM = NQ * TILE + STAGES * STAGE + 1024;
  static constexpr uint32_t COL_S0 = 0;    // S (buffer 0) | jvp S
  static constexpr uint32_t COL_S1 = 128;  // S (buffer 1) | jvp (D = 128) T
  static constexpr uint32_t COL_T = JVP2 ? 256 : 128;  // jvp T
  static constexpr uint32_t COL_O = JVP2 ? 384 : 256;
  static constexpr uint32_t COL_U = COL_O + D;  // jvp tangent accumulator
  static constexpr uint32_t COL_X = 256 + D;  // piecewise: S(q2, k2) of a tile that needs both products
  static_assert(STAGES >= 1, "tile does not fit in shared memory");
  static_assert(!JVP2 || STAGES >= 2, "the JVP's second S buffer needs a second K/V stage");
  static_assert(COL_U + (MODE == kJvp ? D : 0) <= 512, "TMEM overflow");
  static_assert(MODE != kPiecewise || COL_X + 128 <= 512, "TMEM overflow");
};

enum : int { kNear = 1, kFar = 2 };

// Which score products a piecewise tile needs: far iff i + P_SEQ - j >= w.
__device__ __forceinline__ int pw_class(int q0, int k0, int P_SEQ, int w) {
  const long long lo = (long long)q0 + P_SEQ - k0 - w;  // smallest i - j + P_SEQ - w
  const long long hi = lo + (kBM - 1);                  // largest
  if (lo >= kBN - 1) return kFar;   // every column c <= i + P_SEQ - k0 - w
  if (hi < 0) return kNear;
  return kNear | kFar;
}

template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row0, int bh) {
#pragma unroll
  for (int kb = 0; kb < D / 64; ++kb) tma_load_3d(dst + kb * (kBM * 128), map, bar, kb * 64, row0, bh);
}

// d = A B^T over the head dimension: A, B are 128 x D K-major swizzled tiles.
// The descriptors are built once; each K-step adds its byte offset / 16 to
// the 14-bit start-address field (shared addresses stay below 256 KB, so the
// add never carries out of the field).
template <int D>
__device__ __forceinline__ void mma_qk(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, uint32_t idesc,
                                       bool accumulate) {
  const uint64_t da0 = sdesc_sw128(a_smem, 16, 1024);
  const uint64_t db0 = sdesc_sw128(b_smem, 16, 1024);
  uint64_t da[D / 16], db[D / 16];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * (kBM * 128) + (kk & 3) * 32) >> 4);
    da[kk] = da0 + off;
    db[kk] = db0 + off;
  }
  mma_ss_n<D / 16>(d_tmem, da, db, idesc, accumulate ? 1u : 0u);
}

// d (+)= P V: P is 128 x 128 (16-bit, TMEM), V is 128 keys x D stored with D
// contiguous (MN-major B operand; 64-column blocks kBM*128 bytes apart).
template <int D>
__device__ __forceinline__ void mma_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem, uint32_t idesc,
                                       bool accumulate) {
  const uint64_t dv = sdesc_sw128(v_smem, kBM * 128, 1024);
  uint32_t a[kBN / 16];
  uint64_t b[kBN / 16];
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk) {
    a[kk] = p_tmem + kk * 8;
    b[kk] = dv + static_cast<uint64_t>((kk * 16 * 128) >> 4);
  }
  mma_ts_n<kBN / 16>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}

// Stores the first 8 * ng (ng <= 4) of 32 fp32 values (x scale) as T.
template <typename T>
__device__ __forceinline__ void store_row_chunk(T* dst, const float* v32, float scale, int ng = 4) {
  constexpr bool BF = DT<T>::bf16;
  if (!TA_CHECK((reinterpret_cast<uintptr_t>(dst) & 15u) == 0u && ng >= 0 && ng <= 4)) return;
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack2<BF>(v32[8 * q + 0] * scale, v32[8 * q + 1] * scale);
    u.y = pack2<BF>(v32[8 * q + 2] * scale, v32[8 * q + 3] * scale);
    u.z = pack2<BF>(v32[8 * q + 4] * scale, v32[8 * q + 5] * scale);
    u.w = pack2<BF>(v32[8 * q + 6] * scale, v32[8 * q + 7] * scale);
    if (q < ng) d4[q] = u;
  }
}

#define TA_CHUNK(arr, c) (*reinterpret_cast<uint32_t(*)[32]>(&(arr)[32 * (c)]))

// Key split (SPLIT): the kernel runs as clusters of two CTAs per query tile.
// The first CTA of a pair takes the tile's first ceil(n/2) key tiles, the
// second the rest; at the end the second CTA leaves its raw state (running
// maximum m, sum l, JVP mu, and the unnormalised O and U rows) in its own
// shared memory and the first CTA reads it over distributed shared memory and
// combines the two online-softmax states before its epilogue:
//   m = max(m0, m1), a_i = 2^(m_i - m), l = a0 l0 + a1 l1, O = a0 O0 + a1 O1
// (mu and U like l and O), which is the rescale the softmax applies between
// key tiles, applied once between the two halves.  Layout of the hand-over
// area (the second CTA's dynamic shared memory, free once its last MMA is
// done): m, l, mu as float[128] each, then O and U as float4 [D/32 chunks]
// [8 quads][128 rows], so a warp's stores and loads are contiguous.
constexpr int kSplitHdr = 2048;

template <typename T, int MODE, int D, bool SPLIT>
__device__ __forceinline__ void fwd1_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                          const CUtensorMap& tm_q2, const CUtensorMap& tm_k2,
                                          const CUtensorMap& tm_v2, const FwdArgs& args) {
  using C = FwdCfg<MODE, D>;
  constexpr bool BF = DT<T>::bf16;
  constexpr int STAGES = C::STAGES;
  constexpr int NBUF = C::NBUF;
  constexpr int NACC = (MODE == kJvp) ? 2 : 1;  // accumulators handed over: O (and U)
  static_assert(!SPLIT || kSplitHdr + NACC * D * 512 <= C::SMEM - 1024, "hand-over area does not fit");
  // each CTA takes all 512 TMEM columns: the two CTAs of a pair must sit on
  // different SMs, which more than half an SM's shared memory guarantees
  static_assert(!SPLIT || C::SMEM > kSmemMax / 2, "the CTAs of a pair could share an SM");

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q;
  __shared__ __align__(8) uint64_t bar_k[STAGES], bar_v[STAGES], bar_empty[STAGES];
  __shared__ __align__(8) uint64_t bar_s[NBUF], bar_p[NBUF];
  __shared__ __align__(8) uint64_t bar_o, bar_ofinal;
  __shared__ __align__(8) uint64_t bar_peer;  // SPLIT: the second CTA's state is ready (first CTA's copy)
  __shared__ __align__(8) uint64_t bar_t, bar_tfree;  // JVP2: T(t) computed / T(t) read by the softmax
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int part = SPLIT ? static_cast<int>(blockIdx.y & 1) : 0;  // = rank in the (1, 2, 1) cluster
  const int qt = args.num_q_tiles - 1 - static_cast<int>(SPLIT ? blockIdx.y >> 1 : blockIdx.y);  // heaviest first
  if (!TA_CHECK(bh < args.BH && qt >= 0 && qt < args.num_q_tiles)) return;  // both CTAs of a pair alike
  const int q0 = qt * kBM;
  const int nkv_all = kv_tiles_for(q0, args.M, args.N, args.P_SEQ, args.causal);
  const int h_split = (nkv_all + 1) >> 1;
  const int t0 = (SPLIT && part) ? h_split : 0;  // first key tile of this CTA
  const int nkv = SPLIT ? (part ? nkv_all - h_split : h_split) : nkv_all;
  const int n_peer = (SPLIT && !part) ? nkv_all - h_split : 0;  // key tiles the partner CTA took

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                                  // Q | Q1 | Q  (+ Q2 | TQ)
  uint8_t* sStages = base + C::NQ * C::TILE;
  auto sKt = [&](int st, int i) { return sStages + st * C::STAGE + i * C::TILE; };
  auto sVt = [&](int st, int i) { return sStages + st * C::STAGE + (C::NKT + i) * C::TILE; };

  WaitCtl ctl{args.err, args.timeout_ns, &abort_flag};

  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bar_k[s], 1);
      mbar_init(&bar_v[s], 1);
      mbar_init(&bar_empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&bar_s[b], 1);
      mbar_init(&bar_p[b], 4);
    }
    mbar_init(&bar_o, 1);
    mbar_init(&bar_ofinal, 1);
    mbar_init(&bar_peer, kBM);
    mbar_init(&bar_t, 1);
    mbar_init(&bar_tfree, 4);
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (SPLIT) cluster_sync_all();  // the partner's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0 && nkv > 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int qrow = q0;
      mbar_expect_tx(&bar_q, C::NQ * C::TILE);
      load_tile<D>(sQ, &tm_q, &bar_q, qrow, bh);
      if constexpr (C::NQ == 2) load_tile<D>(sQ + C::TILE, &tm_q2, &bar_q, qrow, bh);
      uint32_t last_phase[STAGES];
      int used = 0;
      for (int t = 0; t < nkv; ++t) {
        const int st = t % STAGES;
        if (t >= STAGES) {
          if (!mbar_wait(&bar_empty[st], ((t / STAGES) - 1) & 1, ctl, kErrTimeoutMma)) break;
        }
        const int k0 = (t0 + t) * kBN;
        if constexpr (MODE == kStd) {
          mbar_expect_tx(&bar_k[st], C::TILE);
          load_tile<D>(sKt(st, 0), &tm_k, &bar_k[st], k0, bh);
          mbar_expect_tx(&bar_v[st], C::TILE);
          load_tile<D>(sVt(st, 0), &tm_v, &bar_v[st], k0, bh);
        } else if constexpr (MODE == kPiecewise) {
          const int cls = pw_class(q0, k0, args.P_SEQ, args.w);
          const int nk = ((cls & kNear) ? 1 : 0) + ((cls & kFar) ? 1 : 0);
          mbar_expect_tx(&bar_k[st], nk * C::TILE);
          if (cls & kNear) load_tile<D>(sKt(st, 0), &tm_k, &bar_k[st], k0, bh);
          if (cls & kFar) load_tile<D>(sKt(st, 1), &tm_k2, &bar_k[st], k0, bh);
          mbar_expect_tx(&bar_v[st], C::TILE);
          load_tile<D>(sVt(st, 0), &tm_v, &bar_v[st], k0, bh);
        } else {
          mbar_expect_tx(&bar_k[st], 2 * C::TILE);
          load_tile<D>(sKt(st, 0), &tm_k, &bar_k[st], k0, bh);
          load_tile<D>(sKt(st, 1), &tm_k2, &bar_k[st], k0, bh);
          mbar_expect_tx(&bar_v[st], 2 * C::TILE);
          load_tile<D>(sVt(st, 0), &tm_v, &bar_v[st], k0, bh);
          load_tile<D>(sVt(st, 1), &tm_v2, &bar_v[st], k0, bh);
        }
        last_phase[st] = (t / STAGES) & 1;
        used = t + 1 < STAGES ? t + 1 : STAGES;
      }
      // Never leave a TMA write in flight behind an early exit.
      WaitCtl drain{args.err, args.timeout_ns, &abort_flag};
      int zero = 0;
      drain.abort = reinterpret_cast<volatile int*>(&zero);
      mbar_wait(&bar_q, 0, drain, kErrTimeoutTma);
      for (int s = 0; s < used; ++s) {
        mbar_wait(&bar_k[s], last_phase[s], drain, kErrTimeoutTma);
        mbar_wait(&bar_v[s], last_phase[s], drain, kErrTimeoutTma);
      }
    }
  } else if (warp == 5) {
    // --------------------------------------------------------- MMA issuer
    if (nkv > 0) {
      constexpr uint32_t idesc_qk = idesc_f16(kBM, kBN, BF, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kBM, D, BF, false, true);
      const uint32_t aQ = smem_u32(sQ);
      const uint32_t aQ2 = aQ + C::TILE;
      auto issue_pv = [&](int u, uint64_t* done_bar) -> bool {
        const int b = u % NBUF;
        const int st = u % STAGES;
        if (!warp_wait(&bar_p[b], (u / NBUF) & 1, ctl, kErrTimeoutSoftmax)) return false;
        if (!warp_wait(&bar_v[st], (u / STAGES) & 1, ctl, kErrTimeoutTma)) return false;
        tc_fence_after();
        const uint32_t p_col = (NBUF == 2) ? (b ? C::COL_S1 : C::COL_S0) : C::COL_S0;
        mma_pv<D>(tmem + C::COL_O, tmem + p_col, smem_u32(sVt(st, 0)), idesc_pv, u > 0);
        if constexpr (MODE == kJvp) {  // U += (P o T) V + P tV
          const uint32_t pt_col = C::JVP2 ? p_col + 64 : C::COL_T;
          mma_pv<D>(tmem + C::COL_U, tmem + pt_col, smem_u32(sVt(st, 0)), idesc_pv, u > 0);
          mma_pv<D>(tmem + C::COL_U, tmem + p_col, smem_u32(sVt(st, 1)), idesc_pv, true);
        }
        commit_el(&bar_empty[st]);
        commit_el(done_bar);
        return true;
      };
      bool ok = warp_wait(&bar_q, 0, ctl, kErrTimeoutTma);
      for (int t = 0; ok && t < nkv; ++t) {
        const int st = t % STAGES;
        if (NBUF == 1 && t > 0) {
          ok = issue_pv(t - 1, &bar_o);
          if (!ok) break;
        }
        if (!warp_wait(&bar_k[st], (t / STAGES) & 1, ctl, kErrTimeoutTma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int b = t % NBUF;
        const uint32_t aK = smem_u32(sKt(st, 0));
        if constexpr (MODE == kStd) {
          mma_qk<D>(tmem + (b ? C::COL_S1 : C::COL_S0), aQ, aK, idesc_qk, false);
        } else if constexpr (MODE == kPiecewise) {
          const int cls = pw_class(q0, (t0 + t) * kBN, args.P_SEQ, args.w);
          const uint32_t sb = tmem + (b ? C::COL_S1 : C::COL_S0);
          if (cls == kNear) {
            mma_qk<D>(sb, aQ, aK, idesc_qk, false);
          } else if (cls == kFar) {
            mma_qk<D>(sb, aQ2, smem_u32(sKt(st, 1)), idesc_qk, false);
          } else {
            // the previous tile's softmax must be done with the third buffer
            if (t > 0 && pw_class(q0, (t0 + t - 1) * kBN, args.P_SEQ, args.w) == (kNear | kFar)) {
              if (!warp_wait(&bar_p[(t - 1) % NBUF], ((t - 1) / NBUF) & 1, ctl, kErrTimeoutSoftmax)) {
                ok = false;
                break;
              }
              tc_fence_after();
            }
            mma_qk<D>(sb, aQ, aK, idesc_qk, false);
            mma_qk<D>(tmem + C::COL_X, aQ2, smem_u32(sKt(st, 1)), idesc_qk, false);
          }
        } else {
          mma_qk<D>(tmem + (b ? C::COL_S1 : C::COL_S0), aQ, aK, idesc_qk, false);
          if constexpr (C::JVP2) {
            commit_el(&bar_s[b]);
            // T's columns are free once the softmax has read T(t - 1)
            if (t > 0 && !warp_wait(&bar_tfree, (t - 1) & 1, ctl, kErrTimeoutSoftmax)) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          // T = tq K^T + q tk^T (the sm_scale factor is applied by the softmax)
          mma_qk<D>(tmem + C::COL_T, aQ2, aK, idesc_qk, false);
          mma_qk<D>(tmem + C::COL_T, aQ, smem_u32(sKt(st, 1)), idesc_qk, true);
        }
        commit_el(C::JVP2 ? &bar_t : &bar_s[b]);
        if (NBUF == 2 && t > 0) {
          ok = issue_pv(t - 1, &bar_o);
        }
      }
      if (ok) issue_pv(nkv - 1, &bar_ofinal);
    }
  } else {
    // ------------------------------------------- softmax / correction / epilogue
    const int r = threadIdx.x;  // 0..127: query row within the tile, TMEM lane
    const int row = q0 + r;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m_ref = -INFINITY;  // running (lazily raised) row max, log2 domain
    float l = 0.f;
    float mu = 0.f;
    bool ok = true;
    for (int t = 0; t < nkv; ++t) {
      const int b = t % NBUF;
      if (!warp_wait(&bar_s[b], (t / NBUF) & 1, ctl, kErrTimeoutMma)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int k0 = (t0 + t) * kBN;
      uint32_t s[128];
      const uint32_t s_col = (NBUF == 2 && b) ? C::COL_S1 : C::COL_S0;
      int cls = kNear;
      if constexpr (MODE == kPiecewise) cls = pw_class(q0, k0, args.P_SEQ, args.w);
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_x32(lane_addr + s_col + 32 * c, TA_CHUNK(s, c));
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(TA_CHUNK(s, c));
      // raw scores; sm_scale * log2(e) > 0 is applied inside the exponent FMA
      float x[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) x[j] = __uint_as_float(s[j]);
      if constexpr (MODE == kPiecewise) {
        if (cls == (kNear | kFar)) {
          // far iff c <= row + P_SEQ - k0 - w: take the (q2, k2) score there
          const long long pwl = (long long)row + args.P_SEQ - k0 - args.w;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t s2[32];
            tmem_ld_x32(lane_addr + C::COL_X + 32 * c, s2);
            tmem_ld_wait(s2);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (32 * c + j <= pwl) x[32 * c + j] = __uint_as_float(s2[j]);
          }
        }
      }
      const bool need_mask =
          (args.causal && k0 + kBN - 1 > q0 + args.P_SEQ) || (k0 + kBN > args.N);
      if (need_mask) {
        int lim = args.N - 1 - k0;
        if (args.causal) lim = min(lim, row + args.P_SEQ - k0);
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j > lim) x[j] = -INFINITY;
      }
      // tree reductions: eight independent chains instead of one 128-long chain
      float mx8[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mx8[k] = x[k];
#pragma unroll
      for (int j = 8; j < 128; j += 8)
#pragma unroll
        for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(mx8[k], x[j + k]);
      const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                             fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
      const float m_new = fmaxf(m_ref, mx * args.scale_log2);
      bool resc = false;
      float alpha = 1.f;
      if (t == 0) {
        m_ref = m_new;
      } else if (m_new > m_ref + kRescaleThreshold) {
        resc = true;
        alpha = ex2(m_ref - m_new);
        m_ref = m_new;
      }
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
      float rs8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 128; ++j) {
        x[j] = ex2(fmaf(x[j], args.scale_log2, neg_m));
        rs8[j & 7] += x[j];
      }
      const float rs = ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
      l = l * alpha + rs;
      // P (16-bit, two per column) over the first 64 columns of the S buffer
      const uint32_t p_col = s_col;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = pack2<BF>(x[32 * c + 2 * j], x[32 * c + 2 * j + 1]);
        tmem_st_x16(lane_addr + p_col + 16 * c, pk);
      }
      if constexpr (MODE == kJvp) {
        // P o T (T = sm_scale * (tq k^T + q tk^T)), 16-bit, over the second
        // half of the S buffer (JVP2) or the first 64 columns of T
        if constexpr (C::JVP2) {
          if (!warp_wait(&bar_t, t & 1, ctl, kErrTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint32_t pt_col = C::JVP2 ? s_col + 64 : C::COL_T;
        float mp4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t tr[32];
          tmem_ld_x32(lane_addr + C::COL_T + 32 * c, tr);
          tmem_ld_wait(tr);
          if (C::JVP2 && c == 3) {  // every T column read: T(t + 1) may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_tfree);
          }
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float a0 = x[32 * c + 2 * j] * __uint_as_float(tr[2 * j]) * args.sm_scale;
            const float a1 = x[32 * c + 2 * j + 1] * __uint_as_float(tr[2 * j + 1]) * args.sm_scale;
            mp4[j & 3] += a0 + a1;
            pk[j] = pack2<BF>(a0, a1);
          }
          tmem_st_x16(lane_addr + pt_col + 16 * c, pk);
        }
        mu = mu * alpha + ((mp4[0] + mp4[1]) + (mp4[2] + mp4[3]));
      }
      // Correction: rescale the O (and U) rows once the previous P V landed.
      if (t > 0 && __any_sync(0xffffffffu, resc)) {
        if (!warp_wait(&bar_o, (t - 1) & 1, ctl, kErrTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        constexpr int NACC = (MODE == kJvp) ? 2 : 1;
#pragma unroll
        for (int a = 0; a < NACC; ++a) {
          const uint32_t col0 = a ? C::COL_U : C::COL_O;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tmem_ld_x32(lane_addr + col0 + 32 * c, ov);
            tmem_ld_wait(ov);
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            tmem_st_x32(lane_addr + col0 + 32 * c, ov);
          }
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[b]);
    }
    // ------------------------------------------------------------ epilogue
    if (nkv > 0) ok = warp_wait(&bar_ofinal, 0, ctl, kErrTimeoutMma) && __all_sync(0xffffffffu, ok);
    tc_fence_after();
    const bool live = ok && nkv > 0;
    if (SPLIT && part == 1) {
      // Hand the raw state over to the first CTA of the pair (which writes
      // every output row); a CTA without key tiles has nothing to hand over.
      if (nkv > 0) {
        float* hs = reinterpret_cast<float*>(base);
        hs[r] = live ? m_ref : -INFINITY;
        hs[kBM + r] = live ? l : 0.f;
        hs[2 * kBM + r] = live ? mu : 0.f;
        float4* ho = reinterpret_cast<float4*>(base + kSplitHdr);
        if (live) {
#pragma unroll
          for (int a = 0; a < NACC; ++a) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ov[32];
              tmem_ld_x32(lane_addr + (a ? C::COL_U : C::COL_O) + 32 * c, ov);
              tmem_ld_wait(ov);
#pragma unroll
              for (int g = 0; g < 8; ++g)
                ho[((a * (D / 32) + c) * 8 + g) * kBM + r] =
                    make_float4(__uint_as_float(ov[4 * g]), __uint_as_float(ov[4 * g + 1]),
                                __uint_as_float(ov[4 * g + 2]), __uint_as_float(ov[4 * g + 3]));
            }
          }
        }
        mbar_arrive_cluster(mapa_shared(smem_u32(&bar_peer), 0));
      }
    } else {
      // SPLIT: fold the partner's state in (a0, a1 scale this CTA's and the
      // partner's accumulators; a1 = 0 leaves this CTA's own state).
      float a0 = 1.f, a1 = 0.f;
      uint32_t peer = 0;
      if constexpr (SPLIT) {
        if (n_peer > 0) {
          const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&bar_peer, 0, ctl, kErrTimeoutOther));
          peer = mapa_shared(smem_u32(base), 1);
          if (got && live) {
            const float m1 = ld_cluster_f32(peer + 4 * r);
            const float l1 = ld_cluster_f32(peer + 4 * (kBM + r));
            const float mu1 = ld_cluster_f32(peer + 4 * (2 * kBM + r));
            if (l1 > 0.f) {
              if (l > 0.f) {
                const float m = fmaxf(m_ref, m1);
                a0 = ex2(m_ref - m);
                a1 = ex2(m1 - m);
                m_ref = m;
              } else {
                a0 = 0.f;
                a1 = 1.f;
                m_ref = m1;
              }
              l = a0 * l + a1 * l1;
              mu = a0 * mu + a1 * mu1;
            }
          }
        }
      }
      // acc chunk c of accumulator a (0: O, 1: U), this CTA's TMEM rows merged with the partner's
      auto acc_chunk = [&](int a, int c, const uint32_t (&ov)[32], float (&out)[32], float scale) {
#pragma unroll
        for (int j = 0; j < 32; ++j) out[j] = __uint_as_float(ov[j]) * a0;
        if (SPLIT && a1 != 0.f) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const float4 pv = ld_cluster_v4(peer + kSplitHdr + (((a * (D / 32) + c) * 8 + g) * kBM + r) * 16);
            out[4 * g] = fmaf(a1, pv.x, out[4 * g]);
            out[4 * g + 1] = fmaf(a1, pv.y, out[4 * g + 1]);
            out[4 * g + 2] = fmaf(a1, pv.z, out[4 * g + 2]);
            out[4 * g + 3] = fmaf(a1, pv.w, out[4 * g + 3]);
          }
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) out[j] *= scale;
      };
      const float inv_l = (live && l > 0.f) ? 1.f / l : 0.f;
      if (row < args.M) {
        T* orow = reinterpret_cast<T*>(args.o) + (static_cast<size_t>(bh) * args.M + row) * args.dg;
        T* trow = nullptr;
        if constexpr (MODE == kJvp) trow = reinterpret_cast<T*>(args.to) + (static_cast<size_t>(bh) * args.M + row) * args.dg;
        args.lse[static_cast<size_t>(bh) * args.M + row] =
            (live && l > 0.f) ? (m_ref + lg2(l)) * kLn2 : -INFINITY;
        if constexpr (MODE == kJvp) {  // tL = sum_j P_ij T_ij = mu / l
          if (args.tlse) args.tlse[static_cast<size_t>(bh) * args.M + row] = (live && l > 0.f) ? mu * inv_l : 0.f;
        }
        (void)trow;
        if (!live) {
          float z[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) z[j] = 0.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            store_row_chunk<T>(orow + 32 * c, z, 0.f, chunk_groups(args.dg, 32 * c));
            if constexpr (MODE == kJvp) store_row_chunk<T>(trow + 32 * c, z, 0.f, chunk_groups(args.dg, 32 * c));
          }
        }
      }
      if (live) {
        // tcgen05.ld is warp-collective: every lane loads, rows >= M skip the store.
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld_x32(lane_addr + C::COL_O + 32 * c, ov);
          tmem_ld_wait(ov);
          float of[32];
          acc_chunk(0, c, ov, of, inv_l);
          if (row < args.M) {
            T* orow = reinterpret_cast<T*>(args.o) + (static_cast<size_t>(bh) * args.M + row) * args.dg;
            store_row_chunk<T>(orow + 32 * c, of, 1.f, chunk_groups(args.dg, 32 * c));
          }
          if constexpr (MODE == kJvp) {
            uint32_t uv[32];
            tmem_ld_x32(lane_addr + C::COL_U + 32 * c, uv);
            tmem_ld_wait(uv);
            const float mu_l = mu * inv_l;
            float tv[32];
            acc_chunk(1, c, uv, tv, inv_l);
#pragma unroll
            for (int j = 0; j < 32; ++j) tv[j] -= mu_l * of[j];
            if (row < args.M) {
              T* trow = reinterpret_cast<T*>(args.to) + (static_cast<size_t>(bh) * args.M + row) * args.dg;
              store_row_chunk<T>(trow + 32 * c, tv, 1.f, chunk_groups(args.dg, 32 * c));
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // SPLIT: the second CTA's shared memory stays alive until the first has read it
  if constexpr (SPLIT) cluster_sync_all();
  tc_fence_after();
  if (warp == 5) tmem_dealloc(tmem, 512);
}

template <typename T, int MODE, int D>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q2,
                    const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v2,
                    const FwdArgs args) {
  fwd1_body<T, MODE, D, false>(tm_q, tm_k, tm_v, tm_q2, tm_k2, tm_v2, args);
}

// Grid (BH, 2 x query tiles): blocks (x, 2i) and (x, 2i + 1) form a cluster.
template <typename T, int MODE, int D>
__global__ void __cluster_dims__(1, 2, 1) __launch_bounds__(192, 1)
    attn_fwd_split_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q2,
                          const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_v2,
                          const FwdArgs args) {
  fwd1_body<T, MODE, D, true>(tm_q, tm_k, tm_v, tm_q2, tm_k2, tm_v2, args);
}

// ======================================================================
//   Two query tiles per CTA (ping-pong softmax groups): the standard
//   forward, and the piecewise forward at D = 64
// ======================================================================
// One CTA owns query rows [q0, q0 + 256) of one head as two 128-row tiles
// that share every K/V tile.  Warps 0-3 run the softmax of tile 0, warps 4-7
// that of tile 1, warp 8 is the TMA producer and warp 9 the MMA issuer, which
// alternates between the tiles so one group's softmax overlaps the other
// group's MMAs:  S0(t) S1(t) | PV0(t) S0(t+1) | PV1(t) S1(t+1) | ...
// K and V have separate rings: a K tile is released as soon as both score
// MMAs that read it have finished, so the K ring runs further ahead of the
// MMAs than a joint K/V ring of the same size could.
// Piecewise (PW): Q1 and Q2 of both tiles stay resident and a K stage holds
// K1 and/or K2 as the two tiles' classes need; a tile whose keys are all
// near (or all far) runs one score MMA, one that straddles the distance w
// runs S(q1, k1) into its own buffer and S(q2, k2) into a third buffer that
// the two tiles share (its reader's arrival on bar_xfree releases it).
template <int D, bool PW = false>
struct Fwd2Cfg {
  static constexpr int BLK = kBM * 128;
  static constexpr int TILE = (D / 64) * BLK;
  // piecewise: Q1 and Q2 of both query tiles resident, K1 and K2 per K stage,
  // and a third 128-column score buffer for S(q2, k2) of a tile that needs both
  static constexpr int NQ = PW ? 4 : 2;
  static constexpr int NK = PW ? 2 : 1;
  static constexpr int KST = PW ? 3 : (D == 128) ? 3 : 4;  // K ring depth
  static constexpr int VST = PW ? 3 : (D == 128) ? 2 : 4;  // V ring depth
  static constexpr int SMEM = (NQ + NK * KST + VST) * TILE + 1024;
  static constexpr uint32_t COL_X = 256 + 2 * D;
  static_assert(SMEM + 2048 <= kSmemMax, "tiles do not fit in shared memory");
  static_assert(256 + 2 * D + (PW ? 128 : 0) <= 512, "TMEM overflow");
};

// The kernel body; the standard entry point below takes three tensor maps,
// the piecewise one five.  The maps arrive by reference to the __grid_constant__
// kernel parameters, whose addresses the TMA instructions take.
template <typename T, int D, bool PW>
__device__ __forceinline__ void fwd2_body(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                          const CUtensorMap& tm_q2, const CUtensorMap& tm_k2, const CUtensorMap& tm_o,
                                          const FwdArgs args) {
  using C = Fwd2Cfg<D, PW>;
  constexpr bool BF = DT<T>::bf16;
  constexpr int KST = C::KST, VST = C::VST;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q;
  __shared__ __align__(8) uint64_t bar_k[KST], bar_kempty[KST], bar_v[VST], bar_vempty[VST];
  __shared__ __align__(8) uint64_t bar_s[2], bar_p[2], bar_o[2], bar_ofinal;
  __shared__ __align__(8) uint64_t bar_xfree;  // piecewise: the third score buffer has been read
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pairs = (args.M + 2 * kBM - 1) / (2 * kBM);
  int bh, rank;
  if (!grouped_tile(blockIdx.x, args.BH, pairs, args.group_heads, &bh, &rank)) return;
  const int pair = pairs - 1 - rank;  // heaviest causal pairs first
  const int q0 = pair * 2 * kBM;
  int n_t[2];
  n_t[0] = kv_tiles_for(q0, args.M, args.N, args.P_SEQ, args.causal);
  n_t[1] = kv_tiles_for(q0 + kBM, args.M, args.N, args.P_SEQ, args.causal);
  const int nt = n_t[1] > n_t[0] ? n_t[1] : n_t[0];

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;  // tile 0 at sQ, tile 1 at sQ + TILE (piecewise: then Q2 of both)
  auto sK = [&](int st) { return base + (C::NQ + C::NK * st) * C::TILE; };  // K | K1 (+ K2 next)
  auto sV = [&](int st) { return base + (C::NQ + C::NK * KST + st) * C::TILE; };
  // piecewise: which score products query tile w needs for key tile t
  auto cls_of = [&](int w, int t) { return pw_class(q0 + w * kBM, t * kBN, args.P_SEQ, args.w); };

  WaitCtl ctl{args.err, args.timeout_ns, &abort_flag};
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar_q, 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(&bar_k[s], 1);
      mbar_init(&bar_kempty[s], 1);
    }
    for (int s = 0; s < VST; ++s) {
      mbar_init(&bar_v[s], 1);
      mbar_init(&bar_vempty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&bar_s[w], 1);
      mbar_init(&bar_p[w], 4);
      mbar_init(&bar_o[w], 1);
    }
    mbar_init(&bar_ofinal, 1);
    if constexpr (PW) mbar_init(&bar_xfree, 4);
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t col_s[2] = {0u, 128u};
  const uint32_t col_o[2] = {256u, 256u + D};

  if (warp == 8) {
    // ------------------------------------------------------ TMA producer
    // lane 0 feeds Q and the K ring, lane 1 the V ring, independently
    if (lane < 2 && nt > 0) {
      const bool is_k = (lane == 0);
      const int depth = is_k ? KST : VST;
      uint64_t* full = is_k ? bar_k : bar_v;
      uint64_t* empty = is_k ? bar_kempty : bar_vempty;
      const CUtensorMap* map = is_k ? &tm_k : &tm_v;
      if (is_k) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        mbar_expect_tx(&bar_q, C::NQ * C::TILE);
        load_tile<D>(sQ, &tm_q, &bar_q, q0, bh);
        load_tile<D>(sQ + C::TILE, &tm_q, &bar_q, q0 + kBM, bh);
        if constexpr (PW) {
          load_tile<D>(sQ + 2 * C::TILE, &tm_q2, &bar_q, q0, bh);
          load_tile<D>(sQ + 3 * C::TILE, &tm_q2, &bar_q, q0 + kBM, bh);
        }
      } else {
        tma_prefetch_desc(&tm_v);
      }
      int issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int st = t % depth;
        if (t >= depth && !mbar_wait(&empty[st], ((t / depth) - 1) & 1, ctl, kErrTimeoutMma)) break;
        if (PW && is_k) {  // K1 if either query tile needs a near product, K2 if either needs a far one
          int need = 0;
          for (int w = 0; w < 2; ++w)
            if (t < n_t[w]) need |= cls_of(w, t);
          mbar_expect_tx(&full[st], (((need & kNear) ? 1 : 0) + ((need & kFar) ? 1 : 0)) * C::TILE);
          if (need & kNear) load_tile<D>(sK(st), &tm_k, &full[st], t * kBN, bh);
          if (need & kFar) load_tile<D>(sK(st) + C::TILE, &tm_k2, &full[st], t * kBN, bh);
        } else {
          mbar_expect_tx(&full[st], C::TILE);
          load_tile<D>(is_k ? sK(st) : sV(st), map, &full[st], t * kBN, bh);
        }
        issued = t + 1;
      }
      int zero = 0;
      WaitCtl drain{args.err, args.timeout_ns, reinterpret_cast<volatile int*>(&zero)};
      if (is_k) mbar_wait(&bar_q, 0, drain, kErrTimeoutTma);
      for (int t = issued - depth > 0 ? issued - depth : 0; t < issued; ++t)
        mbar_wait(&full[t % depth], (t / depth) & 1, drain, kErrTimeoutTma);
    }
  } else if (warp == 9) {
    // --------------------------------------------------------- MMA issuer
    if (nt > 0) {
      constexpr uint32_t idesc_qk = idesc_f16(kBM, kBN, BF, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kBM, D, BF, false, true);
      const uint32_t aQ[2] = {smem_u32(sQ), smem_u32(sQ) + C::TILE};
      int nx = 0;  // piecewise: uses of the third score buffer so far
      // S of query tile w against key tile t (stage sk); false if a wait ran out
      auto issue_s = [&](int w, int t, int sk) -> bool {
        if constexpr (!PW) {
          mma_qk<D>(tmem + col_s[w], aQ[w], smem_u32(sK(sk)), idesc_qk, false);
        } else {
          const int cls = cls_of(w, t);
          const uint32_t aK1 = smem_u32(sK(sk)), aK2 = aK1 + C::TILE, aQ2 = aQ[w] + 2 * C::TILE;
          if (cls == kNear) {
            mma_qk<D>(tmem + col_s[w], aQ[w], aK1, idesc_qk, false);
          } else if (cls == kFar) {
            mma_qk<D>(tmem + col_s[w], aQ2, aK2, idesc_qk, false);
          } else {  // S(q1, k1) in its own buffer, S(q2, k2) in the shared third one
            if (nx > 0) {
              if (!warp_wait(&bar_xfree, (nx - 1) & 1, ctl, kErrTimeoutSoftmax)) return false;
              tc_fence_after();
            }
            ++nx;
            mma_qk<D>(tmem + col_s[w], aQ[w], aK1, idesc_qk, false);
            mma_qk<D>(tmem + C::COL_X, aQ2, aK2, idesc_qk, false);
          }
        }
        commit_el(&bar_s[w]);
        return true;
      };
      bool ok = warp_wait(&bar_q, 0, ctl, kErrTimeoutTma) && warp_wait(&bar_k[0], 0, ctl, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        for (int w = 0; w < 2; ++w)
          if (n_t[w] > 0) {
            if constexpr (PW) {
              if (ok) ok = issue_s(w, 0, 0);
            } else {
              mma_qk<D>(tmem + col_s[w], aQ[w], smem_u32(sK(0)), idesc_qk, false);
              commit_el(&bar_s[w]);
            }
          }
      }
      if (ok) commit_el(&bar_kempty[0]);  // K tile 0 is consumed once both score MMAs finish
      for (int t = 0; ok && t < nt; ++t) {
        const int sv = t % VST;
        const int sk1 = (t + 1) % KST;
        if (!(ok = warp_wait(&bar_v[sv], (t / VST) & 1, ctl, kErrTimeoutTma))) break;
        const bool next = t + 1 < nt;
        if (next && !(ok = warp_wait(&bar_k[sk1], ((t + 1) / KST) & 1, ctl, kErrTimeoutTma))) break;
        for (int w = 0; w < 2; ++w) {
          if (t < n_t[w]) {
            if (!(ok = warp_wait(&bar_p[w], t & 1, ctl, kErrTimeoutSoftmax))) break;
            tc_fence_after();
            mma_pv<D>(tmem + col_o[w], tmem + col_s[w], smem_u32(sV(sv)), idesc_pv, t > 0);
            commit_el(&bar_o[w]);
          }
          if (next && t + 1 < n_t[w]) {
            if constexpr (PW) {
              if (!(ok = issue_s(w, t + 1, sk1))) break;
            } else {  // the standard path keeps the MMA warp's loop as lean as possible
              mma_qk<D>(tmem + col_s[w], aQ[w], smem_u32(sK(sk1)), idesc_qk, false);
              commit_el(&bar_s[w]);
            }
          }
        }
        if (!ok) break;
        commit_el(&bar_vempty[sv]);
        if (next) commit_el(&bar_kempty[sk1]);
      }
      if (ok) commit_el(&bar_ofinal);
    }
  } else {
    // ------------------------------- softmax / correction / epilogue (tile w)
    const int w = warp >> 2;
    const int r = threadIdx.x & 127;
    const int row = q0 + w * kBM + r;
    const int tq0 = q0 + w * kBM;  // first row of this group's tile
    const int n = n_t[w];
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      if (!(ok = warp_wait(&bar_s[w], t & 1, ctl, kErrTimeoutMma))) break;
      tc_fence_after();
      const int k0 = t * kBN;
      uint32_t s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_x32(lane_addr + col_s[w] + 32 * c, TA_CHUNK(s, c));
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(TA_CHUNK(s, c));
      float x[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) x[j] = __uint_as_float(s[j]);
      if constexpr (PW) {
        if (cls_of(w, t) == (kNear | kFar)) {
          // far iff key k0 + c satisfies row + P_SEQ - (k0 + c) >= w: take S(q2, k2) there
          const long long pwl = (long long)row + args.P_SEQ - k0 - args.w;
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 16 columns at a time: the row's 128 scores are live
            uint32_t s2[16];
            tmem_ld_x16(lane_addr + C::COL_X + 16 * c, s2);
            tmem_ld_wait(s2);
#pragma unroll
            for (int j = 0; j < 16; ++j)
              if (16 * c + j <= pwl) x[16 * c + j] = __uint_as_float(s2[j]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bar_xfree);
        }
      }
      if ((args.causal && k0 + kBN - 1 > tq0 + args.P_SEQ) || (k0 + kBN > args.N)) {
        int lim = args.N - 1 - k0;
        if (args.causal) lim = min(lim, row + args.P_SEQ - k0);
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j > lim) x[j] = -INFINITY;
      }
      float mx8[8];  // eight three-input max chains of 16 scores each
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        mx8[k] = fmax3(x[k], x[8 + k], x[16 + k]);
#pragma unroll
        for (int j = 24; j < 120; j += 16) mx8[k] = fmax3(mx8[k], x[j + k], x[j + 8 + k]);
        mx8[k] = fmaxf(mx8[k], x[120 + k]);
      }
      const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      const float m_new = fmaxf(m_ref, mx * args.scale_log2);
      bool resc = false;
      float alpha = 1.f;
      if (t == 0) {
        m_ref = m_new;
      } else if (m_new > m_ref + kRescaleThreshold) {
        resc = true;
        alpha = ex2(m_ref - m_new);
        m_ref = m_new;
      }
      const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
      // P = 2^(x c - m): scale, shift and row sum two columns per packed
      // instruction (the softmax warps share issue slots with the MMA warp,
      // so their instruction count is what limits the step).
      const float2 sc2 = make_float2(args.scale_log2, args.scale_log2);
      const float2 nm2 = make_float2(neg_m, neg_m);
      float2 rs2[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < 8; ++c) {  // 16 columns of S, 8 packed columns of P, at a time
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float2 y = ffma2(make_float2(x[16 * c + 2 * e], x[16 * c + 2 * e + 1]), sc2, nm2);
          const float2 pr = make_float2(ex2(y.x), ex2(y.y));
          rs2[e & 3] = fadd2(rs2[e & 3], pr);
          pk[e] = pack2<BF>(pr.x, pr.y);
        }
        tmem_st_x8(lane_addr + col_s[w] + 8 * c, pk);
      }
      const float2 rsa = fadd2(fadd2(rs2[0], rs2[1]), fadd2(rs2[2], rs2[3]));
      const float rs = rsa.x + rsa.y;
      l = l * alpha + rs;
      if (t > 0 && __any_sync(0xffffffffu, resc)) {
        if (!(ok = warp_wait(&bar_o[w], (t - 1) & 1, ctl, kErrTimeoutMma))) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tmem_ld_x32(lane_addr + col_o[w] + 32 * c, ov);
          tmem_ld_wait(ov);
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
          tmem_st_x32(lane_addr + col_o[w] + 32 * c, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar_p[w]);
    }
    // ------------------------------------------------------------ epilogue
    if (nt > 0) ok = warp_wait(&bar_ofinal, 0, ctl, kErrTimeoutMma) && __all_sync(0xffffffffu, ok);
    tc_fence_after();
    const bool live = ok && n > 0;
    const float inv_l = (live && l > 0.f) ? 1.f / l : 0.f;
    if (row < args.M)
      args.lse[static_cast<size_t>(bh) * args.M + row] = (live && l > 0.f) ? (m_ref + lg2(l)) * kLn2 : -INFINITY;
    // O of the tile, scaled and rounded, is staged over the tile's Q buffer
    // (free: every MMA has finished) in the output map's swizzled box layout
    // and written by TMA stores, which clip rows past M and columns past D.
    const uint32_t stage = smem_u32(sQ) + static_cast<uint32_t>(w * C::TILE);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t ov[32];
      if (live) {
        tmem_ld_x32(lane_addr + col_o[w] + 32 * c, ov);
        tmem_ld_wait(ov);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] = 0u;
      }
      stage_row_chunk_sw128<BF>(stage, r, c, ov, inv_l);
    }
    fence_proxy_async_smem();
    named_bar_sync(1 + w, 4 * 32);  // the tile's four warps have staged their rows
    if ((warp & 3) == 0 && lane == 0 && tq0 < args.M) {
#pragma unroll
      for (int kb = 0; kb < D / 64; ++kb) tma_store_3d(&tm_o, sQ + w * C::TILE + kb * (kBM * 128), kb * 64, tq0, bh);
      tma_store_commit_and_wait_read();
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

template <typename T, int D>
__global__ void __launch_bounds__(320, 1)
    attn_fwd2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                     const FwdArgs args) {
  fwd2_body<T, D, false>(tm_q, tm_k, tm_v, tm_q, tm_k, tm_o, args);
}

template <typename T, int D>
__global__ void __launch_bounds__(320, 1)
    attn_fwd2_pw_kernel(const __grid_constant__ CUtensorMap tm_q1, const __grid_constant__ CUtensorMap tm_k1,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q2,
                        const __grid_constant__ CUtensorMap tm_k2, const __grid_constant__ CUtensorMap tm_o,
                        const FwdArgs args) {
  fwd2_body<T, D, true>(tm_q1, tm_k1, tm_v, tm_q2, tm_k2, tm_o, args);
}

// ---------------------------------------------------------------- host side
template <typename T, int MODE, int D>
static cudaError_t launch_fwd_t(const FwdMaps& maps, const FwdArgs& a, bool split, cudaStream_t stream) {
  using C = FwdCfg<MODE, D>;
  if (split) {
    if (2ll * a.num_q_tiles > 65535) return cudaErrorInvalidValue;
    auto kern = attn_fwd_split_kernel<T, MODE, D>;
    static std::atomic<bool> attr[kMaxDevices];
    cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
    if (e_attr != cudaSuccess) return e_attr;
    dim3 grid(a.BH, 2 * a.num_q_tiles);
    kern<<<grid, 192, C::SMEM, stream>>>(maps.q, maps.k, maps.v, maps.q2, maps.k2, maps.v2, a);
    return cudaGetLastError();
  }
  auto kern = attn_fwd_kernel<T, MODE, D>;
  static std::atomic<bool> attr[kMaxDevices];
  cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
  if (e_attr != cudaSuccess) return e_attr;
  dim3 grid(a.BH, a.num_q_tiles);
  kern<<<grid, 192, C::SMEM, stream>>>(maps.q, maps.k, maps.v, maps.q2, maps.k2, maps.v2, a);
  return cudaGetLastError();
}

template <typename T, int D, bool PW = false>
static cudaError_t launch_fwd2_t(const FwdMaps& maps, const FwdArgs& a, cudaStream_t stream) {
  using C = Fwd2Cfg<D, PW>;
  static std::atomic<bool> attr[kMaxDevices];
  const long long pairs = (a.M + 2 * kBM - 1) / (2 * kBM);
  const long long blocks = pairs * a.BH;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  if constexpr (PW) {
    auto kern = attn_fwd2_pw_kernel<T, D>;
    cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
    if (e_attr != cudaSuccess) return e_attr;
    kern<<<static_cast<unsigned>(blocks), 320, C::SMEM, stream>>>(maps.q, maps.k, maps.v, maps.q2, maps.k2, maps.o,
                                                                   a);
  } else {
    auto kern = attn_fwd2_kernel<T, D>;
    cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
    if (e_attr != cudaSuccess) return e_attr;
    kern<<<static_cast<unsigned>(blocks), 320, C::SMEM, stream>>>(maps.q, maps.k, maps.v, maps.o, a);
  }
  return cudaGetLastError();
}

bool fwd_split_capable(int mode, int D) { return mode == kJvp || (mode == kPiecewise && D == 128); }

cudaError_t launch_fwd(int mode, bool bf16, int D, const FwdMaps& maps, const FwdArgs& a, bool split,
                       cudaStream_t s) {
  if (split && !fwd_split_capable(mode, D)) return cudaErrorInvalidValue;
  if (mode == kStd) {
    if (D == 64) return bf16 ? launch_fwd2_t<__nv_bfloat16, 64>(maps, a, s) : launch_fwd2_t<__half, 64>(maps, a, s);
    if (D == 128) return bf16 ? launch_fwd2_t<__nv_bfloat16, 128>(maps, a, s) : launch_fwd2_t<__half, 128>(maps, a, s);
  }
  if (mode == kPiecewise && D == 64)  // two query tiles per CTA; TMEM has room for the third score buffer
    return bf16 ? launch_fwd2_t<__nv_bfloat16, 64, true>(maps, a, s) : launch_fwd2_t<__half, 64, true>(maps, a, s);
#define TA_FWD_CASE(MODE_, D_)                                                          \
  if (mode == MODE_ && D == D_)                                                         \
    return bf16 ? launch_fwd_t<__nv_bfloat16, MODE_, D_>(maps, a, split, s)             \
                : launch_fwd_t<__half, MODE_, D_>(maps, a, split, s);
  TA_FWD_CASE(kPiecewise, 128)
  TA_FWD_CASE(kJvp, 64)
  TA_FWD_CASE(kJvp, 128)
#undef TA_FWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace ta

TA_GUARD_ACCESSOR(fwd)
