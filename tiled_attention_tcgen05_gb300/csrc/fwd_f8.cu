// FP8 (e5m2) attention forward: the 8-bit path of "Triton fused attention
// tutorial, updated with JVP support" (_attn_fwd with FP8_OUTPUT and its fp8
// benchmark): q and k in float8 e5m2, v passed transposed ([B,H,D,N], the
// layout the tutorial builds for fp8 so that the second operand of P V is
// K-major), P rounded to e5m2 for the P V product, O written in e5m2 and L
// in fp32.  The softmax is the same online softmax as the 16-bit forward.
//
// Structure as the 16-bit two-tile forward (fwd.cu, attn_fwd2_kernel): two
// 128-row query tiles per CTA share every K / V^T tile, warps 0-3 and 4-7
// run their softmaxes, warp 8 feeds TMA rings and warp 9 issues the MMAs,
// alternating between the tiles.  The MMAs are tcgen05 kind::f8f6f4 (K = 32
// per instruction): S = Q K^T from two K-major shared-memory tiles, O += P V
// with P packed four e5m2 per TMEM column and V^T as the K-major B operand.
// Rows are 128 bytes (one 128-byte swizzle atom); for D = 64 the TMA box is
// still 128 elements wide and the columns past D load as zeros.
#include "common.cuh"
#include "launch.h"

namespace ta {

template <int D>
struct F8Cfg {
  static constexpr int QT = kBM * 128;  // Q or K tile: 128 rows x 128 bytes
  static constexpr int VT = D * 128;    // V^T tile: D rows x 128 keys
  static constexpr int KST = 4;         // K ring depth
  static constexpr int VST = 4;         // V^T ring depth
  static constexpr int SMEM = (2 + KST) * QT + VST * VT + 1024;
  static_assert(SMEM + 2048 <= kSmemMax, "tiles do not fit in shared memory");
  static_assert(256 + 2 * D <= 512, "TMEM overflow");
};

// S = Q K^T over D (e5m2): 128-row K-major tiles with 128-byte rows; each
// K-step is 32 elements = 32 bytes further along the swizzle atom.
template <int D>
__device__ __forceinline__ void mma_qk_f8(uint32_t d_tmem, uint32_t a_smem, uint32_t b_smem, uint32_t idesc) {
  const uint64_t da0 = sdesc_sw128(a_smem, 16, 1024);
  const uint64_t db0 = sdesc_sw128(b_smem, 16, 1024);
  uint64_t da[D / 32], db[D / 32];
#pragma unroll
  for (int kk = 0; kk < D / 32; ++kk) {
    da[kk] = da0 + static_cast<uint64_t>((kk * 32) >> 4);
    db[kk] = db0 + static_cast<uint64_t>((kk * 32) >> 4);
  }
  mma_ss_f8_n<D / 32>(d_tmem, da, db, idesc, 0u);
}

// O (+)= P V: P is 128 x 128 e5m2 in TMEM (four per 32-bit column, 8 columns
// per K-step of 32 keys), V^T a D-row K-major tile with 128-byte rows.
__device__ __forceinline__ void mma_pv_f8(uint32_t d_tmem, uint32_t p_tmem, uint32_t vt_smem, uint32_t idesc,
                                          bool accumulate) {
  const uint64_t dv = sdesc_sw128(vt_smem, 16, 1024);
  uint32_t a[kBN / 32];
  uint64_t b[kBN / 32];
#pragma unroll
  for (int kk = 0; kk < kBN / 32; ++kk) {
    a[kk] = p_tmem + kk * 8;
    b[kk] = dv + static_cast<uint64_t>((kk * 32) >> 4);
  }
  mma_ts_f8_n<kBN / 32>(d_tmem, a, b, idesc, accumulate ? 1u : 0u);
}

// Four fp32 values -> four e5m2 bytes (round to nearest even, saturating to
// the largest finite value), the lowest-index value in the lowest byte.
__device__ __forceinline__ uint32_t pack4_e5m2(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// 32 fp32 values (x scale) -> 32 e5m2 bytes at dst (16-byte aligned).
__device__ __forceinline__ void store_chunk32_e5m2(uint8_t* dst, const float* v, float scale) {
  if (!TA_CHECK((reinterpret_cast<uintptr_t>(dst) & 15u) == 0u)) return;
  uint4 u[2];
  uint32_t* w = reinterpret_cast<uint32_t*>(u);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = pack4_e5m2(v[4 * i] * scale, v[4 * i + 1] * scale, v[4 * i + 2] * scale, v[4 * i + 3] * scale);
  reinterpret_cast<uint4*>(dst)[0] = u[0];
  reinterpret_cast<uint4*>(dst)[1] = u[1];
}

#define TA8_CHUNK(arr, c) (*reinterpret_cast<uint32_t(*)[32]>(&(arr)[32 * (c)]))

template <int D>
__global__ void __launch_bounds__(320, 1)
    attn_fwd_f8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_vt, const FwdArgs args) {
  using C = F8Cfg<D>;
  constexpr int KST = C::KST, VST = C::VST;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bar_q;
  __shared__ __align__(8) uint64_t bar_k[KST], bar_kempty[KST], bar_v[VST], bar_vempty[VST];
  __shared__ __align__(8) uint64_t bar_s[2], bar_p[2], bar_o[2], bar_ofinal;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int pairs = (args.M + 2 * kBM - 1) / (2 * kBM);
  int bh, rank;
  if (!grouped_tile(blockIdx.x, args.BH, pairs, kGroupHeads, &bh, &rank)) return;
  const int pair = pairs - 1 - rank;  // heaviest causal pairs first
  const int q0 = pair * 2 * kBM;
  int n_t[2];
  n_t[0] = kv_tiles_for(q0, args.M, args.N, args.P_SEQ, args.causal);
  n_t[1] = kv_tiles_for(q0 + kBM, args.M, args.N, args.P_SEQ, args.causal);
  const int nt = n_t[1] > n_t[0] ? n_t[1] : n_t[0];

  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;  // tile 0 at sQ, tile 1 at sQ + QT
  auto sK = [&](int st) { return base + (2 + st) * C::QT; };
  auto sV = [&](int st) { return base + (2 + KST) * C::QT + st * C::VT; };

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
    // lane 0 feeds Q and the K ring, lane 1 the V^T ring, independently
    if (lane < 2 && nt > 0) {
      const bool is_k = (lane == 0);
      const int depth = is_k ? KST : VST;
      uint64_t* full = is_k ? bar_k : bar_v;
      uint64_t* empty = is_k ? bar_kempty : bar_vempty;
      if (is_k) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        mbar_expect_tx(&bar_q, 2 * C::QT);
        tma_load_3d(sQ, &tm_q, &bar_q, 0, q0, bh);
        tma_load_3d(sQ + C::QT, &tm_q, &bar_q, 0, q0 + kBM, bh);
      } else {
        tma_prefetch_desc(&tm_vt);
      }
      int issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int st = t % depth;
        if (t >= depth && !mbar_wait(&empty[st], ((t / depth) - 1) & 1, ctl, kErrTimeoutMma)) break;
        if (is_k) {
          mbar_expect_tx(&full[st], C::QT);
          tma_load_3d(sK(st), &tm_k, &full[st], 0, t * kBN, bh);
        } else {
          mbar_expect_tx(&full[st], C::VT);
          tma_load_3d(sV(st), &tm_vt, &full[st], t * kBN, 0, bh);  // keys t*128.. of all D rows of V^T
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
      // e5m2 has the format code of bf16 in the kind::f16 descriptor; both
      // operands K-major (V arrives transposed)
      constexpr uint32_t idesc_qk = idesc_f16(kBM, kBN, true, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(kBM, D, true, false, false);
      const uint32_t aQ[2] = {smem_u32(sQ), smem_u32(sQ) + C::QT};
      bool ok = warp_wait(&bar_q, 0, ctl, kErrTimeoutTma) && warp_wait(&bar_k[0], 0, ctl, kErrTimeoutTma);
      if (ok) {
        tc_fence_after();
        for (int w = 0; w < 2; ++w)
          if (n_t[w] > 0) {
            mma_qk_f8<D>(tmem + col_s[w], aQ[w], smem_u32(sK(0)), idesc_qk);
            commit_el(&bar_s[w]);
          }
      }
      if (ok) commit_el(&bar_kempty[0]);
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
            mma_pv_f8(tmem + col_o[w], tmem + col_s[w], smem_u32(sV(sv)), idesc_pv, t > 0);
            commit_el(&bar_o[w]);
          }
          if (next && t + 1 < n_t[w]) {
            mma_qk_f8<D>(tmem + col_s[w], aQ[w], smem_u32(sK(sk1)), idesc_qk);
            commit_el(&bar_s[w]);
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
    const int tq0 = q0 + w * kBM;
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
      for (int c = 0; c < 4; ++c) tmem_ld_x32(lane_addr + col_s[w] + 32 * c, TA8_CHUNK(s, c));
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_wait(TA8_CHUNK(s, c));
      float x[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) x[j] = __uint_as_float(s[j]);
      if ((args.causal && k0 + kBN - 1 > tq0 + args.P_SEQ) || (k0 + kBN > args.N)) {
        int lim = args.N - 1 - k0;
        if (args.causal) lim = min(lim, row + args.P_SEQ - k0);
#pragma unroll
        for (int j = 0; j < 128; ++j)
          if (j > lim) x[j] = -INFINITY;
      }
      float mx8[8];
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
      const float2 sc2 = make_float2(args.scale_log2, args.scale_log2);
      const float2 nm2 = make_float2(neg_m, neg_m);
      float2 rs2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {  // four keys per packed column
          const int j = 32 * c + 4 * e;
          const float2 y0 = ffma2(make_float2(x[j], x[j + 1]), sc2, nm2);
          const float2 y1 = ffma2(make_float2(x[j + 2], x[j + 3]), sc2, nm2);
          const float2 p0 = make_float2(ex2(y0.x), ex2(y0.y));
          const float2 p1 = make_float2(ex2(y1.x), ex2(y1.y));
          rs2[0] = fadd2(rs2[0], p0);
          rs2[1] = fadd2(rs2[1], p1);
          pk[e] = pack4_e5m2(p0.x, p0.y, p1.x, p1.y);
        }
        tmem_st_x8(lane_addr + col_s[w] + 8 * c, pk);
      }
      const float2 rsa = fadd2(rs2[0], rs2[1]);
      l = l * alpha + (rsa.x + rsa.y);
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
    uint8_t* orow = reinterpret_cast<uint8_t*>(args.o) + (static_cast<size_t>(bh) * args.M + (row < args.M ? row : 0)) * D;
    if (row < args.M)
      args.lse[static_cast<size_t>(bh) * args.M + row] = (live && l > 0.f) ? (m_ref + lg2(l)) * kLn2 : -INFINITY;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float of[32];
      if (live) {
        uint32_t ov[32];
        tmem_ld_x32(lane_addr + col_o[w] + 32 * c, ov);
        tmem_ld_wait(ov);
#pragma unroll
        for (int j = 0; j < 32; ++j) of[j] = __uint_as_float(ov[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) of[j] = 0.f;
      }
      if (row < args.M) store_chunk32_e5m2(orow + 32 * c, of, inv_l);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 9) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------- host side
template <int D>
static cudaError_t launch_fwd_f8_t(const FwdMaps& maps, const FwdArgs& a, cudaStream_t stream) {
  using C = F8Cfg<D>;
  auto kern = attn_fwd_f8_kernel<D>;
  static std::atomic<bool> attr[kMaxDevices];
  cudaError_t e_attr = smem_attr_once(kern, C::SMEM, attr);
  if (e_attr != cudaSuccess) return e_attr;
  const long long pairs = (a.M + 2 * kBM - 1) / (2 * kBM);
  const long long blocks = static_cast<long long>(a.BH) * pairs;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidValue;
  kern<<<static_cast<unsigned>(blocks), 320, C::SMEM, stream>>>(maps.q, maps.k, maps.v, a);
  return cudaGetLastError();
}

cudaError_t launch_fwd_f8(int D, const FwdMaps& maps, const FwdArgs& a, cudaStream_t s) {
  if (D == 64) return launch_fwd_f8_t<64>(maps, a, s);
  if (D == 128) return launch_fwd_f8_t<128>(maps, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace ta

TA_GUARD_ACCESSOR(fwd_f8)
