// fp32 mode: the same five operations on float32 tensors, computed in float32
// with FFMA and accurate expf/logf (no 16-bit rounding of P or dS, no tensor
// cores).  A correctness path for fp32 callers, not a throughput path.
//
// Layout: one warp per row; each lane keeps DP/32 of the row's elements in
// registers (DP = D rounded up to a multiple of 32; lanes past D hold zeros),
// and the eight warps of a block share key (or query) tiles staged in shared
// memory with rows of DP floats.  Dot products are a lane-local FMA chain plus a five-step
// butterfly reduction, so every lane ends with the full value.
//
// Page sources as for the 16-bit kernels: "Triton fused attention tutorial,
// updated with JVP support" (_attn_fwd / _attn_fwd_inner with ENABLE_JVP,
// _attn_bwd_preprocess, _attn_bwd_dkdv, _attn_bwd_dq) and "FlagAttention
// piecewise.py" (_fwd_kernel, _bwd_kv_kernel, _bwd_q_kernel).  The online
// softmax here works in natural-log units: m = running max of s * sm_scale,
// p = exp(s * sm_scale - m), L = m + ln l.
#include "common.cuh"
#include "launch.h"

namespace ta {

constexpr int kF32Warps = 8;
constexpr int kF32Tile = 32;  // rows per shared-memory tile

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <int E>
__device__ __forceinline__ float dot_lane(const float (&a)[E], const float* b_row, int lane) {
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) s = fmaf(a[e], b_row[lane + 32 * e], s);
  return warp_sum(s);
}

// Row width in shared memory and registers: D rounded up to whole warps.
template <int D>
constexpr int padded_d() { return (D + 31) / 32 * 32; }

// Column lane + 32 e exists in a D-column row.
template <int D>
__device__ __forceinline__ bool col_ok(int lane, int e) { return D % 32 == 0 || lane + 32 * e < D; }

template <int E, int D>
__device__ __forceinline__ void load_row(float (&r)[E], const float* row, int lane) {
#pragma unroll
  for (int e = 0; e < E; ++e) r[e] = col_ok<D>(lane, e) ? row[lane + 32 * e] : 0.f;
}

template <int E, int D>
__device__ __forceinline__ void store_row(float* row, const float (&r)[E], float scale, int lane) {
#pragma unroll
  for (int e = 0; e < E; ++e)
    if (col_ok<D>(lane, e)) row[lane + 32 * e] = r[e] * scale;
}

// Cooperative copy of kF32Tile rows (from row0) of a [S, D] slice into smem
// rows of DP floats; rows past S and columns past D are zero-filled.
template <int D>
__device__ __forceinline__ void stage(float* dst, const float* src, int row0, int S) {
  constexpr int DP = padded_d<D>();
  for (int idx = threadIdx.x; idx < kF32Tile * DP; idx += blockDim.x) {
    const int r = idx / DP, c = idx % DP;
    dst[idx] = (row0 + r < S && c < D) ? src[static_cast<size_t>(row0 + r) * D + c] : 0.f;
  }
}

// ---------------------------------------------------------------- forward
template <int MODE, int D>
__global__ void __launch_bounds__(kF32Warps * 32) f32_fwd_kernel(const float* __restrict__ q,
                                                                 const float* __restrict__ k,
                                                                 const float* __restrict__ v,
                                                                 const float* __restrict__ q2,
                                                                 const float* __restrict__ k2,
                                                                 const float* __restrict__ v2, FwdArgs a) {
  constexpr int DP = padded_d<D>();
  constexpr int E = DP / 32;
  constexpr bool PW = MODE == kPiecewise, JVP = MODE == kJvp;
  __shared__ float sK[kF32Tile * DP], sV[kF32Tile * DP];
  __shared__ float sK2[(PW || JVP) ? kF32Tile * DP : 1], sV2[JVP ? kF32Tile * DP : 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int i = blockIdx.y * kF32Warps + warp;
  const bool live = i < a.M;
  const size_t qoff = (static_cast<size_t>(bh) * a.M + (live ? i : 0)) * D;
  const size_t koff = static_cast<size_t>(bh) * a.N * D;
  float qr[E], q2r[E], acc[E], uacc[E];
  load_row<E, D>(qr, q + qoff, lane);
  if constexpr (PW || JVP) load_row<E, D>(q2r, q2 + qoff, lane);  // q2 | tq
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = uacc[e] = 0.f;
  float m = -INFINITY, l = 0.f, mu = 0.f;
  int hi = a.N;  // keys this block needs
  if (a.causal) {
    const int last_row = min(a.M - 1, static_cast<int>(blockIdx.y) * kF32Warps + kF32Warps - 1);
    hi = max(0, min(a.N, last_row + a.P_SEQ + 1));
  }
  const int lim = a.causal ? min(a.N - 1, i + a.P_SEQ) : a.N - 1;
  for (int j0 = 0; j0 < hi; j0 += kF32Tile) {
    __syncthreads();
    stage<D>(sK, k + koff, j0, a.N);
    stage<D>(sV, v + koff, j0, a.N);
    if constexpr (PW || JVP) stage<D>(sK2, k2 + koff, j0, a.N);  // k2 | tk
    if constexpr (JVP) stage<D>(sV2, v2 + koff, j0, a.N);        // tv
    __syncthreads();
    if (!live) continue;
    const int jn = min(kF32Tile, lim - j0 + 1);
    for (int jj = 0; jj < jn; ++jj) {
      const int j = j0 + jj;
      float s;
      if (PW && (static_cast<long long>(i) + a.P_SEQ - j >= a.w)) s = dot_lane<E>(q2r, sK2 + jj * DP, lane);
      else s = dot_lane<E>(qr, sK + jj * DP, lane);
      s *= a.sm_scale;
      const float m_new = fmaxf(m, s);
      const float alpha = expf(m - m_new);  // m = -inf on the first key: alpha = 0
      const float p = expf(s - m_new);
      l = l * alpha + p;
      m = m_new;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(p, sV[jj * DP + lane + 32 * e], acc[e] * alpha);
      if constexpr (JVP) {
        // t = sm_scale (tq . k + q . tk)
        const float t = a.sm_scale * (dot_lane<E>(q2r, sK + jj * DP, lane) + dot_lane<E>(qr, sK2 + jj * DP, lane));
        mu = mu * alpha + p * t;
#pragma unroll
        for (int e = 0; e < E; ++e)
          uacc[e] = fmaf(p, fmaf(t, sV[jj * DP + lane + 32 * e], sV2[jj * DP + lane + 32 * e]), uacc[e] * alpha);
      }
    }
  }
  if (!live) return;
  float* orow = reinterpret_cast<float*>(a.o) + qoff;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  store_row<E, D>(orow, acc, inv, lane);
  if constexpr (JVP) {
    float tv[E];
#pragma unroll
    for (int e = 0; e < E; ++e) tv[e] = uacc[e] * inv - (mu * inv) * (acc[e] * inv);
    store_row<E, D>(reinterpret_cast<float*>(a.to) + qoff, tv, 1.f, lane);
  }
  if (lane == 0) a.lse[static_cast<size_t>(bh) * a.M + i] = l > 0.f ? m + logf(l) : -INFINITY;
  if constexpr (JVP) {  // tL = sum_j P_ij T_ij
    if (lane == 0 && a.tlse) a.tlse[static_cast<size_t>(bh) * a.M + i] = l > 0.f ? mu * inv : 0.f;
  }
}

// ------------------------------------------------------------ delta (fp32)
template <int D>
__global__ void __launch_bounds__(256) f32_delta_kernel(const float* o, const float* dO, float* delta,
                                                        long long rows) {
  constexpr int E = padded_d<D>() / 32;
  const int lane = threadIdx.x & 31;
  for (long long r = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)); r < rows;
       r += static_cast<long long>(gridDim.x) * 8) {
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (col_ok<D>(lane, e)) s = fmaf(o[r * D + lane + 32 * e], dO[r * D + lane + 32 * e], s);
    s = warp_sum(s);
    if (lane == 0) delta[r] = s;
  }
}

// ------------------------------------------------------- dQ (query rows)
template <int MODE, int D>
__global__ void __launch_bounds__(kF32Warps * 32) f32_dq_kernel(const float* __restrict__ q,
                                                                const float* __restrict__ k,
                                                                const float* __restrict__ v,
                                                                const float* __restrict__ dO,
                                                                const float* __restrict__ q2,
                                                                const float* __restrict__ k2, BwdArgs a) {
  constexpr int DP = padded_d<D>();
  constexpr int E = DP / 32;
  constexpr bool PW = MODE == kPiecewise;
  __shared__ float sK[kF32Tile * DP], sV[kF32Tile * DP], sK2[PW ? kF32Tile * DP : 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int i = blockIdx.y * kF32Warps + warp;
  const bool live = i < a.M;
  const size_t qoff = (static_cast<size_t>(bh) * a.M + (live ? i : 0)) * D;
  const size_t koff = static_cast<size_t>(bh) * a.N * D;
  float qr[E], q2r[E], dor[E], g1[E], g2[E];
  load_row<E, D>(qr, q + qoff, lane);
  if constexpr (PW) load_row<E, D>(q2r, q2 + qoff, lane);
  load_row<E, D>(dor, dO + qoff, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) g1[e] = g2[e] = 0.f;
  const float L = live ? a.lse[static_cast<size_t>(bh) * a.M + i] : 0.f;
  const float dl = live ? a.delta[static_cast<size_t>(bh) * a.M + i] : 0.f;
  int hi = a.N;
  if (a.causal) {
    const int last_row = min(a.M - 1, static_cast<int>(blockIdx.y) * kF32Warps + kF32Warps - 1);
    hi = max(0, min(a.N, last_row + a.P_SEQ + 1));
  }
  const int lim = a.causal ? min(a.N - 1, i + a.P_SEQ) : a.N - 1;
  for (int j0 = 0; j0 < hi; j0 += kF32Tile) {
    __syncthreads();
    stage<D>(sK, k + koff, j0, a.N);
    stage<D>(sV, v + koff, j0, a.N);
    if constexpr (PW) stage<D>(sK2, k2 + koff, j0, a.N);
    __syncthreads();
    if (!live) continue;
    const int jn = min(kF32Tile, lim - j0 + 1);
    for (int jj = 0; jj < jn; ++jj) {
      const int j = j0 + jj;
      const bool far = PW && (static_cast<long long>(i) + a.P_SEQ - j >= a.w);
      const float s = far ? dot_lane<E>(q2r, sK2 + jj * DP, lane) : dot_lane<E>(qr, sK + jj * DP, lane);
      const float p = expf(s * a.sm_scale - L);
      const float ds = p * (dot_lane<E>(dor, sV + jj * DP, lane) - dl);
      const float* kr = far ? sK2 + jj * DP : sK + jj * DP;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (far) g2[e] = fmaf(ds, kr[lane + 32 * e], g2[e]);
        else g1[e] = fmaf(ds, kr[lane + 32 * e], g1[e]);
      }
    }
  }
  if (!live) return;
  store_row<E, D>(reinterpret_cast<float*>(a.dq) + qoff, g1, a.sm_scale, lane);
  if constexpr (PW) store_row<E, D>(reinterpret_cast<float*>(a.dq2) + qoff, g2, a.sm_scale, lane);
}

// ------------------------------------------------------- dK, dV (key rows)
template <int MODE, int D>
__global__ void __launch_bounds__(kF32Warps * 32) f32_dkdv_kernel(const float* __restrict__ q,
                                                                  const float* __restrict__ k,
                                                                  const float* __restrict__ v,
                                                                  const float* __restrict__ dO,
                                                                  const float* __restrict__ q2,
                                                                  const float* __restrict__ k2, BwdArgs a) {
  constexpr int DP = padded_d<D>();
  constexpr int E = DP / 32;
  constexpr bool PW = MODE == kPiecewise;
  __shared__ float sQ[kF32Tile * DP], sDO[kF32Tile * DP], sQ2[PW ? kF32Tile * DP : 1];
  __shared__ float sL[kF32Tile], sDl[kF32Tile];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int j = blockIdx.y * kF32Warps + warp;
  const bool live = j < a.N;
  const size_t koff = (static_cast<size_t>(bh) * a.N + (live ? j : 0)) * D;
  const size_t qoff = static_cast<size_t>(bh) * a.M * D;
  float kr[E], k2r[E], vr[E], gk1[E], gk2[E], gv[E];
  load_row<E, D>(kr, k + koff, lane);
  if constexpr (PW) load_row<E, D>(k2r, k2 + koff, lane);
  load_row<E, D>(vr, v + koff, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) gk1[e] = gk2[e] = gv[e] = 0.f;
  int lo = 0;  // first query any key of this block is visible from
  if (a.causal) lo = max(0, static_cast<int>(blockIdx.y) * kF32Warps - a.P_SEQ);
  const int first = a.causal ? max(0, j - a.P_SEQ) : 0;  // this key's first visible query
  for (int i0 = (lo / kF32Tile) * kF32Tile; i0 < a.M; i0 += kF32Tile) {
    __syncthreads();
    stage<D>(sQ, q + qoff, i0, a.M);
    stage<D>(sDO, dO + qoff, i0, a.M);
    if constexpr (PW) stage<D>(sQ2, q2 + qoff, i0, a.M);
    for (int r = threadIdx.x; r < kF32Tile; r += blockDim.x) {
      const bool in = i0 + r < a.M;
      sL[r] = in ? a.lse[static_cast<size_t>(bh) * a.M + i0 + r] : INFINITY;
      sDl[r] = in ? a.delta[static_cast<size_t>(bh) * a.M + i0 + r] : 0.f;
    }
    __syncthreads();
    if (!live) continue;
    const int ib = max(0, first - i0);
    const int ie = min(kF32Tile, a.M - i0);
    for (int ii = ib; ii < ie; ++ii) {
      const int i = i0 + ii;
      const bool far = PW && (static_cast<long long>(i) + a.P_SEQ - j >= a.w);
      const float s = far ? dot_lane<E>(k2r, sQ2 + ii * DP, lane) : dot_lane<E>(kr, sQ + ii * DP, lane);
      const float p = expf(s * a.sm_scale - sL[ii]);
      const float ds = p * (dot_lane<E>(vr, sDO + ii * DP, lane) - sDl[ii]);
      const float* qrow = far ? sQ2 + ii * DP : sQ + ii * DP;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        gv[e] = fmaf(p, sDO[ii * DP + lane + 32 * e], gv[e]);
        if (far) gk2[e] = fmaf(ds, qrow[lane + 32 * e], gk2[e]);
        else gk1[e] = fmaf(ds, qrow[lane + 32 * e], gk1[e]);
      }
    }
  }
  if (!live) return;
  store_row<E, D>(reinterpret_cast<float*>(a.dv) + koff, gv, 1.f, lane);
  store_row<E, D>(reinterpret_cast<float*>(a.dk) + koff, gk1, a.sm_scale, lane);
  if constexpr (PW) store_row<E, D>(reinterpret_cast<float*>(a.dk2) + koff, gk2, a.sm_scale, lane);
}

// ------------------------------------------- backward of the JVP (fp32)
// Gradients of <dO, O> + <dtO, tO> with respect to q, k, v; per (i, j), with
// t = T - mu:  dT = P (dtO.v_j - eps_i),  dS = P (dO.v_j + dtO.tv_j - delta2_i)
// + t dT,  dq_i += dS k_j + dT tk_j,  dk_j += dS q_i + dT tq_i,
// dv_j += P dO_i + P t dtO_i  (dq and dk times sm_scale at the end).
template <int D>
__global__ void __launch_bounds__(256) f32_jvp_delta_kernel(const float* o, const float* dO, const float* to,
                                                            const float* dto, float* eps, float* delta2,
                                                            long long rows) {
  constexpr int E = padded_d<D>() / 32;
  const int lane = threadIdx.x & 31;
  for (long long r = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)); r < rows;
       r += static_cast<long long>(gridDim.x) * 8) {
    float e1 = 0.f, e2 = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e)
      if (col_ok<D>(lane, e)) {
        const long long x = r * D + lane + 32 * e;
        e1 = fmaf(dto[x], o[x], e1);
        e2 = fmaf(dO[x], o[x], fmaf(dto[x], to[x], e2));
      }
    e1 = warp_sum(e1);
    e2 = warp_sum(e2);
    if (lane == 0) {
      eps[r] = e1;
      delta2[r] = e2;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kF32Warps * 32) f32_jvp_dq_kernel(F32JvpPtrs P, BwdArgs a) {
  constexpr int DP = padded_d<D>();
  constexpr int E = DP / 32;
  __shared__ float sK[kF32Tile * DP], sTK[kF32Tile * DP], sV[kF32Tile * DP], sTV[kF32Tile * DP];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int i = blockIdx.y * kF32Warps + warp;
  const bool live = i < a.M;
  const size_t qoff = (static_cast<size_t>(bh) * a.M + (live ? i : 0)) * D;
  const size_t koff = static_cast<size_t>(bh) * a.N * D;
  float qr[E], tqr[E], dor[E], dtor[E], g[E];
  load_row<E, D>(qr, P.q + qoff, lane);
  load_row<E, D>(tqr, P.tq + qoff, lane);
  load_row<E, D>(dor, P.dO + qoff, lane);
  load_row<E, D>(dtor, P.dtO + qoff, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) g[e] = 0.f;
  const size_t ri = static_cast<size_t>(bh) * a.M + (live ? i : 0);
  const float L = live ? a.lse[ri] : 0.f, mu = live ? a.mu[ri] : 0.f;
  const float eps = live ? a.eps[ri] : 0.f, d2 = live ? a.delta[ri] : 0.f;
  int hi = a.N;
  if (a.causal) {
    const int last_row = min(a.M - 1, static_cast<int>(blockIdx.y) * kF32Warps + kF32Warps - 1);
    hi = max(0, min(a.N, last_row + a.P_SEQ + 1));
  }
  const int lim = a.causal ? min(a.N - 1, i + a.P_SEQ) : a.N - 1;
  for (int j0 = 0; j0 < hi; j0 += kF32Tile) {
    __syncthreads();
    stage<D>(sK, P.k + koff, j0, a.N);
    stage<D>(sTK, P.tk + koff, j0, a.N);
    stage<D>(sV, P.v + koff, j0, a.N);
    stage<D>(sTV, P.tv + koff, j0, a.N);
    __syncthreads();
    if (!live) continue;
    const int jn = min(kF32Tile, lim - j0 + 1);
    for (int jj = 0; jj < jn; ++jj) {
      const float* kr = sK + jj * DP;
      const float* tkr = sTK + jj * DP;
      const float p = expf(dot_lane<E>(qr, kr, lane) * a.sm_scale - L);
      const float t = a.sm_scale * (dot_lane<E>(tqr, kr, lane) + dot_lane<E>(qr, tkr, lane)) - mu;
      const float dtp = dot_lane<E>(dtor, sV + jj * DP, lane);
      const float dpa = dot_lane<E>(dor, sV + jj * DP, lane) + dot_lane<E>(dtor, sTV + jj * DP, lane);
      const float dT = p * (dtp - eps);
      const float dS = fmaf(t, dT, p * (dpa - d2));
#pragma unroll
      for (int e = 0; e < E; ++e) g[e] = fmaf(dS, kr[lane + 32 * e], fmaf(dT, tkr[lane + 32 * e], g[e]));
    }
  }
  if (!live) return;
  store_row<E, D>(reinterpret_cast<float*>(a.dq) + qoff, g, a.sm_scale, lane);
}

template <int D>
__global__ void __launch_bounds__(kF32Warps * 32) f32_jvp_dkdv_kernel(F32JvpPtrs P, BwdArgs a) {
  constexpr int DP = padded_d<D>();
  constexpr int E = DP / 32;
  __shared__ float sQ[kF32Tile * DP], sTQ[kF32Tile * DP], sDO[kF32Tile * DP], sDTO[kF32Tile * DP];
  __shared__ float sL[kF32Tile], sMu[kF32Tile], sEps[kF32Tile], sD2[kF32Tile];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.x;
  const int j = blockIdx.y * kF32Warps + warp;
  const bool live = j < a.N;
  const size_t koff = (static_cast<size_t>(bh) * a.N + (live ? j : 0)) * D;
  const size_t qoff = static_cast<size_t>(bh) * a.M * D;
  float kr[E], tkr[E], vr[E], tvr[E], gk[E], gv[E];
  load_row<E, D>(kr, P.k + koff, lane);
  load_row<E, D>(tkr, P.tk + koff, lane);
  load_row<E, D>(vr, P.v + koff, lane);
  load_row<E, D>(tvr, P.tv + koff, lane);
#pragma unroll
  for (int e = 0; e < E; ++e) gk[e] = gv[e] = 0.f;
  int lo = 0;
  if (a.causal) lo = max(0, static_cast<int>(blockIdx.y) * kF32Warps - a.P_SEQ);
  const int first = a.causal ? max(0, j - a.P_SEQ) : 0;
  for (int i0 = (lo / kF32Tile) * kF32Tile; i0 < a.M; i0 += kF32Tile) {
    __syncthreads();
    stage<D>(sQ, P.q + qoff, i0, a.M);
    stage<D>(sTQ, P.tq + qoff, i0, a.M);
    stage<D>(sDO, P.dO + qoff, i0, a.M);
    stage<D>(sDTO, P.dtO + qoff, i0, a.M);
    for (int r = threadIdx.x; r < kF32Tile; r += blockDim.x) {
      const bool in = i0 + r < a.M;
      const size_t g = static_cast<size_t>(bh) * a.M + (in ? i0 + r : 0);
      sL[r] = in ? a.lse[g] : INFINITY;
      sMu[r] = in ? a.mu[g] : 0.f;
      sEps[r] = in ? a.eps[g] : 0.f;
      sD2[r] = in ? a.delta[g] : 0.f;
    }
    __syncthreads();
    if (!live) continue;
    const int ib = max(0, first - i0);
    const int ie = min(kF32Tile, a.M - i0);
    for (int ii = ib; ii < ie; ++ii) {
      const float* qr = sQ + ii * DP;
      const float* tqr = sTQ + ii * DP;
      const float* dor = sDO + ii * DP;
      const float* dtor = sDTO + ii * DP;
      const float p = expf(dot_lane<E>(kr, qr, lane) * a.sm_scale - sL[ii]);
      const float t = a.sm_scale * (dot_lane<E>(kr, tqr, lane) + dot_lane<E>(tkr, qr, lane)) - sMu[ii];
      const float dtp = dot_lane<E>(vr, dtor, lane);
      const float dpa = dot_lane<E>(vr, dor, lane) + dot_lane<E>(tvr, dtor, lane);
      const float dT = p * (dtp - sEps[ii]);
      const float dS = fmaf(t, dT, p * (dpa - sD2[ii]));
      const float pt = p * t;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        gv[e] = fmaf(p, dor[lane + 32 * e], fmaf(pt, dtor[lane + 32 * e], gv[e]));
        gk[e] = fmaf(dS, qr[lane + 32 * e], fmaf(dT, tqr[lane + 32 * e], gk[e]));
      }
    }
  }
  if (!live) return;
  store_row<E, D>(reinterpret_cast<float*>(a.dv) + koff, gv, 1.f, lane);
  store_row<E, D>(reinterpret_cast<float*>(a.dk) + koff, gk, a.sm_scale, lane);
}

// ---------------------------------------------------------------- host side
template <int MODE, int D>
static cudaError_t f32_fwd_t(const F32Ptrs& p, const FwdArgs& a, cudaStream_t s) {
  dim3 grid(a.BH, (a.M + kF32Warps - 1) / kF32Warps);
  f32_fwd_kernel<MODE, D><<<grid, kF32Warps * 32, 0, s>>>(p.q, p.k, p.v, p.q2, p.k2, p.v2, a);
  return cudaGetLastError();
}

cudaError_t launch_f32_fwd(int mode, int D, const F32Ptrs& p, const FwdArgs& a, cudaStream_t s) {
#define TA_F32_FWD(MODE_, D_) \
  if (mode == MODE_ && D == D_) return f32_fwd_t<MODE_, D_>(p, a, s);
  TA_F32_FWD(kStd, 16)
  TA_F32_FWD(kStd, 32)
  TA_F32_FWD(kStd, 64)
  TA_F32_FWD(kStd, 128)
  TA_F32_FWD(kPiecewise, 16)
  TA_F32_FWD(kPiecewise, 32)
  TA_F32_FWD(kPiecewise, 64)
  TA_F32_FWD(kPiecewise, 128)
  TA_F32_FWD(kJvp, 16)
  TA_F32_FWD(kJvp, 32)
  TA_F32_FWD(kJvp, 64)
  TA_F32_FWD(kJvp, 128)
#undef TA_F32_FWD
  return cudaErrorInvalidValue;
}

cudaError_t launch_f32_delta(int D, const float* o, const float* dO, float* delta, long long rows,
                             cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  long long blocks = (rows + 7) / 8;
  if (blocks > 65535ll * 8) blocks = 65535ll * 8;
  if (D == 16) f32_delta_kernel<16><<<blocks, 256, 0, s>>>(o, dO, delta, rows);
  else if (D == 32) f32_delta_kernel<32><<<blocks, 256, 0, s>>>(o, dO, delta, rows);
  else if (D == 64) f32_delta_kernel<64><<<blocks, 256, 0, s>>>(o, dO, delta, rows);
  else if (D == 128) f32_delta_kernel<128><<<blocks, 256, 0, s>>>(o, dO, delta, rows);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

template <int MODE, int D>
static cudaError_t f32_bwd_t(const F32Ptrs& p, const BwdArgs& a, cudaStream_t s) {
  dim3 gq(a.BH, (a.M + kF32Warps - 1) / kF32Warps);
  f32_dq_kernel<MODE, D><<<gq, kF32Warps * 32, 0, s>>>(p.q, p.k, p.v, p.dO, p.q2, p.k2, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 gk(a.BH, (a.N + kF32Warps - 1) / kF32Warps);
  f32_dkdv_kernel<MODE, D><<<gk, kF32Warps * 32, 0, s>>>(p.q, p.k, p.v, p.dO, p.q2, p.k2, a);
  return cudaGetLastError();
}

cudaError_t launch_f32_bwd(int mode, int D, const F32Ptrs& p, const BwdArgs& a, cudaStream_t s) {
  if (mode == kStd && D == 16) return f32_bwd_t<kStd, 16>(p, a, s);
  if (mode == kStd && D == 32) return f32_bwd_t<kStd, 32>(p, a, s);
  if (mode == kPiecewise && D == 16) return f32_bwd_t<kPiecewise, 16>(p, a, s);
  if (mode == kPiecewise && D == 32) return f32_bwd_t<kPiecewise, 32>(p, a, s);
  if (mode == kStd && D == 64) return f32_bwd_t<kStd, 64>(p, a, s);
  if (mode == kStd && D == 128) return f32_bwd_t<kStd, 128>(p, a, s);
  if (mode == kPiecewise && D == 64) return f32_bwd_t<kPiecewise, 64>(p, a, s);
  if (mode == kPiecewise && D == 128) return f32_bwd_t<kPiecewise, 128>(p, a, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_f32_jvp_delta(int D, const float* o, const float* dO, const float* to, const float* dto,
                                 float* eps, float* delta2, long long rows, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  long long blocks = (rows + 7) / 8;
  if (blocks > 65535ll * 8) blocks = 65535ll * 8;
  if (D == 16) f32_jvp_delta_kernel<16><<<blocks, 256, 0, s>>>(o, dO, to, dto, eps, delta2, rows);
  else if (D == 32) f32_jvp_delta_kernel<32><<<blocks, 256, 0, s>>>(o, dO, to, dto, eps, delta2, rows);
  else if (D == 64) f32_jvp_delta_kernel<64><<<blocks, 256, 0, s>>>(o, dO, to, dto, eps, delta2, rows);
  else if (D == 128) f32_jvp_delta_kernel<128><<<blocks, 256, 0, s>>>(o, dO, to, dto, eps, delta2, rows);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

template <int D>
static cudaError_t f32_jvp_bwd_t(const F32JvpPtrs& p, const BwdArgs& a, cudaStream_t s) {
  dim3 gq(a.BH, (a.M + kF32Warps - 1) / kF32Warps);
  f32_jvp_dq_kernel<D><<<gq, kF32Warps * 32, 0, s>>>(p, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 gk(a.BH, (a.N + kF32Warps - 1) / kF32Warps);
  f32_jvp_dkdv_kernel<D><<<gk, kF32Warps * 32, 0, s>>>(p, a);
  return cudaGetLastError();
}

cudaError_t launch_f32_jvp_bwd(int D, const F32JvpPtrs& p, const BwdArgs& a, cudaStream_t s) {
  if (D == 16) return f32_jvp_bwd_t<16>(p, a, s);
  if (D == 32) return f32_jvp_bwd_t<32>(p, a, s);
  if (D == 64) return f32_jvp_bwd_t<64>(p, a, s);
  if (D == 128) return f32_jvp_bwd_t<128>(p, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace ta

TA_GUARD_ACCESSOR(fp32)
