// Host-side declarations shared by the kernel translation units and the
// C-ABI layer.
#pragma once
#include <atomic>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "tattn.h"

namespace ta {

struct FwdMaps {
  CUtensorMap q, k, v;     // standard: q, k, v
  CUtensorMap q2, k2, v2;  // piecewise: q2, k2 (v2 unused); jvp: tq, tk, tv
  CUtensorMap o;           // the output O (the two-tile forward stores it by TMA)
};

struct BwdMaps {
  CUtensorMap q, k, v, dO;  // piecewise: q1, k1, v, dO
  CUtensorMap q2, k2;       // piecewise only
  CUtensorMap dq, dk, dv;   // outputs, stored by TMA (built where not null)
  CUtensorMap dq2, dk2;     // piecewise outputs
  CUtensorMap q64, q264, dO64;  // piecewise D = 128: Q1, Q2, dO in 64-row boxes (the one-pass key side)
  CUtensorMap o;                // standard dQ pass forming delta (BwdArgs::delta_out)
};

// split: run the one-query-tile forward as two-CTA clusters that share each
// query tile's key tiles (fwd_split_capable(mode, D) kernels only).
bool fwd_split_capable(int mode, int D);
// One thread fails a guard check on purpose (guard build; nothing in the
// product build).
cudaError_t launch_guard_selftest(cudaStream_t s);
#ifdef TA_GUARD
// Each translation unit's guard word: returns the failure bits and copies the
// first failure's line, rejected value, shared memory base and size to
// info[0..3] (all cleared).
uint32_t guard_take_aux(uint32_t* info);
uint32_t guard_take_fwd(uint32_t* info);
uint32_t guard_take_fwd_f8(uint32_t* info);
uint32_t guard_take_bwd(uint32_t* info);
uint32_t guard_take_bwd_fused(uint32_t* info);
uint32_t guard_take_bwd_jvp(uint32_t* info);
uint32_t guard_take_merge(uint32_t* info);
uint32_t guard_take_fp32(uint32_t* info);
uint32_t guard_take_bwd_pw_steps(uint32_t* info);
#endif
cudaError_t launch_fwd(int mode, bool bf16, int D, const FwdMaps& maps, const FwdArgs& a, bool split,
                       cudaStream_t s);
// e5m2 forward: maps.q, maps.k are [BH, S, D] 8-bit maps with 128 x 128 boxes,
// maps.v the transposed V [BH, D, N] with 128 x D boxes.
cudaError_t launch_fwd_f8(int D, const FwdMaps& maps, const FwdArgs& a, cudaStream_t s);

// delta_i = sum_d O_id dO_id for BH*M rows; when acc is not null the same
// pass also zeroes acc, a [rows, D] fp32 array (the fused backward's dQ
// accumulator).
cudaError_t launch_delta(bool bf16, int D, const void* o, const void* dO, float* delta, long long rows,
                         cudaStream_t s, float* acc = nullptr);
// dq = acc * scale rounded to the element type, for rows x D elements.
cudaError_t launch_dq_convert(bool bf16, int D, const float* acc, void* dq, long long rows, float scale,
                              cudaStream_t s);
// Fused backward (dK, dV and the fp32 dQ accumulator a.dq_acc in one
// key-stationary pass) for the standard mode at the kernel head dimensions
// bwd_fused_supported() accepts.
bool bwd_fused_supported(int D);
// Query rows per streamed step of the fused backward: its Q and dO maps take
// boxes of this many rows (K and V keep 128-row boxes).
int bwd_fused_step_rows();
cudaError_t launch_bwd_fused(bool bf16, int D, const BwdMaps& maps, const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dkdv(int mode, bool bf16, int D, const BwdMaps& maps, const BwdArgs& a,
                            cudaStream_t s);
// Piecewise key side in one pass with 64-query steps (dV, dK1, dK2 of a
// key tile; maps.q64, q264, dO64 and the output maps), for the head
// dimensions bwd_pw_steps_supported() accepts.
bool bwd_pw_steps_supported(int D);
cudaError_t launch_bwd_pw_steps(bool bf16, const BwdMaps& maps, const BwdArgs& a, cudaStream_t s);
cudaError_t launch_bwd_dq(int mode, bool bf16, int D, const BwdMaps& maps, const BwdArgs& a, cudaStream_t s);

// Backward of the JVP.  Maps of the eight [BH, S, D] 16-bit inputs with
// 128-row boxes (stationary tiles) and with 64-row boxes (streamed steps).
struct JvpBwdMaps {
  CUtensorMap q128, tq128, do128, dto128, k128, tk128, v128, tv128;
  CUtensorMap q64, tq64, do64, dto64, k64, tk64, v64, tv64;
  // outputs, stored by TMA with 128-row boxes (the tangents' only where the
  // JVP kernels form them)
  CUtensorMap dq, dk, dv, dtq, dtk, dtv;
};
// eps_i = <dtO_i, O_i>, delta2_i = <dO_i, O_i> + <dtO_i, tO_i> for BH*M rows.
cudaError_t launch_jvp_delta(bool bf16, int D, const void* o, const void* dO, const void* to, const void* dto,
                             float* eps, float* delta2, long long rows, cudaStream_t s);
// keys = true: dK, dV (a.dk, a.dv); false: dQ (a.dq).  a.delta = delta2.
// When bwd_jvp_has_tangents(keys, D) the same launch also writes the
// tangents' gradients (keys: a.dtk, a.dtv; otherwise a.dtq).
bool bwd_jvp_has_tangents(bool keys, int D);
cudaError_t launch_bwd_jvp(bool keys, bool bf16, int D, const JvpBwdMaps& maps, const BwdArgs& a, cudaStream_t s);

// Fills O = 0, L = -inf (rows that see no key) for BH*M rows of D elements
// of `esize` bytes.
cudaError_t launch_empty_rows(int esize, int D, void* o, float* lse, void* to, long long rows, cudaStream_t s);
// Zero-fills n bytes (gradients of keys no query sees).
cudaError_t launch_zero(void* p, size_t bytes, cudaStream_t s);

// fp32 mode (SIMT kernels, no TMA): plain float pointers.
struct F32Ptrs {
  const float *q, *k, *v, *q2, *k2, *v2, *dO;
};
cudaError_t launch_f32_fwd(int mode, int D, const F32Ptrs& p, const FwdArgs& a, cudaStream_t s);
cudaError_t launch_f32_delta(int D, const float* o, const float* dO, float* delta, long long rows,
                             cudaStream_t s);
cudaError_t launch_f32_bwd(int mode, int D, const F32Ptrs& p, const BwdArgs& a, cudaStream_t s);
// Backward of the JVP in fp32: dq, dk, dv from q, k, v, tq, tk, tv, dO, dtO.
struct F32JvpPtrs {
  const float *q, *k, *v, *tq, *tk, *tv, *dO, *dtO;
};
cudaError_t launch_f32_jvp_delta(int D, const float* o, const float* dO, const float* to, const float* dto,
                                 float* eps, float* delta2, long long rows, cudaStream_t s);
cudaError_t launch_f32_jvp_bwd(int D, const F32JvpPtrs& p, const BwdArgs& a, cudaStream_t s);

// Merge of two partial attention states (forward and backward); dtype 0 =
// fp16, 1 = bf16, 2 = fp32.  dl may be null (zero).
struct MergePtrs {
  const void *o1, *o2, *dO;
  const float *l1, *l2, *dl;
  void *o, *do1, *do2;
  float *lse, *dl1, *dl2;
};
cudaError_t launch_merge(bool bwd, int dtype, int D, const MergePtrs& p, long long rows, cudaStream_t s);

// Opts kernel `kern` into `bytes` of dynamic shared memory on the current
// device, once per device (the attribute is per device, so a process that
// drives several GPUs sets it on each); `done` is the caller's per-kernel
// table.
constexpr int kMaxDevices = 64;
// Per-device flags and caches are atomics: host threads may make their
// first calls on a device at the same time (each then does the idempotent
// set-up itself).
template <typename K>
inline cudaError_t smem_attr_once(K kern, int bytes, std::atomic<bool> (&done)[kMaxDevices]) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && tracked) done[dev].store(true, std::memory_order_release);
  return e;
}

// attn_bwd with the choice of path: allow_fused = false keeps the two-pass
// backward (key-stationary dK/dV, then query-stationary dQ), whose only
// scratch is delta (ws >= delta's bytes); true takes the fused pass where it
// applies (ws >= attn_bwd_workspace_bytes).
ta_status bwd_entry(bool allow_fused, const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, int B, int H, int M,
                    int N, int D, ta_dtype dt, int causal, float sm_scale, void* stream);

// Profiling hooks (no-ops unless ta_profile_enable(1)).
void prof_begin(const char* name, cudaStream_t s);
void prof_end(cudaStream_t s);

}  // namespace ta
