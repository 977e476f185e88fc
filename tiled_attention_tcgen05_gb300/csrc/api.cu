// C ABI of libtattn.so: argument validation, TMA tensor-map encoding, kernel
// dispatch, the device error word behind the bounded waits, and per-kernel
// CUDA-event timing.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "tattn.h"
#include "common.cuh"
#include "launch.h"

namespace ta {

// ------------------------------------------------------------ error word
static __device__ uint32_t g_err_word;

static uint32_t* error_word_ptr() {
  static std::atomic<uint32_t*> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  uint32_t* w = cache[dev].load(std::memory_order_acquire);
  if (!w) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
    w = static_cast<uint32_t*>(p);
    cache[dev].store(w, std::memory_order_release);
  }
  return w;
}

// ------------------------------------------------------------ guard build
// "unit:line value .. smem base+size" of the first guard failure seen by the
// last ta_sync_status that found one (guard build), "" otherwise.
static char g_guard_last[128] = "";

static ta_status guard_status() {
#ifdef TA_GUARD
  struct Unit {
    const char* name;
    uint32_t (*take)(uint32_t*);
  };
  static const Unit units[] = {{"aux.cu", guard_take_aux},       {"fwd.cu", guard_take_fwd},
                               {"fwd_f8.cu", guard_take_fwd_f8}, {"bwd.cu", guard_take_bwd},
                               {"bwd_fused.cu", guard_take_bwd_fused}, {"bwd_jvp.cu", guard_take_bwd_jvp},
                               {"merge.cu", guard_take_merge},   {"fp32.cu", guard_take_fp32},
                               {"bwd_pw_steps.cu", guard_take_bwd_pw_steps}};
  bool failed = false;
  for (const Unit& u : units) {
    uint32_t info[4] = {0u, 0u, 0u, 0u};  // line, rejected value, shared memory base, size
    if (u.take(info) != 0u) {
      if (!failed)
        std::snprintf(g_guard_last, sizeof(g_guard_last), "%s:%u value 0x%x smem 0x%x+0x%x", u.name, info[0],
                      info[1], info[2], info[3]);
      failed = true;
    }
  }
  return failed ? TA_ERR_GUARD : TA_OK;
#else
  return TA_OK;
#endif
}

static uint64_t g_timeout_ns = [] {
  const char* e = std::getenv("TA_WAIT_TIMEOUT_MS");
  long v = e ? std::strtol(e, nullptr, 10) : 0;
  if (v <= 0) v = 2000;
  return static_cast<uint64_t>(v) * 1000000ull;
}();

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The driver call that encodes tensor maps needs a current context.  A host
// thread whose first CUDA work is a call into this library has none yet
// (cudaGetDevice and the cached look-ups bind nothing), so when the thread
// has no current context the current device's primary context is bound
// first (cudaSetDevice does that).  A thread that has one, including one in
// the middle of a stream capture, is left as it is.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

static bool ensure_context() {
  static CtxGetCurrentFn get = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (get && get(&c) == CUDA_SUCCESS && c != nullptr) return true;
  int dev = 0;
  return cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess;
}

// [BH, S, D] 16-bit tensor viewed as a 3-D map with 64 x box_rows x 1 boxes
// and 128-byte swizzle; rows past S (and, for D < 64, columns past D) read as
// zeros.
static bool make_map(CUtensorMap* map, const void* ptr, long long BH, long long S, int D, bool bf16,
                     int box_rows = 128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !ensure_context()) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(S) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                  const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// [BH, rows, cols] 8-bit tensor as a 3-D map with box_cols x box_rows x 1
// boxes and 128-byte swizzle (cols * 1 byte is the row stride; columns past
// cols and rows past `rows` read as zeros).
static bool make_map_u8(CUtensorMap* map, const void* ptr, long long BH, long long rows, long long cols, int box_cols,
                        int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !ensure_context()) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows * cols)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------- profiling
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
static std::mutex g_prof_mu;
static std::atomic<bool> g_prof_on{false};
static std::vector<ProfRec> g_prof_recs;
static std::vector<cudaEvent_t> g_prof_pool;
static size_t g_prof_pool_next = 0;
static const char* g_prof_pending = nullptr;
static cudaEvent_t g_prof_pending_ev = nullptr;

static cudaEvent_t prof_event() {
  if (g_prof_pool_next == g_prof_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_prof_pool.push_back(e);
  }
  return g_prof_pool[g_prof_pool_next++];
}

void prof_begin(const char* name, cudaStream_t s) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_pending = name;
  g_prof_pending_ev = prof_event();
  if (g_prof_pending_ev) cudaEventRecord(g_prof_pending_ev, s);
}

void prof_end(cudaStream_t s) {
  if (!g_prof_on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_pending || !g_prof_pending_ev) return;
  cudaEvent_t e = prof_event();
  if (!e) return;
  cudaEventRecord(e, s);
  g_prof_recs.push_back({g_prof_pending, g_prof_pending_ev, e});
  g_prof_pending = nullptr;
}

// --------------------------------------------------------------- checks
static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Problem {
  long long BH;
  int M, N, D;
  bool bf16;
  bool f32;   // fp32 mode: SIMT kernels
  int esize;  // bytes per element
  float sm_scale;
};

static ta_status check_common(int B, int H, int M, int N, int D, ta_dtype dt, float sm_scale, Problem* pr) {
  if (B < 0 || H < 0 || M < 0 || N < 0) return TA_ERR_INVALID_ARG;
  if (dt != TA_F16 && dt != TA_BF16 && dt != TA_F32) return TA_ERR_UNSUPPORTED;
  if (D != 16 && D != 32 && D != 64 && D != 128) return TA_ERR_UNSUPPORTED;
  const long long BH = static_cast<long long>(B) * H;
  if (BH > 0x7fffffffll) return TA_ERR_INVALID_ARG;
  if ((M + kBM - 1) / kBM > 65535 || (N + kBN - 1) / kBN > 65535) return TA_ERR_UNSUPPORTED;
  pr->BH = BH;
  pr->M = M;
  pr->N = N;
  pr->D = D;
  pr->bf16 = (dt == TA_BF16);
  pr->f32 = (dt == TA_F32);
  pr->esize = pr->f32 ? 4 : 2;
  pr->sm_scale = (std::isfinite(sm_scale) && sm_scale > 0.f) ? sm_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return TA_OK;
}

static ta_status check_ptrs(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (!p) return TA_ERR_INVALID_ARG;
  for (const void* p : ps)
    if (!aligned16(p)) return TA_ERR_ALIGNMENT;
  return TA_OK;
}

static ta_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TA_OK : TA_ERR_CUDA; }

// Heads per group of the two-tile forward's tile order (grouped_tile): as
// many as keep the group's K and V within a quarter of the 129 MB L2, so the
// CTAs resident at once re-read them from L2, but at least kGroupHeads.
// Larger groups put more of the heaviest causal tiles first: with groups of
// 8 heads at B4 H16 S2048 the last group's heaviest tiles start late and the
// SMs sit idle a fifth of the time (groups of 32 there; 8 at B1 H32 S8192).
static int fwd_group_heads(const Problem& p) {
  const long long per_head = 2ll * p.N * p.D * p.esize;
  long long g = per_head > 0 ? (32ll << 20) / per_head : p.BH;
  if (g < kGroupHeads) g = kGroupHeads;
  if (g > p.BH) g = p.BH;
  return g < 1 ? 1 : static_cast<int>(g);
}

static FwdArgs fwd_args(const Problem& p, int causal, int w, void* o, float* lse, void* to, float* tlse) {
  FwdArgs a;
  a.o = o;
  a.lse = lse;
  a.to = to;
  a.tlse = tlse;
  a.BH = static_cast<int>(p.BH);
  a.M = p.M;
  a.N = p.N;
  a.P_SEQ = p.N - p.M;
  a.num_q_tiles = (p.M + kBM - 1) / kBM;
  a.causal = causal ? 1 : 0;
  a.w = w;
  a.group_heads = fwd_group_heads(p);
  a.sm_scale = p.sm_scale;
  a.scale_log2 = p.sm_scale * kLog2e;
  a.dg = p.D;
  a.err = error_word_ptr();
  a.timeout_ns = g_timeout_ns;
  return a;
}

static BwdArgs bwd_args(const Problem& p, int causal, int w, const float* lse, const float* delta) {
  BwdArgs a{};
  a.lse = lse;
  a.delta = delta;
  a.BH = static_cast<int>(p.BH);
  a.M = p.M;
  a.N = p.N;
  a.P_SEQ = p.N - p.M;
  a.causal = causal ? 1 : 0;
  a.w = w;
  a.sm_scale = p.sm_scale;
  a.scale_log2 = p.sm_scale * kLog2e;
  a.dg = p.D;
  a.err = error_word_ptr();
  a.timeout_ns = g_timeout_ns;
  return a;
}

// Head dimension the 16-bit tensor-core kernels are instantiated for: D = 16
// and 32 run the D = 64 kernels, whose TMA boxes are 64 columns wide; the
// columns past D read as zeros and are never stored.
static int kernel_d(int D) { return D <= 64 ? 64 : 128; }

static size_t delta_bytes(long long BH, int M) {
  return (static_cast<size_t>(BH) * static_cast<size_t>(M) * sizeof(float) + 255) & ~size_t(255);
}

// attn_bwd_fused (16-bit, D = 128) runs the fused key-stationary kernel,
// which adds dQ into an fp32 accumulator [BH, M, D] kept in the workspace
// after delta.
static bool bwd_fused_applies(int D, ta_dtype dt) {
  return (dt == TA_F16 || dt == TA_BF16) && bwd_fused_supported(kernel_d(D)) && kernel_d(D) == D;
}

static size_t dq_acc_bytes(long long BH, int M, int D) {
  return static_cast<size_t>(BH) * static_cast<size_t>(M) * static_cast<size_t>(D) * sizeof(float);
}

// ---------------------------------------- key split of the one-tile forward
// The JVP forward and the D = 128 piecewise forward run one 128-row query
// tile per CTA (one CTA per SM: each takes all 512 TMEM columns).  When the
// grid is less than one wave, the slowest CTA (the query tile with the most
// key tiles) sets the kernel's time; the key split gives each query tile a
// cluster of two CTAs that take half of its key tiles each.  The choice
// compares the two grids' makespans under list scheduling: CTAs start in
// launch order on the first free SM, a CTA costs its key tiles plus
// kSplitFixed tiles of set-up and epilogue, and the first CTA of a pair
// kSplitMerge more for reading its partner's state; the split must save 15 %.
// The fixed cost is measured: the JVP forward on [2, 8, 1024, 64] takes
// ~27 us whether its CTAs walk 8 key tiles (one wave) or at most 4 (the
// split: 256 CTAs, two waves), i.e. a CTA's set-up and epilogue cost about
// as much as two to three key tiles.  Long key ranges with few query tiles
// (decoding-like shapes) are where the split pays.
static std::atomic<int> g_fwd_split_mode{0};  // 0 by the cost model, 1 never, 2 wherever a kernel can
constexpr double kSplitFixed = 2.5, kSplitMerge = 0.5, kSplitGain = 0.85;

static double list_makespan(const std::vector<double>& costs, int sms) {
  std::vector<double> free_at(static_cast<size_t>(sms), 0.0);  // min-heap of SM free times
  auto cmp = [](double a, double b) { return a > b; };
  double span = 0.0;
  for (double c : costs) {
    std::pop_heap(free_at.begin(), free_at.end(), cmp);
    free_at.back() += c;
    span = std::max(span, free_at.back());
    std::push_heap(free_at.begin(), free_at.end(), cmp);
  }
  return span;
}

static int device_sms() {
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

static bool fwd_split_plan(int mode, const Problem& p, int causal, int sms) {
  if (p.f32 || p.BH == 0 || p.M == 0 || p.N == 0 || !fwd_split_capable(mode, kernel_d(p.D))) return false;
  const int nq = (p.M + kBM - 1) / kBM;
  if (2ll * nq > 65535) return false;
  const int setting = g_fwd_split_mode.load(std::memory_order_relaxed);
  if (setting == 1) return false;
  if (setting == 2) return true;
  if (sms <= 0 || p.BH * nq > sms) return false;  // a wave or more: the grid balances itself
  std::vector<double> one, two;
  for (int y = 0; y < nq; ++y) {  // launch order: heaviest query tile first, heads fastest
    const int n = kv_tiles_for((nq - 1 - y) * kBM, p.M, p.N, p.N - p.M, causal);
    const int h = (n + 1) / 2;
    for (long long x = 0; x < p.BH; ++x) {
      one.push_back(n + kSplitFixed);
      two.push_back(h + kSplitFixed + (n - h > 0 ? kSplitMerge : 0.0));
      two.push_back(n - h + kSplitFixed);
    }
  }
  return list_makespan(two, sms) < kSplitGain * list_makespan(one, sms);
}

static ta_status run_fwd(int mode, const Problem& p, const void* q, const void* k, const void* v,
                         const void* q2, const void* k2, const void* v2, void* o, float* lse, void* to,
                         float* tlse, int causal, int w, cudaStream_t s) {
  if (p.BH == 0 || p.M == 0) return TA_OK;
  if (p.N == 0) {
    prof_begin("empty_rows", s);
    cudaError_t e = launch_empty_rows(p.esize, p.D, o, lse, to, p.BH * p.M, s);
    if (e == cudaSuccess && tlse) e = launch_zero(tlse, static_cast<size_t>(p.BH) * p.M * sizeof(float), s);
    prof_end(s);
    return cuda_status(e);
  }
  static const char* f32_names[3] = {"attn_fwd_f32", "piecewise_fwd_f32", "attn_fwd_jvp_f32"};
  if (p.f32) {
    F32Ptrs fp{static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
               static_cast<const float*>(q2), static_cast<const float*>(k2), static_cast<const float*>(v2),
               nullptr};
    FwdArgs a = fwd_args(p, causal, w, o, lse, to, tlse);
    prof_begin(f32_names[mode], s);
    cudaError_t e = launch_f32_fwd(mode, p.D, fp, a, s);
    prof_end(s);
    return cuda_status(e);
  }
  FwdMaps maps;
  bool ok = make_map(&maps.q, q, p.BH, p.M, p.D, p.bf16) && make_map(&maps.k, k, p.BH, p.N, p.D, p.bf16) &&
            make_map(&maps.v, v, p.BH, p.N, p.D, p.bf16) &&
            make_map(&maps.q2, q2 ? q2 : q, p.BH, p.M, p.D, p.bf16) &&
            make_map(&maps.k2, k2 ? k2 : k, p.BH, p.N, p.D, p.bf16) &&
            make_map(&maps.v2, v2 ? v2 : v, p.BH, p.N, p.D, p.bf16) && make_map(&maps.o, o, p.BH, p.M, p.D, p.bf16);
  if (!ok) return TA_ERR_CUDA;
  FwdArgs a = fwd_args(p, causal, w, o, lse, to, tlse);
  static const char* names[3] = {"attn_fwd", "piecewise_fwd", "attn_fwd_jvp"};
  prof_begin(names[mode], s);
  cudaError_t e = launch_fwd(mode, p.bf16, kernel_d(p.D), maps, a, fwd_split_plan(mode, p, causal, device_sms()), s);
  prof_end(s);
  return cuda_status(e);
}

// Maps of the gradients the backward kernels store by TMA (those that are
// not null).
static bool make_grad_maps(BwdMaps* m, const Problem& p, void* dq, void* dk, void* dv, void* dq2 = nullptr,
                           void* dk2 = nullptr) {
  return (!dq || make_map(&m->dq, dq, p.BH, p.M, p.D, p.bf16)) &&
         (!dk || make_map(&m->dk, dk, p.BH, p.N, p.D, p.bf16)) &&
         (!dv || make_map(&m->dv, dv, p.BH, p.N, p.D, p.bf16)) &&
         (!dq2 || make_map(&m->dq2, dq2, p.BH, p.M, p.D, p.bf16)) &&
         (!dk2 || make_map(&m->dk2, dk2, p.BH, p.N, p.D, p.bf16));
}

static ta_status run_bwd(int mode, const Problem& p, const void* q, const void* k, const void* v,
                         const void* q2, const void* k2, const void* o, const float* lse, const void* dO,
                         void* dq, void* dk, void* dq2, void* dk2, void* dv, void* ws, size_t ws_bytes,
                         int causal, int w, cudaStream_t s, bool fused = false) {
  if (p.BH == 0) return TA_OK;
  const bool pw = (mode == kPiecewise);
  const size_t kv_bytes = static_cast<size_t>(p.BH) * p.N * p.D * p.esize;
  if (p.M == 0) {  // no query: every key/value gradient is zero
    cudaError_t e = launch_zero(dk, kv_bytes, s);
    if (e == cudaSuccess) e = launch_zero(dv, kv_bytes, s);
    if (e == cudaSuccess && pw) e = launch_zero(dk2, kv_bytes, s);
    return cuda_status(e);
  }
  const bool use_acc = fused && !pw && !p.f32 && p.N > 0;
  // The 16-bit two-pass backward (standard and piecewise) forms delta inside
  // its dQ pass, which then runs before the key side; the fp32 mode and the
  // fused backward run the delta pass first.
  const bool dq_forms_delta = !p.f32 && !use_acc;
  const size_t db = delta_bytes(p.BH, p.M);
  if (ws_bytes < db || (use_acc && ws_bytes - db < dq_acc_bytes(p.BH, p.M, p.D))) return TA_ERR_INVALID_ARG;
  float* delta = static_cast<float*>(ws);
  float* acc = use_acc ? reinterpret_cast<float*>(static_cast<char*>(ws) + db) : nullptr;
  cudaError_t e = cudaSuccess;
  if (!dq_forms_delta) {
    prof_begin("bwd_delta", s);
    e = p.f32 ? launch_f32_delta(p.D, static_cast<const float*>(o), static_cast<const float*>(dO), delta,
                                 p.BH * p.M, s)
              : launch_delta(p.bf16, p.D, o, dO, delta, p.BH * p.M, s, acc);
    prof_end(s);
    if (e != cudaSuccess) return TA_ERR_CUDA;
  }
  const size_t q_bytes = static_cast<size_t>(p.BH) * p.M * p.D * p.esize;
  if (p.N == 0) {
    e = launch_zero(dq, q_bytes, s);
    if (e == cudaSuccess && pw) e = launch_zero(dq2, q_bytes, s);
    return cuda_status(e);
  }
  if (p.f32) {
    F32Ptrs fp{static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v),
               static_cast<const float*>(q2), static_cast<const float*>(k2), nullptr,
               static_cast<const float*>(dO)};
    BwdArgs a = bwd_args(p, causal, w, lse, delta);
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.dq2 = dq2;
    a.dk2 = dk2;
    prof_begin(pw ? "piecewise_bwd_f32" : "attn_bwd_f32", s);
    e = launch_f32_bwd(mode, p.D, fp, a, s);
    prof_end(s);
    return cuda_status(e);
  }
  BwdMaps maps;
  bool ok = make_map(&maps.q, q, p.BH, p.M, p.D, p.bf16) && make_map(&maps.k, k, p.BH, p.N, p.D, p.bf16) &&
            make_map(&maps.v, v, p.BH, p.N, p.D, p.bf16) && make_map(&maps.dO, dO, p.BH, p.M, p.D, p.bf16) &&
            make_map(&maps.q2, q2 ? q2 : q, p.BH, p.M, p.D, p.bf16) &&
            make_map(&maps.k2, k2 ? k2 : k, p.BH, p.N, p.D, p.bf16) && make_grad_maps(&maps, p, dq, dk, dv, dq2, dk2);
  if (!ok) return TA_ERR_CUDA;
  BwdArgs a = bwd_args(p, causal, w, lse, delta);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dq2 = dq2;
  a.dk2 = dk2;
  if (use_acc) {  // dK, dV and the dQ accumulator in one pass, then dQ = sm_scale * acc
    BwdMaps fm = maps;  // Q and dO stream in steps of bwd_fused_step_rows() rows
    if (!make_map(&fm.q, q, p.BH, p.M, p.D, p.bf16, bwd_fused_step_rows()) ||
        !make_map(&fm.dO, dO, p.BH, p.M, p.D, p.bf16, bwd_fused_step_rows()))
      return TA_ERR_CUDA;
    a.dq_acc = acc;
    prof_begin("attn_bwd_fused", s);
    e = launch_bwd_fused(p.bf16, p.D, fm, a, s);
    prof_end(s);
    if (e != cudaSuccess) return TA_ERR_CUDA;
    prof_begin("bwd_dq_convert", s);
    e = launch_dq_convert(p.bf16, p.D, acc, dq, p.BH * p.M, p.sm_scale, s);
    prof_end(s);
    return cuda_status(e);
  }
  // dQ, forming delta (dq_forms_delta holds on every path that reaches here),
  // then the key side, which reads delta
  if (!make_map(&maps.o, o, p.BH, p.M, p.D, p.bf16)) return TA_ERR_CUDA;
  a.delta_out = delta;
  prof_begin(pw ? "piecewise_bwd_dq" : "attn_bwd_dq", s);
  e = launch_bwd_dq(mode, p.bf16, kernel_d(p.D), maps, a, s);
  prof_end(s);
  if (e != cudaSuccess) return TA_ERR_CUDA;
  a.delta_out = nullptr;
  prof_begin(pw ? "piecewise_bwd_dkdv" : "attn_bwd_dkdv", s);
  if (pw && bwd_pw_steps_supported(kernel_d(p.D))) {  // the key side in one pass, 64-query steps
    if (!make_map(&maps.q64, q, p.BH, p.M, p.D, p.bf16, 64) || !make_map(&maps.q264, q2, p.BH, p.M, p.D, p.bf16, 64) ||
        !make_map(&maps.dO64, dO, p.BH, p.M, p.D, p.bf16, 64)) {
      prof_end(s);
      return TA_ERR_CUDA;
    }
    e = launch_bwd_pw_steps(p.bf16, maps, a, s);
  } else {
    e = launch_bwd_dkdv(mode, p.bf16, kernel_d(p.D), maps, a, s);
  }
  prof_end(s);
  return cuda_status(e);
}

// Backward of the JVP.  The workspace holds eps = <dtO, O> and
// delta2 = <dO, O> + <dtO, tO> per query row.  The tangents' gradients are the
// plain backward with dO := dtO (whose delta is eps): the JVP kernels form
// them alongside the primal gradients where TMEM has room (dtK and dtV at
// D <= 64, dtQ at every D), the plain backward's dK/dV kernel otherwise.
static ta_status run_bwd_jvp(const Problem& p, const void* q, const void* k, const void* v, const void* tq,
                             const void* tk, const void* tv, const void* o, const float* lse, const void* to,
                             const float* tlse, const void* dO, const void* dtO, void* dq, void* dk, void* dv,
                             void* dtq, void* dtk, void* dtv, void* ws, size_t ws_bytes, int causal,
                             cudaStream_t s) {
  if (p.BH == 0) return TA_OK;
  const size_t kv_bytes = static_cast<size_t>(p.BH) * p.N * p.D * p.esize;
  if (p.M == 0) {  // no query: every key-side gradient is zero
    cudaError_t e = cudaSuccess;
    for (void* g : {dk, dv, dtk, dtv})
      if (e == cudaSuccess) e = launch_zero(g, kv_bytes, s);
    return cuda_status(e);
  }
  const size_t rb = delta_bytes(p.BH, p.M);
  if (ws_bytes < 2 * rb) return TA_ERR_INVALID_ARG;
  float* eps = static_cast<float*>(ws);
  float* delta2 = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + rb);
  prof_begin("bwd_jvp_delta", s);
  cudaError_t e = p.f32 ? launch_f32_jvp_delta(p.D, static_cast<const float*>(o), static_cast<const float*>(dO),
                                               static_cast<const float*>(to), static_cast<const float*>(dtO), eps,
                                               delta2, p.BH * p.M, s)
                        : launch_jvp_delta(p.bf16, p.D, o, dO, to, dtO, eps, delta2, p.BH * p.M, s);
  prof_end(s);
  if (e != cudaSuccess) return TA_ERR_CUDA;
  const size_t q_bytes = static_cast<size_t>(p.BH) * p.M * p.D * p.esize;
  if (p.N == 0) {
    e = launch_zero(dq, q_bytes, s);
    if (e == cudaSuccess) e = launch_zero(dtq, q_bytes, s);
    return cuda_status(e);
  }
  BwdArgs at = bwd_args(p, causal, 0, lse, eps);  // tangents: plain backward of dtO
  at.dq = dtq;
  at.dk = dtk;
  at.dv = dtv;
  BwdArgs ap = bwd_args(p, causal, 0, lse, delta2);  // primal gradients
  ap.mu = tlse;
  ap.eps = eps;
  ap.dq = dq;
  ap.dk = dk;
  ap.dv = dv;
  if (p.f32) {
    F32Ptrs fp{static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v), nullptr,
               nullptr, nullptr, static_cast<const float*>(dtO)};
    prof_begin("attn_bwd_jvp_tangents_f32", s);
    e = launch_f32_bwd(kStd, p.D, fp, at, s);
    prof_end(s);
    if (e != cudaSuccess) return TA_ERR_CUDA;
    F32JvpPtrs jp{static_cast<const float*>(q),  static_cast<const float*>(k),  static_cast<const float*>(v),
                  static_cast<const float*>(tq), static_cast<const float*>(tk), static_cast<const float*>(tv),
                  static_cast<const float*>(dO), static_cast<const float*>(dtO)};
    prof_begin("attn_bwd_jvp_f32", s);
    e = launch_f32_jvp_bwd(p.D, jp, ap, s);
    prof_end(s);
    return cuda_status(e);
  }
  BwdMaps maps;
  JvpBwdMaps jm;
  bool ok = make_map(&maps.q, q, p.BH, p.M, p.D, p.bf16) && make_map(&maps.k, k, p.BH, p.N, p.D, p.bf16) &&
            make_map(&maps.v, v, p.BH, p.N, p.D, p.bf16) && make_map(&maps.dO, dtO, p.BH, p.M, p.D, p.bf16);
  maps.q2 = maps.q;
  maps.k2 = maps.k;
  const void* mrows[4] = {q, tq, dO, dtO};
  const void* nrows[4] = {k, tk, v, tv};
  CUtensorMap* m128[4] = {&jm.q128, &jm.tq128, &jm.do128, &jm.dto128};
  CUtensorMap* m64[4] = {&jm.q64, &jm.tq64, &jm.do64, &jm.dto64};
  CUtensorMap* n128[4] = {&jm.k128, &jm.tk128, &jm.v128, &jm.tv128};
  CUtensorMap* n64[4] = {&jm.k64, &jm.tk64, &jm.v64, &jm.tv64};
  for (int i = 0; ok && i < 4; ++i)
    ok = make_map(m128[i], mrows[i], p.BH, p.M, p.D, p.bf16, 128) &&
         make_map(m64[i], mrows[i], p.BH, p.M, p.D, p.bf16, 64) &&
         make_map(n128[i], nrows[i], p.BH, p.N, p.D, p.bf16, 128) &&
         make_map(n64[i], nrows[i], p.BH, p.N, p.D, p.bf16, 64);
  if (!ok || !make_grad_maps(&maps, p, dtq, dtk, dtv)) return TA_ERR_CUDA;
  const int kd = kernel_d(p.D);
  // the JVP kernels write the tangents' gradients too where TMEM has room;
  // otherwise the plain backward of dtO computes them
  if (bwd_jvp_has_tangents(true, kd)) {
    ap.dtk = dtk;
    ap.dtv = dtv;
  } else {
    prof_begin("attn_bwd_jvp_tangents_dkdv", s);
    e = launch_bwd_dkdv(kStd, p.bf16, kd, maps, at, s);
    prof_end(s);
    if (e != cudaSuccess) return TA_ERR_CUDA;
  }
  if (bwd_jvp_has_tangents(false, kd)) {
    ap.dtq = dtq;
  } else {
    prof_begin("attn_bwd_jvp_tangents_dq", s);
    e = launch_bwd_dq(kStd, p.bf16, kd, maps, at, s);
    prof_end(s);
    if (e != cudaSuccess) return TA_ERR_CUDA;
  }
  ok = make_map(&jm.dq, dq, p.BH, p.M, p.D, p.bf16) && make_map(&jm.dk, dk, p.BH, p.N, p.D, p.bf16) &&
       make_map(&jm.dv, dv, p.BH, p.N, p.D, p.bf16) &&
       (!ap.dtq || make_map(&jm.dtq, dtq, p.BH, p.M, p.D, p.bf16)) &&
       (!ap.dtk || make_map(&jm.dtk, dtk, p.BH, p.N, p.D, p.bf16)) &&
       (!ap.dtv || make_map(&jm.dtv, dtv, p.BH, p.N, p.D, p.bf16));
  if (!ok) return TA_ERR_CUDA;
  prof_begin("attn_bwd_jvp_dkdv", s);
  e = launch_bwd_jvp(true, p.bf16, kd, jm, ap, s);
  prof_end(s);
  if (e != cudaSuccess) return TA_ERR_CUDA;
  prof_begin("attn_bwd_jvp_dq", s);
  e = launch_bwd_jvp(false, p.bf16, kd, jm, ap, s);
  prof_end(s);
  return cuda_status(e);
}

// attn_bwd with the choice of path: allow_fused = false keeps the two-pass
// backward (dK/dV pass, then dQ pass), whose only scratch is delta.
ta_status bwd_entry(bool allow_fused, const void* q, const void* k, const void* v, const void* o, const float* lse,
                    const void* dO, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, int B, int H, int M,
                    int N, int D, ta_dtype dt, int causal, float sm_scale, void* stream) {
  Problem p;
  ta_status st = check_common(B, H, M, N, D, dt, sm_scale, &p);
  if (st != TA_OK) return st;
  if (p.BH == 0 || (M == 0 && N == 0)) return TA_OK;
  if (M == 0) st = check_ptrs({dk, dv});
  else if (N == 0) st = check_ptrs({o, dO, dq, ws});
  else st = check_ptrs({q, k, v, o, lse, dO, dq, dk, dv, ws});
  if (st != TA_OK) return st;
  return run_bwd(kStd, p, q, k, v, nullptr, nullptr, o, lse, dO, dq, dk, nullptr, nullptr, dv, ws, ws_bytes,
                 causal, 0, static_cast<cudaStream_t>(stream), allow_fused && bwd_fused_applies(D, dt));
}

}  // namespace ta

using namespace ta;

extern "C" {

int ta_guard_build(void) { return ta::kGuardBuild ? 1 : 0; }

const char* ta_guard_last(void) { return ta::g_guard_last; }

ta_status ta_selftest_guard(void* stream) {
  return ta::launch_guard_selftest(static_cast<cudaStream_t>(stream)) == cudaSuccess ? TA_OK : TA_ERR_CUDA;
}

const char* ta_status_str(ta_status s) {
  switch (s) {
    case TA_OK: return "TA_OK";
    case TA_ERR_INVALID_ARG: return "TA_ERR_INVALID_ARG";
    case TA_ERR_UNSUPPORTED: return "TA_ERR_UNSUPPORTED";
    case TA_ERR_ALIGNMENT: return "TA_ERR_ALIGNMENT";
    case TA_ERR_CUDA: return "TA_ERR_CUDA";
    case TA_ERR_TIMEOUT: return "TA_ERR_TIMEOUT";
    case TA_ERR_GUARD: return "TA_ERR_GUARD";
  }
  return "TA_ERR_UNKNOWN";
}

void ta_set_fwd_kv_split(int mode) { g_fwd_split_mode.store(mode == 1 || mode == 2 ? mode : 0); }

int ta_fwd_kv_split(int entry, int B, int H, int M, int N, int D, ta_dtype dt, int causal, int num_sms) {
  Problem p;
  if (entry < 0 || entry > 2 || B < 1 || H < 1) return 0;
  if (check_common(B, H, M, N, D, dt, -1.f, &p) != TA_OK) return 0;
  const int mode = entry == 0 ? kStd : entry == 1 ? kPiecewise : kJvp;
  return fwd_split_plan(mode, p, causal, num_sms > 0 ? num_sms : device_sms()) ? 2 : 1;
}

void ta_set_wait_timeout_ms(int ms) { g_timeout_ns = static_cast<uint64_t>(ms > 0 ? ms : 2000) * 1000000ull; }

ta_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int M, int N,
                   int D, ta_dtype dt, int causal, float sm_scale, void* stream) {
  Problem p;
  ta_status st = check_common(B, H, M, N, D, dt, sm_scale, &p);
  if (st != TA_OK) return st;
  if (p.BH * M == 0) return TA_OK;
  st = (N > 0) ? check_ptrs({q, k, v, o, lse}) : check_ptrs({o, lse});
  if (st != TA_OK) return st;
  return run_fwd(kStd, p, q, k, v, nullptr, nullptr, nullptr, o, lse, nullptr, nullptr, causal, 0,
                 static_cast<cudaStream_t>(stream));
}

ta_status attn_fwd_jvp(const void* q, const void* k, const void* v, const void* tq, const void* tk,
                       const void* tv, void* o, float* lse, void* to, float* tlse, int B, int H, int M, int N,
                       int D, ta_dtype dt, int causal, float sm_scale, void* stream) {
  Problem p;
  ta_status st = check_common(B, H, M, N, D, dt, sm_scale, &p);
  if (st != TA_OK) return st;
  if (p.BH * M == 0) return TA_OK;
  st = (N > 0) ? check_ptrs({q, k, v, tq, tk, tv, o, lse, to}) : check_ptrs({o, lse, to});
  if (st != TA_OK) return st;
  if (tlse && !aligned16(tlse)) return TA_ERR_ALIGNMENT;
  return run_fwd(kJvp, p, q, k, v, tq, tk, tv, o, lse, to, tlse, causal, 0, static_cast<cudaStream_t>(stream));
}

ta_status piecewise_fwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v, void* o,
                        float* lse, int B, int H, int M, int N, int D, ta_dtype dt, int causal, float sm_scale,
                        int w, void* stream) {
  Problem p;
  ta_status st = check_common(B, H, M, N, D, dt, sm_scale, &p);
  if (st != TA_OK) return st;
  if (p.BH * M == 0) return TA_OK;
  st = (N > 0) ? check_ptrs({q1, k1, q2, k2, v, o, lse}) : check_ptrs({o, lse});
  if (st != TA_OK) return st;
  return run_fwd(kPiecewise, p, q1, k1, v, q2, k2, nullptr, o, lse, nullptr, nullptr, causal, w,
                 static_cast<cudaStream_t>(stream));
}

static ta_status check_merge(int B, int H, int M, int D, ta_dtype dt, long long* rows) {
  if (B < 0 || H < 0 || M < 0) return TA_ERR_INVALID_ARG;
  if (dt != TA_F16 && dt != TA_BF16 && dt != TA_F32) return TA_ERR_UNSUPPORTED;
  if (D != 16 && D != 32 && D != 64 && D != 128) return TA_ERR_UNSUPPORTED;
  *rows = static_cast<long long>(B) * H * M;
  return TA_OK;
}

ta_status attn_merge_fwd(const void* o1, const float* lse1, const void* o2, const float* lse2, void* o,
                         float* lse, int B, int H, int M, int D, ta_dtype dt, void* stream) {
  long long rows = 0;
  ta_status st = check_merge(B, H, M, D, dt, &rows);
  if (st != TA_OK) return st;
  if (rows == 0) return TA_OK;
  st = check_ptrs({o1, lse1, o2, lse2, o, lse});
  if (st != TA_OK) return st;
  MergePtrs mp{};
  mp.o1 = o1, mp.o2 = o2, mp.l1 = lse1, mp.l2 = lse2, mp.o = o, mp.lse = lse;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prof_begin("attn_merge_fwd", s);
  cudaError_t e = launch_merge(false, static_cast<int>(dt), D, mp, rows, s);
  prof_end(s);
  return cuda_status(e);
}

ta_status attn_merge_bwd(const void* o1, const float* lse1, const void* o2, const float* lse2, const void* dO,
                         const float* dlse, void* do1, float* dlse1, void* do2, float* dlse2, int B, int H,
                         int M, int D, ta_dtype dt, void* stream) {
  long long rows = 0;
  ta_status st = check_merge(B, H, M, D, dt, &rows);
  if (st != TA_OK) return st;
  if (rows == 0) return TA_OK;
  st = check_ptrs({o1, lse1, o2, lse2, dO, do1, dlse1, do2, dlse2});
  if (st != TA_OK) return st;
  if (dlse && !aligned16(dlse)) return TA_ERR_ALIGNMENT;
  MergePtrs mp{};
  mp.o1 = o1, mp.o2 = o2, mp.l1 = lse1, mp.l2 = lse2, mp.dO = dO, mp.dl = dlse;
  mp.do1 = do1, mp.do2 = do2, mp.dl1 = dlse1, mp.dl2 = dlse2;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  prof_begin("attn_merge_bwd", s);
  cudaError_t e = launch_merge(true, static_cast<int>(dt), D, mp, rows, s);
  prof_end(s);
  return cuda_status(e);
}

ta_status attn_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int H, int M,
                       int N, int D, int causal, float sm_scale, void* stream) {
  Problem p;
  ta_status st = check_common(B, H, M, N, D, TA_BF16, sm_scale, &p);  // shapes and scale
  if (st != TA_OK) return st;
  if (D != 64 && D != 128) return TA_ERR_UNSUPPORTED;
  if (N % 16 != 0) return TA_ERR_UNSUPPORTED;  // the rows of V^T must start 16-byte aligned
  p.esize = 1;
  if (p.BH * M == 0) return TA_OK;
  st = (N > 0) ? check_ptrs({q, k, vt, o, lse}) : check_ptrs({o, lse});
  if (st != TA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (N == 0) {
    prof_begin("empty_rows", s);
    cudaError_t e = launch_empty_rows(1, D, o, lse, nullptr, p.BH * M, s);
    prof_end(s);
    return cuda_status(e);
  }
  FwdMaps maps;
  bool ok = make_map_u8(&maps.q, q, p.BH, M, D, 128, 128) && make_map_u8(&maps.k, k, p.BH, N, D, 128, 128) &&
            make_map_u8(&maps.v, vt, p.BH, D, N, 128, D);
  if (!ok) return TA_ERR_CUDA;
  FwdArgs a = fwd_args(p, causal, 0, o, lse, nullptr, nullptr);
  prof_begin("attn_fwd_fp8", s);
  cudaError_t e = launch_fwd_f8(D, maps, a, s);
  prof_end(s);
  return cuda_status(e);
}

size_t attn_bwd_workspace_bytes(int B, int H, int M, int N, int D, ta_dtype dt) {
  (void)N;
  (void)D;
  (void)dt;
  if (B <= 0 || H <= 0 || M <= 0) return 0;
  return delta_bytes(static_cast<long long>(B) * H, M);
}

size_t attn_bwd_fused_workspace_bytes(int B, int H, int M, int N, int D, ta_dtype dt) {
  (void)N;
  if (B <= 0 || H <= 0 || M <= 0) return 0;
  const long long BH = static_cast<long long>(B) * H;
  return delta_bytes(BH, M) + (bwd_fused_applies(D, dt) ? dq_acc_bytes(BH, M, D) : 0);
}

size_t piecewise_bwd_workspace_bytes(int B, int H, int M, int N, int D, ta_dtype dt) {
  (void)N;
  (void)D;
  (void)dt;
  if (B <= 0 || H <= 0 || M <= 0) return 0;
  return delta_bytes(static_cast<long long>(B) * H, M);
}

ta_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                   void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, int B, int H, int M, int N, int D,
                   ta_dtype dt, int causal, float sm_scale, void* stream) {
  return ta::bwd_entry(false, q, k, v, o, lse, dO, dq, dk, dv, ws, ws_bytes, B, H, M, N, D, dt, causal, sm_scale,
                       stream);
}

ta_status attn_bwd_fused(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, int B, int H,
                         int M, int N, int D, ta_dtype dt, int causal, float sm_scale, void* stream) {
  if (dt != TA_F16 && dt != TA_BF16) return TA_ERR_UNSUPPORTED;
  if (!bwd_fused_applies(D, dt)) return TA_ERR_UNSUPPORTED;
  return ta::bwd_entry(true, q, k, v, o, lse, dO, dq, dk, dv, ws, ws_bytes, B, H, M, N, D, dt, causal, sm_scale,
                       stream);
}

size_t attn_bwd_jvp_workspace_bytes(int B, int H, int M, int N, int D, ta_dtype dt) {
  return 2 * piecewise_bwd_workspace_bytes(B, H, M, N, D, dt);  // eps and delta2
}

ta_status attn_bwd_jvp(const void* q, const void* k, const void* v, const void* tq, const void* tk, const void* tv,
                       const void* o, const float* lse, const void* to, const float* tlse, const void* dO,
                       const void* dtO, void* dq, void* dk, void* dv, void* dtq, void* dtk, void* dtv, void* ws,
                       size_t ws_bytes, int B, int H, int M, int N, int D, ta_dtype dt, int causal,
                       float sm_scale, void* stream) {
  Problem p;
  ta_status st = check_common(B, H, M, N, D, dt, sm_scale, &p);
  if (st != TA_OK) return st;
  if (p.BH == 0 || (M == 0 && N == 0)) return TA_OK;
  if (M == 0) st = check_ptrs({dk, dv, dtk, dtv});
  else if (N == 0) st = check_ptrs({o, to, dO, dtO, dq, dtq, ws});
  else st = check_ptrs({q, k, v, tq, tk, tv, o, lse, to, tlse, dO, dtO, dq, dk, dv, dtq, dtk, dtv, ws});
  if (st != TA_OK) return st;
  return run_bwd_jvp(p, q, k, v, tq, tk, tv, o, lse, to, tlse, dO, dtO, dq, dk, dv, dtq, dtk, dtv, ws, ws_bytes,
                     causal, static_cast<cudaStream_t>(stream));
}

ta_status piecewise_bwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                        const void* o, const float* lse, const void* dO, void* dq1, void* dk1, void* dq2,
                        void* dk2, void* dv, void* ws, size_t ws_bytes, int B, int H, int M, int N, int D,
                        ta_dtype dt, int causal, float sm_scale, int w, void* stream) {
  Problem p;
  ta_status st = check_common(B, H, M, N, D, dt, sm_scale, &p);
  if (st != TA_OK) return st;
  if (p.BH == 0 || (M == 0 && N == 0)) return TA_OK;
  if (M == 0) st = check_ptrs({dk1, dk2, dv});
  else if (N == 0) st = check_ptrs({o, dO, dq1, dq2, ws});
  else st = check_ptrs({q1, k1, q2, k2, v, o, lse, dO, dq1, dk1, dq2, dk2, dv, ws});
  if (st != TA_OK) return st;
  return run_bwd(kPiecewise, p, q1, k1, v, q2, k2, o, lse, dO, dq1, dk1, dq2, dk2, dv, ws, ws_bytes, causal, w,
                 static_cast<cudaStream_t>(stream));
}

ta_status ta_sync_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return TA_ERR_CUDA;
  uint32_t* w = error_word_ptr();
  if (!w) return TA_ERR_CUDA;
  uint32_t h = 0;
  if (cudaMemcpy(&h, w, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return TA_ERR_CUDA;
  if (h) {
    const uint32_t zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return TA_ERR_CUDA;
    return TA_ERR_TIMEOUT;
  }
  return ta::guard_status();
}

ta_status ta_profile_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (on) {
    g_prof_recs.clear();
    g_prof_pool_next = 0;
    g_prof_pending = nullptr;
  }
  g_prof_on = on != 0;
  return TA_OK;
}

int ta_profile_read(const char** names, int* launches, double* total_ms, int cap) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  std::vector<std::string> keys;
  std::vector<int> cnt;
  std::vector<double> ms;
  for (const ProfRec& r : g_prof_recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) return -1;
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) return -1;
    size_t i = 0;
    while (i < keys.size() && keys[i] != r.name) ++i;
    if (i == keys.size()) {
      keys.push_back(r.name);
      cnt.push_back(0);
      ms.push_back(0.0);
    }
    cnt[i] += 1;
    ms[i] += t;
  }
  for (size_t i = 0; i < keys.size() && static_cast<int>(i) < cap; ++i) {
    // names point at the static strings passed to prof_begin
    for (const ProfRec& r : g_prof_recs)
      if (keys[i] == r.name) {
        names[i] = r.name;
        break;
      }
    launches[i] = cnt[i];
    total_ms[i] = ms[i];
  }
  return static_cast<int>(keys.size());
}

}  // extern "C"

// ------------------------------------------------------ wait self-test
namespace ta {
__global__ void wait_selftest_kernel(uint32_t* err, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  WaitCtl ctl{err, timeout_ns, &abort_flag};
  // Nothing ever arrives on `bar`: the bounded wait must give up.
  mbar_wait(&bar, 0, ctl, kErrTimeoutOther);
}
}  // namespace ta

extern "C" ta_status ta_selftest_wait_timeout(int timeout_ms, void* stream) {
  if (timeout_ms <= 0 || timeout_ms > 10000) return TA_ERR_INVALID_ARG;
  uint32_t* w = error_word_ptr();
  if (!w) return TA_ERR_CUDA;
  ta::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      w, static_cast<uint64_t>(timeout_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? TA_OK : TA_ERR_CUDA;
}
