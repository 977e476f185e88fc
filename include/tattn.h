/*
 * tattn.h -- C ABI of libtattn.so: fused scaled-dot-product attention on one
 * GB300 (sm_103a) GPU, hand-written tcgen05/TMA kernels.
 *
 * Sources of the operations (web pages, by title and section):
 *   [FA-JVP]  "Triton fused attention tutorial, updated with JVP support"
 *             (gist _06_fused_attention_blockptr_jvp.py): _attn_fwd,
 *             _attn_fwd_inner (online softmax, JVP extras), _attn_bwd_preprocess,
 *             _attn_bwd_dkdv, _attn_bwd_dq, JVPAttn.forward / JVPAttn.backward,
 *             and the comment thread's non-causal backward fix.
 *   [PW]      "FlagAttention src/flag_attn/piecewise.py": _fwd_kernel,
 *             _bwd_preprocess, _bwd_kv_kernel, _bwd_q_kernel, attention().
 *   [MERGE]   "backward_phase_2": a two-state online-softmax merge
 *             (reference_forward) and its backward.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are device pointers to contiguous [B, H, S, D] arrays (row-major,
 *    D fastest).  Queries, dO, O and tangents of queries have S = M rows; keys,
 *    values and their tangents have S = N rows.  All of q/k/v (and tangents,
 *    dO) share one element type `dt`; O, dQ, dK, dV and tO are written in `dt`.
 *  - `lse` is float32 [B, H, M]: the natural-log log-sum-exp of the scaled
 *    scores of each query row, L_i = ln sum_j exp(sm_scale * q_i . k_j) over
 *    the visible keys; rows that see no key get O = 0 and L = -inf.
 *  - causal != 0 keeps key j for query i iff j <= i + (N - M) (bottom-right
 *    alignment, [PW] _fwd_kernel; for M == N this is j <= i as in [FA-JVP]).
 *  - sm_scale <= 0 (or not finite) selects 1/sqrt(D), like the pages' None.
 *  - D must be 16, 32, 64 or 128 (the head sizes both pages' kernels accept
 *    up to 128; D = 16 and 32 run the D = 64 kernels with the columns past D
 *    read as zeros and never written).  dt TA_F16 / TA_BF16 run the tcgen05
 *    kernels (P
 *    and dS rounded to 16 bits as MMA operands, fp32 accumulation); TA_F32
 *    is the fp32 mode: float32 tensors computed in float32 with SIMT FMA
 *    and accurate expf/logf (a correctness path, not a throughput path).
 *  - Every pointer must be 16-byte aligned (TMA).  B, H >= 1 and M, N >= 0;
 *    B*H*M == 0 is a no-op returning TA_OK.
 *  - The caller owns every buffer.  Nothing is allocated on the call path;
 *    backward scratch lives in the caller's workspace `ws`.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Argument errors are reported synchronously before any
 *    launch; a bounded-wait timeout inside a kernel is recorded in a device
 *    error word that ta_sync_status() reads.
 *  - Host threads may call the entry points concurrently (the library's
 *    per-device set-up is idempotent and its caches are atomic).  A thread
 *    needs no CUDA set-up of its own: with no current context, a call binds
 *    the current device's primary context first.  The device error word is
 *    shared by every call on a device, and ta_profile_* expect one host
 *    thread issuing the calls they time.
 */
#ifndef TATTN_H_
#define TATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TA_OK = 0,
  TA_ERR_INVALID_ARG = 1, /* null pointer, negative size, B*H overflow, ... */
  TA_ERR_UNSUPPORTED = 2, /* D or dtype outside the supported set */
  TA_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned */
  TA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
  TA_ERR_TIMEOUT = 5,     /* a kernel's bounded wait ran out (ta_sync_status) */
  TA_ERR_GUARD = 6        /* guard build only: a device-side check failed (ta_sync_status) */
} ta_status;

typedef enum { TA_F16 = 0, TA_BF16 = 1, TA_F32 = 2 } ta_dtype;

/* Forward: O = softmax(sm_scale * Q K^T) V with per-row LSE.
 * [FA-JVP] _attn_fwd (+ _attn_fwd_inner stages), [PW] _fwd_kernel.
 * In: q [B,H,M,D], k,v [B,H,N,D].  Out: o [B,H,M,D] (dt), lse [B,H,M] fp32. */
ta_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int M,
                   int N, int D, ta_dtype dt, int causal, float sm_scale, void* stream);

/* Bytes of workspace attn_bwd needs: delta [B,H,M] fp32 (16-byte padded). */
size_t attn_bwd_workspace_bytes(int B, int H, int M, int N, int D, ta_dtype dt);

/* Backward of attn_fwd for the loss <dO, O>.
 * [FA-JVP] _attn_bwd_preprocess (delta = rowsum(dO o O)), _attn_bwd_dkdv,
 * _attn_bwd_dq and JVPAttn.backward, with the thread's non-causal fix;
 * [PW] _bwd_preprocess / _bwd_kv_kernel / _bwd_q_kernel.
 * In: q,k,v, o and lse from attn_fwd, dO [B,H,M,D].  Out: dq [B,H,M,D],
 * dk, dv [B,H,N,D] (dt).  ws: >= attn_bwd_workspace_bytes(...) bytes of
 * device memory, 16-byte aligned, contents need not be initialised.
 * In 16-bit types the dQ pass forms delta itself (from O and dO, while
 * its first score products run) and stores it in ws for the dK/dV pass that
 * follows; in fp32 a delta pass runs first.
 * Returns TA_ERR_INVALID_ARG if ws is null or too small. */
ta_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, int B, int H,
                   int M, int N, int D, ta_dtype dt, int causal, float sm_scale, void* stream);

/* Bytes of workspace attn_bwd_fused needs: delta [B,H,M] fp32 (padded to 256
 * bytes) followed by the fp32 dQ accumulator [B,H,M,D] (D = 128 in 16-bit;
 * delta alone otherwise, where attn_bwd_fused returns TA_ERR_UNSUPPORTED). */
size_t attn_bwd_fused_workspace_bytes(int B, int H, int M, int N, int D, ta_dtype dt);

/* attn_bwd in one key-stationary pass: five matmuls per (key, query) block
 * pair (S^T, dP^T, dV, dK and dQ^T = K^T dS^T) instead of the seven of the
 * separate dK/dV and dQ passes.  [FA-JVP] _attn_bwd computes dK/dV of its key
 * block and dQ of its query block in one program, each recomputing S and dP;
 * here the key block's CTA adds its dQ contribution into an fp32 accumulator
 * in `ws` with atomics, and a final pass writes dq = sm_scale * acc in dt.
 * Same arguments and outputs as attn_bwd.
 *  - dt TA_F16 / TA_BF16 and D = 128 only; anything else returns
 *    TA_ERR_UNSUPPORTED before any launch.
 *  - ws: >= attn_bwd_fused_workspace_bytes(...) bytes, 16-byte aligned,
 *    contents need not be initialised (the delta pass zeroes the accumulator).
 *  - dq's fp32 summation order depends on the order the atomics land in, so
 *    dq may differ between calls in its last bit; dk, dv and lse-related
 *    outputs are deterministic.
 *  - attn_bwd (the two passes) is the faster path on GB300 at the benchmark
 *    shapes; this entry point is the five-matmul alternative. */
ta_status attn_bwd_fused(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dO, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes, int B, int H,
                         int M, int N, int D, ta_dtype dt, int causal, float sm_scale, void* stream);

/* attn_bwd for callers that cannot allocate device memory or pass a
 * workspace (for example a host framework that has reserved all device memory
 * for its own pool, or a step loop that must not call cudaMalloc because it
 * synchronises the device).  The pages have no counterpart: this is a
 * packaging variant of attn_bwd, with the same arguments minus `ws`.
 *  - Scratch (delta, one float per query row) lives in a fixed array inside
 *    the library's device image: at most 2^21 rows, i.e. B*H*M <= 2097152
 *    (8 MiB, held on every GPU that loads the library until the process
 *    exits).  Larger problems return TA_ERR_UNSUPPORTED without launching.
 *  - The call allocates nothing.  Its first call on a device looks up the
 *    array's device address (cudaGetSymbolAddress) with that device current;
 *    make that first call before any stream capture.  The address is cached
 *    together with the context it was looked up in; after cudaDeviceReset
 *    (or from another context) the next call looks it up again, so that call,
 *    too, belongs before any capture.
 *  - B*H > 2^31 - 1 returns TA_ERR_INVALID_ARG, as in attn_bwd.
 *  - It runs the two-pass backward of attn_bwd (its only scratch is delta).
 *  - Every call shares the one array and fully rewrites the rows it uses, so
 *    nothing needs clearing between calls; calls that may run at the same
 *    time on the GPU (other streams, other host threads) race on it. */
ta_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                           const void* dO, void* dq, void* dk, void* dv, int B, int H, int M, int N, int D,
                           ta_dtype dt, int causal, float sm_scale, void* stream);

/* Forward with fused forward-mode JVP: also returns
 * tO = d/de attention(q + e tq, k + e tk, v + e tv) at e = 0.
 * [FA-JVP] _attn_fwd_inner ENABLE_JVP branch and the _attn_fwd JVP epilogue:
 * with T = sm_scale (tq K^T + Q tk^T) (zero where masked), mu_i = sum_j P_ij T_ij,
 * tO = (P o T) V - mu o O + P tV.
 * tlse, when not NULL, receives the tangent of L: tL_i = mu_i (the mu the
 * epilogue divides by l), 0 for rows that see no key.
 * In: q,tq [B,H,M,D], k,v,tk,tv [B,H,N,D].  Out: o, to [B,H,M,D] (dt), lse,
 * tlse [B,H,M] fp32. */
ta_status attn_fwd_jvp(const void* q, const void* k, const void* v, const void* tq, const void* tk,
                       const void* tv, void* o, float* lse, void* to, float* tlse, int B, int H, int M, int N,
                       int D, ta_dtype dt, int causal, float sm_scale, void* stream);

/* Bytes of workspace attn_bwd_jvp needs: eps and delta2 [B,H,M] fp32 (each
 * padded to 256 bytes). */
size_t attn_bwd_jvp_workspace_bytes(int B, int H, int M, int N, int D, ta_dtype dt);

/* Backward of attn_fwd_jvp: the gradients of <dO, O> + <dtO, tO> with respect
 * to q, k, v and the tangents tq, tk, tv.  [FA-JVP] gives the JVP forward
 * (above) and a backward for O only; this is the chain rule taken back
 * through that forward's steps.  With P, T and mu as in attn_fwd_jvp,
 * eps_i = <dtO_i, O_i>, delta2_i = <dO_i, O_i> + <dtO_i, tO_i>:
 *   dT = P o (dtO V^T - eps),  dS = P o (dO V^T + dtO tV^T - delta2) + (T - mu) o dT,
 *   dq = sm_scale (dS K + dT tK),  dk = sm_scale (dS^T Q + dT^T tQ),
 *   dv = P^T dO + (P o (T - mu))^T dtO,
 * and (dtq, dtk, dtv) = the plain backward (attn_bwd) of dO := dtO, since tO
 * is the Jacobian of O applied to the tangents.
 * In: q,tq [B,H,M,D], k,v,tk,tv [B,H,N,D]; o, lse, to and tlse from
 * attn_fwd_jvp (tlse is required here); dO, dtO [B,H,M,D].
 * Out: dq, dtq [B,H,M,D], dk, dv, dtk, dtv [B,H,N,D] (dt).
 * ws: >= attn_bwd_jvp_workspace_bytes(...) bytes of device memory, 16-byte
 * aligned, contents need not be initialised; TA_ERR_INVALID_ARG if it is
 * null or too small. */
ta_status attn_bwd_jvp(const void* q, const void* k, const void* v, const void* tq, const void* tk, const void* tv,
                       const void* o, const float* lse, const void* to, const float* tlse, const void* dO,
                       const void* dtO, void* dq, void* dk, void* dv, void* dtq, void* dtk, void* dtv, void* ws,
                       size_t ws_bytes, int B, int H, int M, int N, int D, ta_dtype dt, int causal,
                       float sm_scale, void* stream);

/* Piecewise attention forward ([PW] attention(), _fwd_kernel): the score of
 * (i, j) is sm_scale * q2_i . k2_j when the signed distance i + N - M - j >= w,
 * else sm_scale * q1_i . k1_j (the page's code rule piecewise_mask).
 * In: q1,q2 [B,H,M,D], k1,k2,v [B,H,N,D].  Out: o (dt), lse (fp32). */
ta_status piecewise_fwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                        void* o, float* lse, int B, int H, int M, int N, int D, ta_dtype dt, int causal,
                        float sm_scale, int w, void* stream);

/* Bytes of workspace piecewise_bwd needs (same layout as attn_bwd's). */
size_t piecewise_bwd_workspace_bytes(int B, int H, int M, int N, int D, ta_dtype dt);

/* Piecewise backward ([PW] _bwd_preprocess, _bwd_kv_kernel, _bwd_q_kernel):
 * dS = P o (dP - delta) is routed to (dq1, dk1) where distance < w and to
 * (dq2, dk2) where distance >= w; dv = P^T dO.
 * Out: dq1, dq2 [B,H,M,D], dk1, dk2, dv [B,H,N,D] (dt).
 * At D = 128 in 16-bit the key-stationary pass streams the queries in
 * 64-row steps, so that tensor memory holds all three accumulators of a
 * 128-key tile beside its score buffers and one pass forms dv, dk1, dk2.
 * In 16-bit types the dQ pass runs first and forms delta, as in attn_bwd. */
ta_status piecewise_bwd(const void* q1, const void* k1, const void* q2, const void* k2, const void* v,
                        const void* o, const float* lse, const void* dO, void* dq1, void* dk1, void* dq2,
                        void* dk2, void* dv, void* ws, size_t ws_bytes, int B, int H, int M, int N, int D,
                        ta_dtype dt, int causal, float sm_scale, int w, void* stream);


/* FP8 forward ([FA-JVP] _attn_fwd with FP8_OUTPUT and the tutorial's fp8
 * benchmark path): q [B,H,M,D] and k [B,H,N,D] in float8 e5m2, V passed
 * TRANSPOSED as vt [B,H,D,N] e5m2 (the layout the tutorial builds for fp8),
 * P rounded to e5m2 for the P V product, fp32 accumulation; out: o [B,H,M,D]
 * in e5m2 and lse [B,H,M] fp32 (natural log, as attn_fwd).  Same masking,
 * empty-row and sm_scale rules as attn_fwd.  D in {64, 128}; N a multiple of
 * 16 (rows of vt start 16-byte aligned), else TA_ERR_UNSUPPORTED. */
ta_status attn_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse, int B, int H, int M,
                       int N, int D, int causal, float sm_scale, void* stream);

/* Merge of two partial attention states of the same queries over disjoint
 * key sets (split-KV / context-parallel combine), [MERGE] reference_forward:
 * with m = max(L1, L2), a = exp(L1 - m), b = exp(L2 - m):
 * O = (a O1 + b O2) / (a + b), L = m + ln(a + b).  A row whose parts both
 * saw no key (L1 = L2 = -inf) gives O = 0, L = -inf.
 * In: o1, o2 [B,H,M,D] (dt), lse1, lse2 [B,H,M] fp32.  Out: o (dt), lse.
 * Outputs may alias o1 / lse1 (each element is read before it is written).
 * D in {16, 32, 64, 128}; every pointer 16-byte aligned; errors as attn_fwd. */
ta_status attn_merge_fwd(const void* o1, const float* lse1, const void* o2, const float* lse2, void* o,
                         float* lse, int B, int H, int M, int D, ta_dtype dt, void* stream);

/* Backward of attn_merge_fwd ([MERGE] merge backward kernel), with
 * alpha = a / (a + b), beta = b / (a + b), t = sum_d dO (O1 - O2):
 * dO1 = alpha dO, dO2 = beta dO, dL1 = alpha dL + alpha beta t,
 * dL2 = beta dL - alpha beta t.  dlse (the gradient of the merged L) may be
 * NULL, meaning zero.  Rows with L1 = L2 = -inf get zero gradients.
 * In: o1, o2, dO [B,H,M,D] (dt), lse1, lse2, dlse [B,H,M] fp32.
 * Out: do1, do2 (dt), dlse1, dlse2 (fp32). */
ta_status attn_merge_bwd(const void* o1, const float* lse1, const void* o2, const float* lse2, const void* dO,
                         const float* dlse, void* do1, float* dlse1, void* do2, float* dlse2, int B, int H,
                         int M, int D, ta_dtype dt, void* stream);
/* Synchronises `stream`, then reads and clears the device error word that
 * the kernels set when a bounded wait runs out.  TA_OK, TA_ERR_TIMEOUT or
 * TA_ERR_CUDA (an asynchronous CUDA error); in the guard build also
 * TA_ERR_GUARD when a device-side check failed since the last call. */
ta_status ta_sync_status(void* stream);

/* Human-readable name of a status code (static string). */
const char* ta_status_str(ta_status s);

/* Self-test of the bounded-wait machinery: launches one block that waits on
 * an mbarrier nothing ever arrives on, with a limit of `timeout_ms`.  The
 * kernel gives up, records a timeout and exits; ta_sync_status() then returns
 * TA_ERR_TIMEOUT and the context stays usable.  No counterpart on the pages. */
ta_status ta_selftest_wait_timeout(int timeout_ms, void* stream);

/* Per-kernel timing with CUDA events recorded on the launch stream around
 * every kernel the library launches (no counterpart on the pages).
 * ta_profile_enable(1) clears the counters and starts recording;
 * ta_profile_read() synchronises and fills, for up to `cap` kernels, the
 * name, launch count and total milliseconds; it returns the number of
 * kernels seen.  ta_profile_enable(0) stops recording. */
ta_status ta_profile_enable(int on);
int ta_profile_read(const char** names, int* launches, double* total_ms, int cap);

/* Key split of the one-query-tile forward (no counterpart on the pages; the
 * merge is [MERGE] reference_forward's combine, done on the raw online-softmax
 * state).  attn_fwd_jvp (all D) and piecewise_fwd at D = 128 (16-bit) run one
 * 128-row query tile per CTA.  When that grid is under one wave of the GPU's
 * SMs and a two-CTA split of every query tile's key tiles shortens the
 * estimated schedule (list scheduling in launch order, costs in key tiles),
 * each query tile gets a cluster of two CTAs: the second hands its running
 * max, sum and unnormalised accumulators to the first over distributed shared
 * memory, and the first combines them with the same rescale the online
 * softmax applies between key tiles.  Results equal the unsplit kernel's up
 * to fp32 rounding; nothing is allocated.
 * ta_fwd_kv_split returns 2 when `entry` (0 attn_fwd, 1 piecewise_fwd,
 * 2 attn_fwd_jvp) splits this problem on a GPU of `num_sms` SMs (<= 0: the
 * current device's count), 1 when it does not, 0 for invalid arguments.
 * ta_set_fwd_kv_split(mode) sets the choice for the process: 0 (default) by
 * the estimate, 1 never, 2 wherever the kernel supports it. */
int ta_fwd_kv_split(int entry, int B, int H, int M, int N, int D, ta_dtype dt, int causal, int num_sms);
void ta_set_fwd_kv_split(int mode);

/* Guard build (no counterpart on the pages; it stands in for a memory-error
 * checker).  The same sources compiled with TA_GUARD into libtattn_guard.so
 * check, on the device, the operands of every TMA load (destination inside
 * the block's dynamic shared memory on a 1024-byte boundary, innermost
 * coordinate a multiple of 16 elements, no negative coordinate), every TMEM
 * load and store (lane field = the calling warp's quadrant, columns inside
 * the 512 allocated), every MMA batch (accumulator and TMEM operand inside
 * the allocation, shared-memory descriptors inside the dynamic shared
 * memory), the 16-byte alignment of the row stores and every CTA's work
 * decode.  A failed check skips its access and makes ta_sync_status return
 * TA_ERR_GUARD.  ta_guard_build() is 1 in that library and 0 in libtattn.so;
 * ta_guard_last() describes the first failing check ("unit.cu:line", the
 * value it rejected and the block's dynamic shared memory base and size) that the
 * last TA_ERR_GUARD reported; ta_selftest_guard() launches one thread that
 * fails a check on purpose without touching memory (TA_ERR_GUARD at the next
 * ta_sync_status in the guard build, TA_OK in the product build). */
int ta_guard_build(void);
const char* ta_guard_last(void);
ta_status ta_selftest_guard(void* stream);

/* Per-launch wait limit in milliseconds used by every kernel (default 2000,
 * or the TA_WAIT_TIMEOUT_MS environment variable at load time). */
void ta_set_wait_timeout_ms(int ms);

#ifdef __cplusplus
}
#endif

#endif /* TATTN_H_ */
