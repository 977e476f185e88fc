"""fp64 CPU oracle for fused scaled-dot-product attention -- TEST INFRASTRUCTURE.

This package is the plain, slow, obviously-correct definition that the CUDA
path is checked against.  It is test infrastructure: only the test-suite,
the smoke check and the benchmark's CPU-baseline leg may import it; the
product path never calls it and has no CPU fallback.

It shares no code with the CUDA path.  Inputs are the exact dtype-rounded
values the GPU sees, upcast to float64; everything here runs in float64 with
numpy (a matrix product is used as a library step, nothing is blocked, fused
or reordered beyond the definitions below).  Every function works on one
(batch, head) slice; the ``*_bhsd`` wrappers loop over heads.

Definitions, and the page passages they follow:

* Scores and mask.  ``S_ij = sm_scale * q_i . k_j``.  With ``P_SEQ = N - M``,
  causal attention keeps key j for query i iff ``j <= i + P_SEQ`` (bottom-right
  alignment) -- "FlagAttention piecewise.py", ``_fwd_kernel`` causal mask; for
  M == N this is the ``offs_m >= start_n + offs_n`` mask of the diagonal stage
  of ``_attn_fwd_inner`` in "Triton fused attention tutorial, updated with JVP
  support".
* Softmax and log-sum-exp.  ``L_i = m_i + ln sum_j exp(S_ij - m_i)`` over the
  kept keys, ``P_ij = exp(S_ij - L_i)``, ``O = P V``.  L is the natural-log
  LSE of the scaled scores (the piecewise ``_fwd_kernel`` epilogue stores
  ``m * sm_scale + log(l)``; the tutorial's ``_attn_fwd`` stores the same
  quantity in base 2, ``m_i + log2(l_i)`` of log2(e)-scaled scores).  Rows with
  no kept key give O = 0 and L = -inf (piecewise ``_fwd_kernel``, empty lines).
* Backward (tutorial ``_attn_bwd_preprocess`` / ``_attn_bwd_dkdv`` /
  ``_attn_bwd_dq``; piecewise ``_bwd_preprocess`` / ``_bwd_kv_kernel`` /
  ``_bwd_q_kernel``): ``delta_i = sum_d dO_id O_id``, ``dV = P^T dO``,
  ``dP = dO V^T``, ``dS = P o (dP - delta)``, ``dQ = sm_scale dS K``,
  ``dK = sm_scale dS^T Q``.
* Forward-mode JVP (tutorial ``_attn_fwd_inner`` with ``ENABLE_JVP`` and the
  ``_attn_fwd`` JVP epilogue): ``T_ij = sm_scale (tq_i . k_j + q_i . tk_j)``,
  ``mu_i = sum_j P_ij T_ij``, ``tO = (P o T) V - mu o O + P tV``.  This is the
  derivative of O along (tq, tk, tv): ``dP = P o (T - mu)``; mu itself is the
  derivative of L (``attention_jvp_tl``).
* Backward of the JVP (``attention_jvp_bwd``): the gradients of
  ``<dO, O> + <dtO, tO>`` with respect to q, k, v and the tangents, taken by
  reverse-mode differentiation through the JVP forward's steps above in
  reverse order.  The pages give the JVP forward and a backward for O only;
  this is the plain chain rule applied to their definitions.
* Piecewise attention ("FlagAttention piecewise.py", ``_fwd_kernel``
  ``piecewise_mask``): with the signed distance ``d_ij = i + N - M - j``, the
  score uses (q2, k2) when ``d_ij >= w`` and (q1, k1) otherwise.  Backward
  (``_bwd_kv_kernel`` / ``_bwd_q_kernel``): dS is routed to (dq1, dk1) where
  ``d_ij < w`` and to (dq2, dk2) where ``d_ij >= w``; dv = P^T dO.

* Merge of two partial attention states (the "backward_phase_2" page:
  ``reference_forward`` and the merge backward kernel): for two normalised
  outputs O1, O2 of the same queries over disjoint key sets, with their
  log-sum-exps L1, L2: ``m = max(L1, L2)``, ``a = exp(L1 - m)``,
  ``b = exp(L2 - m)``, ``alpha = a / (a + b)``, ``beta = b / (a + b)``,
  ``O = alpha O1 + beta O2``, ``L = m + ln(a + b)``.  Backward, with the
  incoming dO and an optional dL (zero when absent): ``dO1 = alpha dO``,
  ``dO2 = beta dO``, ``t = sum_d dO (O1 - O2)``, ``dL1 = alpha dL + alpha beta t``,
  ``dL2 = beta dL - alpha beta t``.  A row whose two parts both saw no key
  (L1 = L2 = -inf) merges to O = 0, L = -inf with zero gradients.

Every function here is pinned by the ``-m "not gpu"`` oracle tests (finite
differences, closed forms, invariants, special cases); none is unpinned.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "allowed_mask", "attention_fwd", "attention_bwd", "attention_jvp",
    "piecewise_fwd", "piecewise_bwd", "attention_fwd_bhsd", "attention_bwd_bhsd",
    "attention_jvp_bhsd", "piecewise_fwd_bhsd", "piecewise_bwd_bhsd", "default_scale",
    "lse_merge_fwd", "lse_merge_bwd", "lse_merge_fwd_bhsd", "lse_merge_bwd_bhsd",
    "attention_jvp_tl", "attention_jvp_tl_bhsd", "attention_jvp_bwd", "attention_jvp_bwd_bhsd",
    "bwd_delta", "bwd_delta_bhsd",
]


def default_scale(D: int, sm_scale=None) -> float:
    """sm_scale None (or <= 0) means 1/sqrt(D), as both pages' wrappers do."""
    if sm_scale is None or sm_scale <= 0:
        return 1.0 / np.sqrt(D)
    return float(sm_scale)


def allowed_mask(M: int, N: int, causal: bool) -> np.ndarray:
    """Boolean [M, N]: key j visible to query i (bottom-right causal alignment)."""
    if not causal:
        return np.ones((M, N), dtype=bool)
    i = np.arange(M)[:, None]
    j = np.arange(N)[None, :]
    return j <= i + (N - M)


def _softmax(S: np.ndarray, keep: np.ndarray):
    """One-shot row softmax of S over the kept entries.  Returns (P, L)."""
    Sm = np.where(keep, S, -np.inf)
    m = Sm.max(axis=1) if S.shape[1] > 0 else np.full(S.shape[0], -np.inf)
    has = np.isfinite(m)
    mref = np.where(has, m, 0.0)
    E = np.where(keep, np.exp(Sm - mref[:, None]), 0.0)
    l = E.sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        L = np.where(has, mref + np.log(np.where(has, l, 1.0)), -np.inf)
        P = np.where(has[:, None], E / np.where(has, l, 1.0)[:, None], 0.0)
    return P, L


def _f64(*xs):
    """float64 copies of numpy arrays or (any-dtype, any-device) torch tensors."""
    out = []
    for x in xs:
        if hasattr(x, "detach"):
            x = x.detach().cpu().double().numpy()
        out.append(np.asarray(x, dtype=np.float64))
    return out


# ----------------------------------------------------------------- standard
def attention_fwd(q, k, v, causal: bool, sm_scale=None):
    """One head: q [M,D], k,v [N,D] -> (O [M,D], L [M]) in float64."""
    q, k, v = _f64(q, k, v)
    s = default_scale(q.shape[1], sm_scale)
    keep = allowed_mask(q.shape[0], k.shape[0], causal)
    P, L = _softmax(s * (q @ k.T), keep)
    return P @ v, L


def attention_bwd(q, k, v, do, causal: bool, sm_scale=None):
    """One head: gradients (dq, dk, dv) of <dO, O(q,k,v)>."""
    q, k, v, do = _f64(q, k, v, do)
    s = default_scale(q.shape[1], sm_scale)
    keep = allowed_mask(q.shape[0], k.shape[0], causal)
    P, _ = _softmax(s * (q @ k.T), keep)
    O = P @ v
    delta = (do * O).sum(axis=1)
    dv = P.T @ do
    dP = do @ v.T
    dS = P * (dP - delta[:, None])
    dq = s * (dS @ k)
    dk = s * (dS.T @ q)
    return dq, dk, dv


def bwd_delta(o, do):
    """One head: the backward preprocess delta_i = sum_d dO_id O_id from a
    given (stored) O [M,D] and dO [M,D] -- tutorial ``_attn_bwd_preprocess``,
    piecewise ``_bwd_preprocess``."""
    o, do = _f64(o, do)
    return (do * o).sum(axis=1)


def attention_jvp(q, k, v, tq, tk, tv, causal: bool, sm_scale=None):
    """One head: (O, L, tO) with tO the derivative of O along (tq, tk, tv)."""
    q, k, v, tq, tk, tv = _f64(q, k, v, tq, tk, tv)
    s = default_scale(q.shape[1], sm_scale)
    keep = allowed_mask(q.shape[0], k.shape[0], causal)
    P, L = _softmax(s * (q @ k.T), keep)
    O = P @ v
    T = np.where(keep, s * (tq @ k.T + q @ tk.T), 0.0)
    PT = P * T
    mu = PT.sum(axis=1)
    tO = PT @ v - mu[:, None] * O + P @ tv
    return O, L, tO


def attention_jvp_tl(q, k, tq, tk, causal: bool, sm_scale=None):
    """One head: tL, the derivative of L along (tq, tk).  L is the log-sum-exp
    of the scaled scores, so tL_i = sum_j P_ij T_ij = mu_i, the quantity the
    JVP epilogue divides by l (mu / l in the "Triton fused attention tutorial,
    updated with JVP support" _attn_fwd JVP epilogue); 0 for rows that see no
    key (L is the constant -inf there)."""
    q, k, tq, tk = _f64(q, k, tq, tk)
    s = default_scale(q.shape[1], sm_scale)
    keep = allowed_mask(q.shape[0], k.shape[0], causal)
    P, _ = _softmax(s * (q @ k.T), keep)
    T = np.where(keep, s * (tq @ k.T + q @ tk.T), 0.0)
    return (P * T).sum(axis=1)


def attention_jvp_bwd(q, k, v, tq, tk, tv, do, dto, causal: bool, sm_scale=None):
    """One head: gradients (dq, dk, dv, dtq, dtk, dtv) of <dO, O> + <dtO, tO>,
    with O and tO the outputs of ``attention_jvp``.

    The pages stop at the JVP's forward; this is reverse-mode differentiation
    of that forward's own steps, taken backwards one at a time:
      S = s q k^T, P = softmax(S), O = P v,
      T = s (tq k^T + q tk^T) (0 where masked), mu = rowsum(P o T),
      tO = (P o T) v - mu o O + P tv.
    """
    q, k, v, tq, tk, tv, do, dto = _f64(q, k, v, tq, tk, tv, do, dto)
    s = default_scale(q.shape[1], sm_scale)
    keep = allowed_mask(q.shape[0], k.shape[0], causal)
    P, _ = _softmax(s * (q @ k.T), keep)
    O = P @ v
    T = np.where(keep, s * (tq @ k.T + q @ tk.T), 0.0)
    PT = P * T
    mu = PT.sum(axis=1)
    # tO = PT v - mu O + P tv
    dPT = dto @ v.T
    dv = PT.T @ dto
    dmu = -(dto * O).sum(axis=1)
    dO_total = do - mu[:, None] * dto
    dP = dto @ tv.T
    dtv = P.T @ dto
    # mu = rowsum(PT)
    dPT = dPT + dmu[:, None]
    # PT = P o T
    dP = dP + dPT * T
    dT = np.where(keep, dPT * P, 0.0)
    # O = P v
    dP = dP + dO_total @ v.T
    dv = dv + P.T @ dO_total
    # P = softmax(S) over the kept keys (dS = P o (dP - rowsum(P o dP)))
    dS = P * (dP - (P * dP).sum(axis=1)[:, None])
    # S = s q k^T and T = s (tq k^T + q tk^T)
    dq = s * (dS @ k) + s * (dT @ tk)
    dk = s * (dS.T @ q) + s * (dT.T @ tq)
    dtq = s * (dT @ k)
    dtk = s * (dT.T @ q)
    return dq, dk, dv, dtq, dtk, dtv


# ---------------------------------------------------------------- piecewise
def far_mask(M: int, N: int, w: int) -> np.ndarray:
    """Boolean [M, N]: True where the signed distance i + N - M - j >= w."""
    i = np.arange(M)[:, None]
    j = np.arange(N)[None, :]
    return (i + (N - M) - j) >= w


def _piecewise_probs(q1, k1, q2, k2, causal, s, w):
    M, N = q1.shape[0], k1.shape[0]
    keep = allowed_mask(M, N, causal)
    far = far_mask(M, N, w)
    S = s * np.where(far, q2 @ k2.T, q1 @ k1.T)
    P, L = _softmax(S, keep)
    return P, L, far


def piecewise_fwd(q1, k1, q2, k2, v, causal: bool, sm_scale=None, w: int = 0):
    """One head of piecewise attention -> (O, L)."""
    q1, k1, q2, k2, v = _f64(q1, k1, q2, k2, v)
    s = default_scale(q1.shape[1], sm_scale)
    P, L, _ = _piecewise_probs(q1, k1, q2, k2, causal, s, w)
    return P @ v, L


def piecewise_bwd(q1, k1, q2, k2, v, do, causal: bool, sm_scale=None, w: int = 0):
    """One head of the piecewise backward -> (dq1, dk1, dq2, dk2, dv)."""
    q1, k1, q2, k2, v, do = _f64(q1, k1, q2, k2, v, do)
    s = default_scale(q1.shape[1], sm_scale)
    P, _, far = _piecewise_probs(q1, k1, q2, k2, causal, s, w)
    O = P @ v
    delta = (do * O).sum(axis=1)
    dv = P.T @ do
    dS = P * (do @ v.T - delta[:, None])
    dS1 = np.where(far, 0.0, dS)
    dS2 = np.where(far, dS, 0.0)
    return (s * (dS1 @ k1), s * (dS1.T @ q1), s * (dS2 @ k2), s * (dS2.T @ q2), dv)


# ---------------------------------------------------------------- LSE merge
def _merge_weights(l1, l2):
    """alpha, beta, m and the mask of rows where both parts are empty."""
    m = np.maximum(l1, l2)
    empty = np.isneginf(m)
    ms = np.where(empty, 0.0, m)
    a = np.exp(l1 - ms)  # exp(-inf) = 0 for an empty part
    b = np.exp(l2 - ms)
    z = np.where(empty, 1.0, a + b)
    alpha = np.where(empty, 0.0, a / z)
    beta = np.where(empty, 0.0, b / z)
    return alpha, beta, ms, z, empty


def lse_merge_fwd(o1, l1, o2, l2):
    """One head: O1, O2 [M, D], L1, L2 [M] -> merged (O, L)."""
    o1, o2, l1, l2 = _f64(o1, o2, l1, l2)
    alpha, beta, ms, z, empty = _merge_weights(l1, l2)
    O = alpha[:, None] * o1 + beta[:, None] * o2
    L = np.where(empty, -np.inf, ms + np.log(z))
    return O, L


def lse_merge_bwd(o1, l1, o2, l2, do, dl=None):
    """One head: gradients (dO1, dL1, dO2, dL2) of the merge given dO [M, D]
    and dL [M] (None = 0)."""
    o1, o2, l1, l2, do = _f64(o1, o2, l1, l2, do)
    dl = np.zeros_like(l1) if dl is None else _f64(dl)[0]
    alpha, beta, _, _, _ = _merge_weights(l1, l2)
    t = (do * (o1 - o2)).sum(axis=1)
    do1 = alpha[:, None] * do
    do2 = beta[:, None] * do
    dl1 = alpha * dl + alpha * beta * t
    dl2 = beta * dl - alpha * beta * t
    return do1, dl1, do2, dl2


# ------------------------------------------------------- [B,H,S,D] wrappers
def _heads(B, H, heads):
    if heads is None:
        return [(b, h) for b in range(B) for h in range(H)]
    return list(heads)


def _np(x):
    if hasattr(x, "detach"):
        x = x.detach().cpu()
        return x.to(dtype=__import__("torch").float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _run_bhsd(fn, tensors, extra, heads, nout):
    arrs = [_np(t) for t in tensors]
    B, H = arrs[0].shape[:2]
    hs = _heads(B, H, heads)
    outs = None
    for (b, h) in hs:
        res = fn(*[a[b, h] for a in arrs], *extra)
        if outs is None:
            outs = [np.zeros((B, H) + r.shape, dtype=np.float64) for r in res]
        for o, r in zip(outs, res):
            o[b, h] = r
    return tuple(outs)


def attention_fwd_bhsd(q, k, v, causal, sm_scale=None, heads=None):
    """[B,H,M,D] inputs -> (O, L); only the listed (b, h) heads are filled."""
    return _run_bhsd(attention_fwd, (q, k, v), (causal, sm_scale), heads, 2)


def attention_bwd_bhsd(q, k, v, do, causal, sm_scale=None, heads=None):
    return _run_bhsd(attention_bwd, (q, k, v, do), (causal, sm_scale), heads, 3)


def bwd_delta_bhsd(o, do, heads=None):
    """[B,H,M,D] O and dO -> delta [B,H,M]."""
    return _run_bhsd(lambda a, b: (bwd_delta(a, b),), (o, do), (), heads, 1)[0]


def attention_jvp_bhsd(q, k, v, tq, tk, tv, causal, sm_scale=None, heads=None):
    return _run_bhsd(attention_jvp, (q, k, v, tq, tk, tv), (causal, sm_scale), heads, 3)


def piecewise_fwd_bhsd(q1, k1, q2, k2, v, causal, sm_scale=None, w=0, heads=None):
    return _run_bhsd(piecewise_fwd, (q1, k1, q2, k2, v), (causal, sm_scale, w), heads, 2)


def piecewise_bwd_bhsd(q1, k1, q2, k2, v, do, causal, sm_scale=None, w=0, heads=None):
    return _run_bhsd(piecewise_bwd, (q1, k1, q2, k2, v, do), (causal, sm_scale, w), heads, 5)


def attention_jvp_bwd_bhsd(q, k, v, tq, tk, tv, do, dto, causal, sm_scale=None, heads=None):
    """[B,H,S,D] inputs -> (dq, dk, dv, dtq, dtk, dtv)."""
    return _run_bhsd(attention_jvp_bwd, (q, k, v, tq, tk, tv, do, dto), (causal, sm_scale), heads, 6)


def attention_jvp_tl_bhsd(q, k, tq, tk, causal, sm_scale=None, heads=None):
    """[B,H,S,D] inputs -> tL [B,H,M]."""
    return _run_bhsd(lambda *a: (attention_jvp_tl(*a),), (q, k, tq, tk), (causal, sm_scale), heads, 1)[0]


def lse_merge_fwd_bhsd(o1, l1, o2, l2, heads=None):
    """[B,H,M,D] / [B,H,M] inputs -> (O, L)."""
    return _run_bhsd(lse_merge_fwd, (o1, l1, o2, l2), (), heads, 2)


def lse_merge_bwd_bhsd(o1, l1, o2, l2, do, dl=None, heads=None):
    if dl is None:
        return _run_bhsd(lambda a, b, c, d, e: lse_merge_bwd(a, b, c, d, e, None), (o1, l1, o2, l2, do), (),
                         heads, 4)
    return _run_bhsd(lse_merge_bwd, (o1, l1, o2, l2, do, dl), (), heads, 4)


# ------------------------------------------------------- sampled query rows
def attention_rows(q, k, v, do, rows, causal: bool, sm_scale=None):
    """One head, only the listed query rows: (O[rows], L[rows], dQ[rows]).

    The same definitions as above restricted to rows i in `rows` (the mask
    uses the absolute index i); query rows are independent, so these are
    exactly the corresponding rows of attention_fwd / attention_bwd.  `do`
    may be None (then dQ is not computed)."""
    q, k, v = _f64(q, k, v)
    rows = np.asarray(rows, dtype=np.int64)
    M, N = q.shape[0], k.shape[0]
    s = default_scale(q.shape[1], sm_scale)
    if causal:
        keep = np.arange(N)[None, :] <= rows[:, None] + (N - M)
    else:
        keep = np.ones((len(rows), N), dtype=bool)
    P, L = _softmax(s * (q[rows] @ k.T), keep)
    O = P @ v
    if do is None:
        return O, L, None
    dor = _f64(do)[0][rows]
    delta = (dor * O).sum(axis=1)
    dS = P * (dor @ v.T - delta[:, None])
    return O, L, s * (dS @ k)
