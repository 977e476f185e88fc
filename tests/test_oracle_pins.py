"""Pins for the fp64 oracle against things other than itself.

Each check is chosen so that a plausible slip in the oracle -- a dropped
term, a wrong sign, a transposed operand, an off-by-one in the causal or
piecewise mask, the wrong log base for L -- fails at least one of them:

* brute force: explicit Python loops over the textbook definition;
* central finite differences of the forward (gradients and the JVP);
* the adjoint identity linking the backward to the JVP;
* closed forms and invariants (rows of P sum to 1, causal row 0, q = 0,
  shift invariances, sum of dK over keys);
* special cases of the piecewise rule that reduce to plain attention;
* a tiled online-softmax recurrence (the one the kernels use, written
  here from the tutorial's ``_attn_fwd_inner``) equal to the one-shot form.
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(12345)


def rand(*shape):
    return RNG.standard_normal(shape)


# ------------------------------------------------------------ brute force
def brute_fwd(q, k, v, causal, s, far=None, q2=None, k2=None, w=None):
    """Textbook softmax attention with explicit loops and math.exp."""
    M, D = q.shape
    N = k.shape[0]
    O = np.zeros((M, v.shape[1]))
    L = np.zeros(M)
    for i in range(M):
        scores = []
        for j in range(N):
            if causal and j > i + (N - M):
                continue
            if w is not None and (i + N - M - j) >= w:
                dot = sum(q2[i, d] * k2[j, d] for d in range(D))
            else:
                dot = sum(q[i, d] * k[j, d] for d in range(D))
            scores.append((j, s * dot))
        if not scores:
            L[i] = -math.inf
            continue
        mx = max(sc for _, sc in scores)
        den = sum(math.exp(sc - mx) for _, sc in scores)
        L[i] = mx + math.log(den)
        for j, sc in scores:
            pij = math.exp(sc - mx) / den
            for d in range(v.shape[1]):
                O[i, d] += pij * v[j, d]
    return O, L


@pytest.mark.parametrize("M,N,causal", [(3, 5, False), (5, 5, True), (3, 6, True), (6, 3, True),
                                        (4, 4, False), (1, 1, True), (7, 2, False)])
def test_fwd_matches_brute_force(M, N, causal):
    D = 4
    q, k, v = rand(M, D), rand(N, D), rand(N, 3 if D == 4 else D)
    s = 0.37
    O, L = oracle.attention_fwd(q, k, v, causal, s)
    Ob, Lb = brute_fwd(q, k, v, causal, s)
    np.testing.assert_allclose(O, Ob, atol=1e-13, rtol=0)
    fin = np.isfinite(Lb)
    assert np.array_equal(np.isfinite(L), fin)
    np.testing.assert_allclose(L[fin], Lb[fin], atol=1e-13, rtol=0)


@pytest.mark.parametrize("M,N,causal,w", [(5, 5, True, 2), (5, 5, False, 0), (4, 6, True, 3),
                                          (6, 4, False, -1), (5, 5, True, 1), (3, 7, False, 5)])
def test_piecewise_fwd_matches_brute_force(M, N, causal, w):
    D = 4
    q1, k1, q2, k2, v = rand(M, D), rand(N, D), rand(M, D), rand(N, D), rand(N, D)
    s = 0.5
    O, L = oracle.piecewise_fwd(q1, k1, q2, k2, v, causal, s, w)
    Ob, Lb = brute_fwd(q1, k1, v, causal, s, q2=q2, k2=k2, w=w)
    np.testing.assert_allclose(O, Ob, atol=1e-13, rtol=0)
    fin = np.isfinite(Lb)
    np.testing.assert_allclose(L[fin], Lb[fin], atol=1e-13, rtol=0)


def test_piecewise_boundary_distance_equal_w_uses_q2k2():
    """At signed distance exactly w the code path picks (q2, k2)."""
    M = N = 4
    D = 2
    w = 2
    q1 = np.zeros((M, D))
    k1 = np.zeros((N, D))
    q2 = np.ones((M, D))
    k2 = np.ones((N, D))
    v = np.eye(N)
    far = oracle.far_mask(M, N, w)
    # row i = 3: distances 3,2,1,0 for j = 0..3 -> far for j = 0, 1 (d >= 2)
    assert far[3].tolist() == [True, True, False, False]
    O, L = oracle.piecewise_fwd(q1, k1, q2, k2, v, False, 1.0, w)
    # far scores are q2.k2 = 2, near scores are 0
    e = math.exp(2.0)
    den = 2 * e + 2
    np.testing.assert_allclose(O[3], [e / den, e / den, 1 / den, 1 / den], atol=1e-15)
    np.testing.assert_allclose(L[3], math.log(den), atol=1e-15)
    # negative distances (future keys) stay on (q1, k1) even for w <= 0 ... only when d < w
    far0 = oracle.far_mask(2, 4, 0)
    assert far0.tolist() == [[True, True, True, False], [True, True, True, True]]


# ------------------------------------------------------------ invariants
@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_P_sum_to_one(causal):
    M, N, D = 9, 9, 5
    q, k = rand(M, D), rand(N, D)
    O, _ = oracle.attention_fwd(q, k, np.ones((N, 2)), causal, 0.8)
    np.testing.assert_allclose(O, 1.0, atol=1e-14)


def test_causal_row0_returns_v0_and_its_score():
    M = N = 6
    D = 4
    q, k, v = rand(M, D), rand(N, D), rand(N, D)
    s = 0.3
    O, L = oracle.attention_fwd(q, k, v, True, s)
    np.testing.assert_allclose(O[0], v[0], atol=1e-15)
    np.testing.assert_allclose(L[0], s * q[0] @ k[0], atol=1e-15)


@pytest.mark.parametrize("M,N,causal", [(6, 6, True), (4, 7, True), (5, 5, False)])
def test_zero_query_gives_mean_and_log_count(M, N, causal):
    D = 3
    k, v = rand(N, D), rand(N, D)
    O, L = oracle.attention_fwd(np.zeros((M, D)), k, v, causal, 1.0)
    for i in range(M):
        vis = [j for j in range(N) if (not causal) or j <= i + N - M]
        np.testing.assert_allclose(O[i], v[vis].mean(axis=0), atol=1e-14)
        np.testing.assert_allclose(L[i], math.log(len(vis)), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_shift_invariances(causal):
    M, N, D = 5, 7, 4
    q, k, v = rand(M, D), rand(N, D), rand(N, D)
    c = rand(D)
    O, L = oracle.attention_fwd(q, k, v, causal, 0.6)
    O2, _ = oracle.attention_fwd(q, k, v + c, causal, 0.6)
    np.testing.assert_allclose(O2, O + c, atol=1e-13)
    O3, L3 = oracle.attention_fwd(q, k + c, v, causal, 0.6)
    np.testing.assert_allclose(O3, O, atol=1e-13)
    # L shifts by s * q_i . c on every row
    np.testing.assert_allclose(L3, L + 0.6 * (q @ c), atol=1e-13)


def test_empty_rows_give_zero_output_minus_inf_lse_and_zero_grads():
    M, N, D = 6, 3, 4
    q, k, v, do = rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    O, L = oracle.attention_fwd(q, k, v, True, 0.5)
    # rows i with i + N - M < 0 see no key
    empty = [i for i in range(M) if i + N - M < 0]
    assert empty == [0, 1, 2]
    assert np.all(O[empty] == 0) and np.all(np.isneginf(L[empty]))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, 0.5)
    assert np.all(dq[empty] == 0)


def test_default_scale_is_inverse_sqrt_d():
    assert oracle.default_scale(64) == 0.125
    assert oracle.default_scale(128, -1.0) == 1.0 / math.sqrt(128)
    assert oracle.default_scale(64, 0.5) == 0.5


# ----------------------------------------------------- finite differences
def _fd_grad(f, x, h=1e-5):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + h
        fp = f()
        x[idx] = old - h
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * h)
    return g


@pytest.mark.parametrize("M,N,D,causal", [(1, 1, 4, True), (3, 3, 4, False), (5, 5, 8, True),
                                          (3, 5, 4, True), (5, 3, 4, True), (17, 17, 4, True),
                                          (4, 6, 8, False)])
def test_backward_matches_finite_differences(M, N, D, causal):
    q, k, v, do = rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    s = 0.7

    def f():
        O, _ = oracle.attention_fwd(q, k, v, causal, s)
        return float((O * do).sum())

    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, s)
    for x, g in ((q, dq), (k, dk), (v, dv)):
        np.testing.assert_allclose(g, _fd_grad(f, x), atol=2e-8, rtol=1e-6)


@pytest.mark.parametrize("M,N,D,causal,w", [(5, 5, 4, True, 2), (5, 5, 4, False, 0), (4, 6, 4, True, 1),
                                            (6, 4, 4, False, -2), (6, 6, 4, True, 0), (6, 6, 4, True, 10),
                                            (6, 6, 4, True, -10)])
def test_piecewise_backward_matches_finite_differences(M, N, D, causal, w):
    q1, k1, q2, k2, v, do = rand(M, D), rand(N, D), rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    s = 0.6

    def f():
        O, _ = oracle.piecewise_fwd(q1, k1, q2, k2, v, causal, s, w)
        return float((O * do).sum())

    grads = oracle.piecewise_bwd(q1, k1, q2, k2, v, do, causal, s, w)
    for x, g in zip((q1, k1, q2, k2, v), grads):
        np.testing.assert_allclose(g, _fd_grad(f, x), atol=2e-8, rtol=1e-6)


@pytest.mark.parametrize("M,N,D,causal", [(4, 4, 4, False), (6, 6, 8, True), (3, 5, 4, True),
                                          (5, 3, 4, True), (17, 17, 4, False)])
def test_jvp_matches_finite_differences(M, N, D, causal):
    q, k, v = rand(M, D), rand(N, D), rand(N, D)
    tq, tk, tv = rand(M, D), rand(N, D), rand(N, D)
    s = 0.45
    eps = 1e-5
    O, L, tO = oracle.attention_jvp(q, k, v, tq, tk, tv, causal, s)
    Op, _ = oracle.attention_fwd(q + eps * tq, k + eps * tk, v + eps * tv, causal, s)
    Om, _ = oracle.attention_fwd(q - eps * tq, k - eps * tk, v - eps * tv, causal, s)
    np.testing.assert_allclose(tO, (Op - Om) / (2 * eps), atol=1e-8, rtol=1e-6)
    O0, L0 = oracle.attention_fwd(q, k, v, causal, s)
    np.testing.assert_array_equal(O, O0)
    np.testing.assert_array_equal(L, L0)


@pytest.mark.parametrize("causal", [False, True])
def test_adjoint_identity_ties_backward_to_jvp(causal):
    M, N, D = 7, 9, 5
    q, k, v, do = rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    tq, tk, tv = rand(M, D), rand(N, D), rand(N, D)
    s = 0.4
    _, _, tO = oracle.attention_jvp(q, k, v, tq, tk, tv, causal, s)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, causal, s)
    lhs = float((do * tO).sum())
    rhs = float((dq * tq).sum() + (dk * tk).sum() + (dv * tv).sum())
    assert abs(lhs - rhs) < 1e-12 * max(1.0, abs(lhs))


@pytest.mark.parametrize("causal", [False, True])
def test_sum_of_dk_over_keys_is_zero(causal):
    M, N, D = 8, 8, 4
    q, k, v, do = rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    _, dk, _ = oracle.attention_bwd(q, k, v, do, causal, 0.9)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-13)


@pytest.mark.parametrize("M,N,causal", [(5, 7, False), (6, 6, True), (7, 4, True)])
def test_delta_is_the_row_sum_of_p_times_dp(M, N, causal):
    """delta_i = <dO_i, O_i> equals sum_j P_ij dP_ij with dP = dO V^T, P taken
    by the brute-force loops (V = identity makes the loop's output P itself);
    rows that see no key have O = 0 and delta = 0."""
    D = 3
    q, k, v, do = rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    P, _ = brute_fwd(q, k, np.eye(N), causal, 0.7)
    O = P @ v
    want = [sum(P[i, j] * sum(do[i, d] * v[j, d] for d in range(D)) for j in range(N)) for i in range(M)]
    np.testing.assert_allclose(oracle.bwd_delta(O, do), want, atol=1e-12)
    got = oracle.bwd_delta_bhsd(O[None, None], do[None, None])
    assert got.shape == (1, 1, M)
    np.testing.assert_allclose(got[0, 0], want, atol=1e-12)


# --------------------------------------------- piecewise special cases
def test_piecewise_all_far_or_all_near_reduces_to_attention():
    M, N, D = 6, 6, 4
    q1, k1, q2, k2, v, do = rand(M, D), rand(N, D), rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    for causal in (False, True):
        # w <= 1 - M: every distance is >= w -> (q2, k2) everywhere
        Of, Lf = oracle.piecewise_fwd(q1, k1, q2, k2, v, causal, 0.5, -(M + N))
        Oa, La = oracle.attention_fwd(q2, k2, v, causal, 0.5)
        np.testing.assert_allclose(Of, Oa, atol=1e-14)
        np.testing.assert_allclose(Lf, La, atol=1e-14)
        # w > N - 1: every distance is < w -> (q1, k1) everywhere
        On, Ln = oracle.piecewise_fwd(q1, k1, q2, k2, v, causal, 0.5, M + N)
        Ob, Lb = oracle.attention_fwd(q1, k1, v, causal, 0.5)
        np.testing.assert_allclose(On, Ob, atol=1e-14)
        g = oracle.piecewise_bwd(q1, k1, q2, k2, v, do, causal, 0.5, M + N)
        ga = oracle.attention_bwd(q1, k1, v, do, causal, 0.5)
        np.testing.assert_allclose(g[0], ga[0], atol=1e-14)
        np.testing.assert_allclose(g[1], ga[1], atol=1e-14)
        np.testing.assert_allclose(g[4], ga[2], atol=1e-14)
        assert np.all(g[2] == 0) and np.all(g[3] == 0)


@pytest.mark.parametrize("w", [-3, 0, 2, 4])
def test_piecewise_with_equal_pairs_is_standard_attention(w):
    M, N, D = 6, 6, 4
    q, k, v, do = rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    O, L = oracle.piecewise_fwd(q, k, q, k, v, True, 0.5, w)
    Oa, La = oracle.attention_fwd(q, k, v, True, 0.5)
    np.testing.assert_allclose(O, Oa, atol=1e-14)
    dq1, dk1, dq2, dk2, dv = oracle.piecewise_bwd(q, k, q, k, v, do, True, 0.5, w)
    dq, dk, dva = oracle.attention_bwd(q, k, v, do, True, 0.5)
    np.testing.assert_allclose(dq1 + dq2, dq, atol=1e-13)
    np.testing.assert_allclose(dk1 + dk2, dk, atol=1e-13)
    np.testing.assert_allclose(dv, dva, atol=1e-13)


# ---------------------------------------- online softmax == one-shot softmax
def online_softmax_fwd(q, k, v, causal, s, block=3):
    """The running (m, l, acc) recurrence of the tutorial's _attn_fwd_inner in
    base 2, visiting keys in blocks; written here only to pin the oracle."""
    M, N = q.shape[0], k.shape[0]
    c = s / math.log(2.0)
    m = np.full(M, -np.inf)
    l = np.zeros(M)
    acc = np.zeros((M, v.shape[1]))
    keep = oracle.allowed_mask(M, N, causal)
    for j0 in range(0, N, block):
        j1 = min(N, j0 + block)
        x = np.where(keep[:, j0:j1], (q @ k[j0:j1].T) * c, -np.inf)
        mnew = np.maximum(m, x.max(axis=1))
        ref = np.where(np.isfinite(mnew), mnew, 0.0)
        p = np.exp2(x - ref[:, None])
        alpha = np.exp2(np.where(np.isfinite(m), m, -np.inf) - ref)
        l = l * alpha + p.sum(axis=1)
        acc = acc * alpha[:, None] + p @ v[j0:j1]
        m = mnew
    with np.errstate(divide="ignore", invalid="ignore"):
        O = np.where(l[:, None] > 0, acc / l[:, None], 0.0)
        L = np.where(l > 0, (m + np.log2(np.where(l > 0, l, 1.0))) * math.log(2.0), -np.inf)
    return O, L


@pytest.mark.parametrize("M,N,causal,block", [(10, 10, True, 3), (10, 13, False, 4), (9, 9, True, 1),
                                              (12, 7, True, 5)])
def test_tiled_online_softmax_equals_one_shot(M, N, causal, block):
    D = 6
    q, k, v = 3 * rand(M, D), 3 * rand(N, D), rand(N, D)
    O, L = oracle.attention_fwd(q, k, v, causal, 0.7)
    Ot, Lt = online_softmax_fwd(q, k, v, causal, 0.7, block)
    np.testing.assert_allclose(Ot, O, atol=1e-12)
    fin = np.isfinite(L)
    assert np.array_equal(fin, np.isfinite(Lt))
    np.testing.assert_allclose(Lt[fin], L[fin], atol=1e-12)


def test_bhsd_wrappers_fill_selected_heads_only():
    import torch
    B, H, M, D = 2, 3, 5, 4
    q = torch.randn(B, H, M, D, dtype=torch.float64)
    k = torch.randn(B, H, M, D, dtype=torch.float64)
    v = torch.randn(B, H, M, D, dtype=torch.float64)
    O, L = oracle.attention_fwd_bhsd(q, k, v, True, None, heads=[(1, 2)])
    Oh, Lh = oracle.attention_fwd(q[1, 2].numpy(), k[1, 2].numpy(), v[1, 2].numpy(), True, None)
    np.testing.assert_array_equal(O[1, 2], Oh)
    assert np.all(O[0] == 0)


@pytest.mark.parametrize("M,N,causal", [(9, 9, True), (7, 11, True), (11, 6, True), (8, 8, False)])
def test_sampled_rows_match_brute_force_and_finite_differences(M, N, causal):
    """Row-sampled O, L, dQ: rows of the textbook loops and of the FD gradient."""
    D = 4
    q, k, v, do = rand(M, D), rand(N, D), rand(N, D), rand(M, D)
    s = 0.55
    rows = [0, M // 2, M - 1]
    O, L, dQ = oracle.attention_rows(q, k, v, do, rows, causal, s)
    Ob, Lb = brute_fwd(q, k, v, causal, s)
    np.testing.assert_allclose(O, Ob[rows], atol=1e-13)
    fin = np.isfinite(Lb[rows])
    np.testing.assert_allclose(L[fin], Lb[rows][fin], atol=1e-13)

    def f():
        Of, _ = brute_fwd(q, k, v, causal, s)
        return float((Of * do).sum())

    g = _fd_grad(f, q)
    np.testing.assert_allclose(dQ, g[rows], atol=2e-8, rtol=1e-6)


# ---------------------------------------------------------------- LSE merge
def _brute_attention_masked(q, k, v, keep, s):
    """Attention over an explicit keep mask with loops (rows with no key: O = 0, L = -inf)."""
    M, N = keep.shape
    O = np.zeros((M, v.shape[1]))
    L = np.full(M, -math.inf)
    for i in range(M):
        sc = [(j, s * float(q[i] @ k[j])) for j in range(N) if keep[i, j]]
        if not sc:
            continue
        mx = max(x for _, x in sc)
        den = sum(math.exp(x - mx) for _, x in sc)
        L[i] = mx + math.log(den)
        for j, x in sc:
            O[i] += math.exp(x - L[i]) * v[j]
    return O, L


@pytest.mark.parametrize("M,N,split,causal", [(7, 11, 4, False), (9, 9, 5, True), (6, 10, 0, False),
                                              (8, 12, 12, True)])
def test_merge_of_two_key_sets_is_attention_over_their_union(M, N, split, causal):
    """Attention over keys [0, split) and [split, N) separately, merged, is
    attention over all N keys -- also when one part is empty for some or all
    rows (causal: the later keys are invisible to the first queries)."""
    q, k, v = rand(M, 5), rand(N, 5), rand(N, 3)
    s = 0.7
    keep = oracle.allowed_mask(M, N, causal)
    part1 = keep.copy()
    part1[:, split:] = False
    part2 = keep.copy()
    part2[:, :split] = False
    O1, L1 = _brute_attention_masked(q, k, v, part1, s)
    O2, L2 = _brute_attention_masked(q, k, v, part2, s)
    O, L = oracle.lse_merge_fwd(O1, L1, O2, L2)
    Of, Lf = oracle.attention_fwd(q, k, v, causal, s)
    np.testing.assert_allclose(O, Of, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(L), np.isneginf(Lf))
    np.testing.assert_allclose(L[np.isfinite(Lf)], Lf[np.isfinite(Lf)], atol=1e-12)


def test_merge_is_symmetric_and_handles_empty_parts():
    M, D = 6, 4
    o1, o2 = rand(M, D), rand(M, D)
    l1, l2 = rand(M) * 3, rand(M) * 3
    O, L = oracle.lse_merge_fwd(o1, l1, o2, l2)
    Os, Ls = oracle.lse_merge_fwd(o2, l2, o1, l1)
    np.testing.assert_allclose(O, Os, atol=1e-14)
    np.testing.assert_allclose(L, Ls, atol=1e-14)
    # closed form: L = ln(e^L1 + e^L2), O = (e^L1 O1 + e^L2 O2) / e^L
    np.testing.assert_allclose(L, np.log(np.exp(l1) + np.exp(l2)), atol=1e-12)
    np.testing.assert_allclose(O, (np.exp(l1)[:, None] * o1 + np.exp(l2)[:, None] * o2) / np.exp(L)[:, None],
                               atol=1e-12)
    # one empty part passes the other through; two empty parts give O = 0, L = -inf
    l2e = l2.copy()
    l2e[:3] = -np.inf
    l1e = l1.copy()
    l1e[1] = -np.inf
    O, L = oracle.lse_merge_fwd(o1, l1e, o2, l2e)
    np.testing.assert_allclose(O[0], o1[0], atol=1e-15)
    assert L[0] == l1e[0] and np.isneginf(L[1]) and np.all(O[1] == 0)
    do1, dl1, do2, dl2 = oracle.lse_merge_bwd(o1, l1e, o2, l2e, rand(M, D), rand(M))
    assert np.all(do1[1] == 0) and np.all(do2[1] == 0) and dl1[1] == 0 and dl2[1] == 0
    assert np.all(do2[0] == 0) and dl2[0] == 0


@pytest.mark.parametrize("with_dl", [False, True])
def test_merge_backward_matches_finite_differences(with_dl):
    M, D = 5, 3
    o1, o2, l1, l2 = rand(M, D), rand(M, D), rand(M), rand(M)
    G, g = rand(M, D), (rand(M) if with_dl else np.zeros(M))

    def f(o1_, l1_, o2_, l2_):
        O, L = oracle.lse_merge_fwd(o1_, l1_, o2_, l2_)
        return float((G * O).sum() + (g * L).sum())

    do1, dl1, do2, dl2 = oracle.lse_merge_bwd(o1, l1, o2, l2, G, g if with_dl else None)
    h = 1e-6
    args = [o1, l1, o2, l2]
    for idx, grad in zip(range(4), (do1, dl1, do2, dl2)):
        fd = np.zeros_like(args[idx])
        for pos in np.ndindex(args[idx].shape):
            a_p = [a.copy() for a in args]
            a_m = [a.copy() for a in args]
            a_p[idx][pos] += h
            a_m[idx][pos] -= h
            fd[pos] = (f(*a_p) - f(*a_m)) / (2 * h)
        np.testing.assert_allclose(grad, fd, atol=1e-8, rtol=1e-7)


@pytest.mark.parametrize("M,N,causal", [(6, 6, True), (5, 9, False), (9, 5, True)])
def test_jvp_tangent_of_lse_matches_finite_differences(M, N, causal):
    """tL = mu is the derivative of L along (tq, tk) (central differences);
    rows that see no key have L = -inf and tL = 0."""
    q, k, tq, tk = rand(M, 4), rand(N, 4), rand(M, 4), rand(N, 4)
    s = 0.6
    tl = oracle.attention_jvp_tl(q, k, tq, tk, causal, s)
    h = 1e-6
    _, Lp = oracle.attention_fwd(q + h * tq, k + h * tk, rand(N, 2), causal, s)
    _, Lm = oracle.attention_fwd(q - h * tq, k - h * tk, rand(N, 2), causal, s)
    fin = np.isfinite(Lp)
    fd = (Lp[fin] - Lm[fin]) / (2 * h)
    np.testing.assert_allclose(tl[fin], fd, atol=1e-7)
    assert np.all(tl[~fin] == 0)
    # and it is the mu of the JVP: tO = (P o T) V - mu O + P tV with tv = 0, v = 1 gives tO = sum(P o T) - mu = 0
    _, _, tO = oracle.attention_jvp(q, k, np.ones((N, 1)), tq, tk, np.zeros((N, 1)), causal, s)
    np.testing.assert_allclose(tO[fin], 0.0, atol=1e-12)


# ------------------------------------------------- backward of the JVP
@pytest.mark.parametrize("M,N,D,causal", [(1, 1, 4, True), (4, 4, 4, False), (5, 5, 4, True),
                                          (3, 6, 4, True), (6, 3, 4, True), (5, 7, 3, False)])
def test_jvp_backward_matches_finite_differences(M, N, D, causal):
    """Gradients of <dO, O> + <dtO, tO> against central differences of that
    scalar, O and tO from the (separately pinned) JVP forward."""
    xs = [rand(M, D), rand(N, D), rand(N, D), rand(M, D), rand(N, D), rand(N, D)]
    do, dto = rand(M, D), rand(M, D)
    s = 0.55

    def f():
        O, _, tO = oracle.attention_jvp(*xs, causal, s)
        return float((O * do).sum() + (tO * dto).sum())

    grads = oracle.attention_jvp_bwd(*xs, do, dto, causal, s)
    for x, g in zip(xs, grads):
        np.testing.assert_allclose(g, _fd_grad(f, x), atol=1e-8, rtol=1e-6)


@pytest.mark.parametrize("causal", [False, True])
def test_jvp_backward_tangent_grads_are_the_plain_backward_of_dto(causal):
    """tO is linear in the tangents with the Jacobian of O, so the tangents'
    gradients are the plain backward with dO replaced by dtO; with dtO = 0
    the primal gradients are the plain backward of dO."""
    M, N, D = 7, 9, 4
    q, k, v, tq, tk, tv = rand(M, D), rand(N, D), rand(N, D), rand(M, D), rand(N, D), rand(N, D)
    do, dto = rand(M, D), rand(M, D)
    s = 0.5
    _, _, _, dtq, dtk, dtv = oracle.attention_jvp_bwd(q, k, v, tq, tk, tv, do, dto, causal, s)
    for a, b in zip((dtq, dtk, dtv), oracle.attention_bwd(q, k, v, dto, causal, s)):
        np.testing.assert_allclose(a, b, atol=1e-13)
    g = oracle.attention_jvp_bwd(q, k, v, tq, tk, tv, do, np.zeros((M, D)), causal, s)
    for a, b in zip(g[:3], oracle.attention_bwd(q, k, v, do, causal, s)):
        np.testing.assert_allclose(a, b, atol=1e-13)
    for a in g[3:]:
        assert np.all(a == 0)
    # Euler: tO is homogeneous of degree 1 in the tangents
    _, _, tO = oracle.attention_jvp(q, k, v, tq, tk, tv, causal, s)
    lhs = float((dtq * tq).sum() + (dtk * tk).sum() + (dtv * tv).sum())
    assert abs(lhs - float((dto * tO).sum())) < 1e-12 * max(1.0, abs(lhs))


@pytest.mark.parametrize("causal", [False, True])
def test_jvp_backward_second_order_part_is_symmetric(causal):
    """With dO = 0 the primal gradients are the gradient of <dtO, J(x) t>, a
    mixed second derivative: <G(t), u> = <G(u), t> for any two tangents."""
    M, N, D = 6, 8, 3
    x = [rand(M, D), rand(N, D), rand(N, D)]
    t = [rand(M, D), rand(N, D), rand(N, D)]
    u = [rand(M, D), rand(N, D), rand(N, D)]
    dto = rand(M, D)
    z = np.zeros((M, D))
    gt = oracle.attention_jvp_bwd(*x, *t, z, dto, causal, 0.6)[:3]
    gu = oracle.attention_jvp_bwd(*x, *u, z, dto, causal, 0.6)[:3]
    a = sum(float((g * w).sum()) for g, w in zip(gt, u))
    b = sum(float((g * w).sum()) for g, w in zip(gu, t))
    assert abs(a - b) < 1e-11 * max(1.0, abs(a))
