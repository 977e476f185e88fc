"""Seeded random sweep of shapes through every 16-bit entry point against the
fp64 oracle: M and N from 1 to 700 (ragged tails, M > N with empty rows,
N < 64), D in {16, 32, 64, 128}, fp16 and bf16, causal or not, piecewise w
anywhere from far below to far above the distances present.  The cases are
drawn once from a fixed seed, so the sweep is the same on every run.

Odd shapes make large values (one key and many queries: dV sums dO over all
of them, |dV| ~ 37), where the stored 16-bit result's own rounding exceeds
the flat unit-scale tolerance; each element is therefore held to the
tolerance plus the output type's unit roundoff times |ref|."""
import numpy as np
import pytest

import oracle
from _parity import ROUND_U, TOL, compare, compare_bounded, inputs, jvp_bwd_bounds, o_tol

pytestmark = pytest.mark.gpu


def _cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.choice([1, 7, 63, 64, 65, 127, 128, 129, 200, 255, 256, 383, 511, 700]))
        N = int(rng.choice([1, 5, 63, 64, 100, 128, 129, 257, 300, 512, 700]))
        D = int(rng.choice([16, 32, 64, 128]))
        dt = str(rng.choice(["f16", "bf16"]))
        causal = bool(rng.integers(0, 2))
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 3))
        w = int(rng.integers(-300, 800))
        out.append((B, H, M, N, D, dt, causal, w))
    return out


CASES = _cases(48, 20261202)


@pytest.mark.parametrize("B,H,M,N,D,dt,causal,w", CASES)
def test_random_shapes_every_entry_point(gpu_lib, B, H, M, N, D, dt, causal, w):
    ta = gpu_lib
    names = ("q", "k", "v", "do", "tq", "tk", "tv", "dto")
    cpu, g = inputs(B, H, M, N, D, dt, 81, names)
    # forward + backward
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    # JVP forward (with tL) and its backward
    o2, lse2, to, tlse = ta.attn_fwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], causal=causal,
                                         with_tlse=True)
    jg = ta.attn_bwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], o2, lse2, to, tlse, g["do"], g["dto"],
                         causal=causal)
    # piecewise: (q, k) near, (tq, tk) far
    po, plse = ta.piecewise_fwd(g["q"], g["k"], g["tq"], g["tk"], g["v"], w, causal)
    pg = ta.piecewise_bwd(g["q"], g["k"], g["tq"], g["tk"], g["v"], po, plse, g["do"], w, causal)
    assert ta.sync_status() == "TA_OK"

    c = cpu
    u = ROUND_U[dt]  # the stored 16-bit results' own rounding, for large sums at odd shapes
    O, L = oracle.attention_fwd_bhsd(c["q"], c["k"], c["v"], causal)
    compare("O", o, O, o_tol(dt), u)
    compare("L", lse, L, TOL["L"])
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), oracle.attention_bwd_bhsd(c["q"], c["k"], c["v"],
                                                                                      c["do"], causal)):
        compare(name, got, r, TOL["grad"], u)
    _, _, tO = oracle.attention_jvp_bhsd(c["q"], c["k"], c["v"], c["tq"], c["tk"], c["tv"], causal)
    compare("O(jvp)", o2, O, o_tol(dt), u)
    compare("tO", to, tO, TOL["tO"], u)
    compare("tL", tlse, oracle.attention_jvp_tl_bhsd(c["q"], c["k"], c["tq"], c["tk"], causal), TOL["L"])
    jref = oracle.attention_jvp_bwd_bhsd(c["q"], c["k"], c["v"], c["tq"], c["tk"], c["tv"], c["do"], c["dto"],
                                         causal)
    bounds = jvp_bwd_bounds(c, causal, u)
    for name, got, r in zip(("dq", "dk", "dv", "dtq", "dtk", "dtv"), jg, jref):
        compare_bounded("jvp " + name, got, r, TOL["grad"], bounds[name])
    PO, PL = oracle.piecewise_fwd_bhsd(c["q"], c["k"], c["tq"], c["tk"], c["v"], causal, None, w)
    compare("O(pw)", po, PO, o_tol(dt), u)
    compare("L(pw)", plse, PL, TOL["L"])
    pref = oracle.piecewise_bwd_bhsd(c["q"], c["k"], c["tq"], c["tk"], c["v"], c["do"], causal, None, w)
    for name, got, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), pg, pref):
        compare("pw " + name, got, r, TOL["grad"], u)


F32_CASES = [c for c in _cases(24, 20261203) if c[2] <= 300 and c[3] <= 300]


@pytest.mark.parametrize("B,H,M,N,D,dt,causal,w", F32_CASES)
def test_random_shapes_fp32_mode(gpu_lib, B, H, M, N, D, dt, causal, w):
    """The same entry points in the fp32 mode (float32 in and out, SIMT
    kernels), held to 1e-4 plus the float32 rounding of large values."""
    import synth_inputs as si
    ta = gpu_lib
    names = ("q", "k", "v", "do", "tq", "tk", "tv", "dto")
    c = {n: si.randn((B, H, M if n in ("q", "do", "tq", "dto") else N, D), "f32", si.seed_for(82, i))
         for i, n in enumerate(names)}
    g = {n: t.cuda() for n, t in c.items()}
    u = 2.0 ** -24
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    o2, lse2, to, tlse = ta.attn_fwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], causal=causal,
                                         with_tlse=True)
    jg = ta.attn_bwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], o2, lse2, to, tlse, g["do"], g["dto"],
                         causal=causal)
    po, plse = ta.piecewise_fwd(g["q"], g["k"], g["tq"], g["tk"], g["v"], w, causal)
    pg = ta.piecewise_bwd(g["q"], g["k"], g["tq"], g["tk"], g["v"], po, plse, g["do"], w, causal)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.attention_fwd_bhsd(c["q"], c["k"], c["v"], causal)
    compare("O", o, O, 1e-4, u)
    compare("L", lse, L, 1e-4)
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), oracle.attention_bwd_bhsd(c["q"], c["k"], c["v"],
                                                                                      c["do"], causal)):
        compare(name, got, r, 1e-4, u)
    _, _, tO = oracle.attention_jvp_bhsd(c["q"], c["k"], c["v"], c["tq"], c["tk"], c["tv"], causal)
    compare("tO", to, tO, 1e-4, u)
    compare("tL", tlse, oracle.attention_jvp_tl_bhsd(c["q"], c["k"], c["tq"], c["tk"], causal), 1e-4)
    jref = oracle.attention_jvp_bwd_bhsd(c["q"], c["k"], c["v"], c["tq"], c["tk"], c["tv"], c["do"], c["dto"],
                                         causal)
    for name, got, r in zip(("dq", "dk", "dv", "dtq", "dtk", "dtv"), jg, jref):
        compare("jvp " + name, got, r, 1e-4, u)
    PO, PL = oracle.piecewise_fwd_bhsd(c["q"], c["k"], c["tq"], c["tk"], c["v"], causal, None, w)
    compare("O(pw)", po, PO, 1e-4, u)
    pref = oracle.piecewise_bwd_bhsd(c["q"], c["k"], c["tq"], c["tk"], c["v"], c["do"], causal, None, w)
    for name, got, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), pg, pref):
        compare("pw " + name, got, r, 1e-4, u)


def _merge_fp8_cases(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        M = int(rng.choice([1, 17, 128, 200, 513]))
        N = int(rng.choice([16, 48, 128, 208, 512]))
        D = int(rng.choice([64, 128]))
        out.append((int(rng.integers(1, 3)), int(rng.integers(1, 3)), M, N, D, bool(rng.integers(0, 2))))
    return out


@pytest.mark.parametrize("B,H,M,N,D,causal", _merge_fp8_cases(12, 20261204))
def test_random_shapes_fp8_forward_and_merge(gpu_lib, B, H, M, N, D, causal):
    """attn_fwd_fp8 (N a multiple of 16) within its e5m2 rounding bound, and
    the merge of two partial states of random shape."""
    import synth_inputs as si
    import torch
    ta = gpu_lib
    U = 2.0 ** -3
    q = si.randn((B, H, M, D), "e5m2", si.seed_for(83, 0))
    k = si.randn((B, H, N, D), "e5m2", si.seed_for(83, 1))
    v = si.randn((B, H, N, D), "e5m2", si.seed_for(83, 2))
    o, lse = ta.attn_fwd_fp8(q.cuda(), k.cuda(), v.transpose(-1, -2).contiguous().cuda(), causal)
    assert ta.sync_status() == "TA_OK"
    o = o.cpu().to(torch.float64).numpy()
    lse = lse.cpu().numpy()
    s = oracle.default_scale(D)
    keep = oracle.allowed_mask(M, N, causal)
    for b in range(B):
        for h in range(H):
            qf, kf, vf = (t[b, h].to(torch.float64).numpy() for t in (q, k, v))
            O, L = oracle.attention_fwd(qf, kf, vf, causal)
            fin = np.isfinite(L)
            S = np.where(keep, s * qf @ kf.T, -np.inf)
            P = np.zeros_like(S)
            P[fin] = np.exp(S[fin] - L[fin, None])
            bound = U * (1 + U) * (P @ np.abs(vf)) + U * np.abs(O) + 1e-6
            assert np.all(np.abs(o[b, h] - O) <= bound)
            np.testing.assert_array_equal(np.isneginf(lse[b, h]), ~fin)
            np.testing.assert_allclose(lse[b, h][fin], L[fin], atol=1e-3)
    # merge of two random partial states of the same shape (bf16)
    o1, o2, dO = (si.randn((B, H, M, D), "bf16", si.seed_for(84, i)) for i in range(3))
    l1, l2, dl = (si.randn((B, H, M), "f32", si.seed_for(84, 3 + i)) * 3 for i in range(3))
    gm = [t.cuda() for t in (o1, l1, o2, l2, dO, dl)]
    mo, ml = ta.merge_fwd(gm[0], gm[1], gm[2], gm[3])
    grads = ta.merge_bwd(*gm)
    assert ta.sync_status() == "TA_OK"
    MO, ML = oracle.lse_merge_fwd_bhsd(o1, l1, o2, l2)
    compare("merge O", mo, MO, o_tol("bf16"), ROUND_U["bf16"])
    compare("merge L", ml, ML, 1e-5)
    for name, got, r in zip(("dO1", "dL1", "dO2", "dL2"), grads, oracle.lse_merge_bwd_bhsd(o1, l1, o2, l2, dO, dl)):
        compare("merge " + name, got, r, TOL["grad"] if name.startswith("dO") else 1e-4,
                ROUND_U["bf16"] if name.startswith("dO") else 2.0 ** -24)
