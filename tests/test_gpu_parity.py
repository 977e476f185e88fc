"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Small cases compare every element of every head; the benchmark-sized
workloads run the same launch configuration the benchmark times and compare
sampled heads (heads are independent) or sampled query rows.  Tolerances
(max_abs, unit-normal inputs): O 1e-2 (fp16) / 2e-2 (bf16), L 1e-3,
gradients and tO 5e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from _parity import TOL, all_heads, compare, heads_of, inputs, o_tol, sample_heads

pytestmark = pytest.mark.gpu

FWD_CASES = [
    # B, H, M, N, D, dtype, causal
    (1, 2, 128, 128, 64, "f16", False),
    (1, 2, 128, 128, 64, "f16", True),
    (2, 3, 256, 256, 128, "bf16", True),
    (1, 2, 384, 384, 128, "f16", False),
    (1, 2, 200, 333, 64, "bf16", True),
    (1, 2, 333, 200, 128, "bf16", True),   # M > N: first rows see no key
    (1, 1, 1, 1, 64, "f16", True),
    (1, 1, 5, 700, 64, "bf16", False),
    (1, 1, 700, 5, 128, "f16", False),
    (2, 1, 129, 257, 64, "bf16", True),
    (1, 2, 200, 200, 32, "bf16", True),    # D = 32, 16: the D = 64 kernels over zero-filled columns
    (1, 2, 131, 257, 16, "f16", False),
]


def _fwd_check(B, H, M, N, D, dtype, causal, workload=11):
    cpu, g = inputs(B, H, M, N, D, dtype, workload, ("q", "k", "v"))
    o, lse = gpu_lib_mod().attn_fwd(g["q"], g["k"], g["v"], causal)
    assert gpu_lib_mod().sync_status() == "TA_OK"
    O, L = oracle.attention_fwd_bhsd(cpu["q"], cpu["k"], cpu["v"], causal)
    compare("O", o, O, o_tol(dtype))
    compare("L", lse, L, TOL["L"])


def gpu_lib_mod():
    import tiled_attention_tcgen05_gb300 as ta
    return ta


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", FWD_CASES)
def test_fwd_small(gpu_lib, B, H, M, N, D, dtype, causal):
    _fwd_check(B, H, M, N, D, dtype, causal)


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", FWD_CASES)
def test_bwd_small(gpu_lib, B, H, M, N, D, dtype, causal):
    ta = gpu_lib
    cpu, g = inputs(B, H, M, N, D, dtype, 12, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    assert ta.sync_status() == "TA_OK"
    dQ, dK, dV = oracle.attention_bwd_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["do"], causal)
    compare("dQ", dq, dQ, TOL["grad"])
    compare("dK", dk, dK, TOL["grad"])
    compare("dV", dv, dV, TOL["grad"])


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", [
    (1, 2, 128, 128, 64, "f16", False), (1, 2, 256, 256, 64, "f16", True), (1, 2, 256, 256, 128, "bf16", True),
    (1, 1, 200, 333, 64, "f16", True), (1, 1, 333, 200, 128, "bf16", False), (1, 1, 300, 100, 64, "f16", True),
    (1, 2, 200, 200, 32, "bf16", True), (1, 1, 130, 190, 16, "f16", False)])
def test_jvp_small(gpu_lib, B, H, M, N, D, dtype, causal):
    ta = gpu_lib
    names = ("q", "k", "v", "tq", "tk", "tv")
    cpu, g = inputs(B, H, M, N, D, dtype, 13, names)
    o, lse, to, tlse = ta.attn_fwd_jvp(*(g[n] for n in names), causal=causal, with_tlse=True)
    assert ta.sync_status() == "TA_OK"
    O, L, tO = oracle.attention_jvp_bhsd(*(cpu[n] for n in names), causal)
    tL = oracle.attention_jvp_tl_bhsd(cpu["q"], cpu["k"], cpu["tq"], cpu["tk"], causal)
    compare("O", o, O, o_tol(dtype))
    compare("L", lse, L, TOL["L"])
    compare("tO", to, tO, TOL["tO"])
    compare("tL", tlse, tL, TOL["tO"])


PW_CASES = [
    # B, H, M, N, D, dtype, causal, w
    (1, 2, 256, 256, 64, "bf16", True, 100),
    (1, 2, 384, 384, 64, "f16", False, 128),
    (1, 1, 256, 256, 64, "bf16", True, 0),
    (1, 1, 256, 256, 64, "bf16", False, -50),
    (1, 1, 256, 256, 64, "bf16", True, 10000),
    (1, 1, 256, 256, 64, "f16", True, -10000),
    (1, 2, 200, 333, 64, "bf16", True, 77),
    (1, 2, 333, 200, 64, "f16", True, 64),
    (1, 1, 512, 512, 128, "bf16", True, 256),  # D = 128: the one-pass key side with 64-query steps
    (1, 2, 300, 333, 128, "f16", False, 40),
    (1, 1, 384, 256, 128, "bf16", True, 0),
    (1, 2, 256, 256, 32, "bf16", True, 60),
    (1, 1, 200, 200, 16, "f16", True, 33),
]


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal,w", PW_CASES)
def test_piecewise_small(gpu_lib, B, H, M, N, D, dtype, causal, w):
    ta = gpu_lib
    names = ("q1", "k1", "q2", "k2", "v", "do")
    cpu, g = inputs(B, H, M, N, D, dtype, 14, names)
    o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w, causal)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.piecewise_fwd_bhsd(cpu["q1"], cpu["k1"], cpu["q2"], cpu["k2"], cpu["v"], causal, None, w)
    compare("O", o, O, o_tol(dtype))
    compare("L", lse, L, TOL["L"])
    grads = ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], w, causal)
    assert ta.sync_status() == "TA_OK"
    ref = oracle.piecewise_bwd_bhsd(cpu["q1"], cpu["k1"], cpu["q2"], cpu["k2"], cpu["v"], cpu["do"], causal,
                                    None, w)
    for name, got, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), grads, ref):
        compare(name, got, r, TOL["grad"])


# ------------------------------------------------------- benchmark workloads
def _fwdbwd_workload(ta, B, H, M, N, D, dtype, causal, workload, heads):
    cpu, g = inputs(B, H, M, N, D, dtype, workload, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.attention_fwd_bhsd(cpu["q"], cpu["k"], cpu["v"], causal, heads=heads)
    dQ, dK, dV = oracle.attention_bwd_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["do"], causal, heads=heads)
    compare("O", heads_of(o, heads), heads_of(O, heads), o_tol(dtype))
    compare("L", heads_of(lse, heads), heads_of(L, heads), TOL["L"])
    for name, got, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        compare(name, heads_of(got, heads), heads_of(ref, heads), TOL["grad"])


def test_workload1_fwd_bwd_fp16_noncausal(gpu_lib):
    """B=1 H=2 M=N=128 D=64 fp16, non-causal: every element."""
    _fwdbwd_workload(gpu_lib, 1, 2, 128, 128, 64, "f16", False, 1, all_heads(1, 2))


def test_workload2_fwd_bwd_bf16_causal(gpu_lib):
    """B=4 H=16 M=N=2048 D=128 bf16 causal: three whole heads."""
    _fwdbwd_workload(gpu_lib, 4, 16, 2048, 2048, 128, "bf16", True, 2, [(0, 0), (1, 7), (3, 15)])


def test_workload3_fwd_bwd_bf16_causal_long(gpu_lib):
    """B=1 H=32 M=N=8192 D=128 bf16 causal (the benchmark workload): first and last heads."""
    _fwdbwd_workload(gpu_lib, 1, 32, 8192, 8192, 128, "bf16", True, 3, [(0, 0), (0, 31)])


@pytest.mark.parametrize("causal", [False, True])
def test_workload4_jvp_fp16(gpu_lib, causal):
    """B=2 H=8 M=N=1024 D=64 fp16 forward + JVP: every head."""
    ta = gpu_lib
    names = ("q", "k", "v", "tq", "tk", "tv")
    cpu, g = inputs(2, 8, 1024, 1024, 64, "f16", 4, names)
    o, lse, to = ta.attn_fwd_jvp(*(g[n] for n in names), causal=causal)
    assert ta.sync_status() == "TA_OK"
    O, L, tO = oracle.attention_jvp_bhsd(*(cpu[n] for n in names), causal)
    compare("O", o, O, TOL["O_f16"])
    compare("L", lse, L, TOL["L"])
    compare("tO", to, tO, TOL["tO"])


def test_workload5_piecewise_bf16_causal(gpu_lib):
    """B=2 H=16 M=N=4096 D=64 bf16 causal piecewise, w=512: three whole heads."""
    ta = gpu_lib
    names = ("q1", "k1", "q2", "k2", "v", "do")
    cpu, g = inputs(2, 16, 4096, 4096, 64, "bf16", 5, names)
    heads = [(0, 0), (1, 5), (1, 15)]
    o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], 512, True)
    grads = ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], 512, True)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.piecewise_fwd_bhsd(*(cpu[n] for n in names[:5]), True, None, 512, heads=heads)
    ref = oracle.piecewise_bwd_bhsd(*(cpu[n] for n in names), True, None, 512, heads=heads)
    compare("O", heads_of(o, heads), heads_of(O, heads), TOL["O_bf16"])
    compare("L", heads_of(lse, heads), heads_of(L, heads), TOL["L"])
    for name, got, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), grads, ref):
        compare(name, heads_of(got, heads), heads_of(r, heads), TOL["grad"])


def test_long_sequence_sampled_rows(gpu_lib):
    """M = N = 32768 (B = H = 1, D = 128, bf16, causal): sampled query rows of O, L, dQ."""
    ta = gpu_lib
    M = 32768
    cpu, g = inputs(1, 1, M, M, 128, "bf16", 21, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    assert ta.sync_status() == "TA_OK"
    rows = np.array([0, 1, 127, 128, 4095, 16384, 32766, 32767])
    O, L, dQ = oracle.attention_rows(cpu["q"][0, 0], cpu["k"][0, 0], cpu["v"][0, 0], cpu["do"][0, 0], rows, True)
    compare("O", o[0, 0, rows], O, TOL["O_bf16"])
    compare("L", lse[0, 0, rows], L, TOL["L"])
    compare("dQ", dq[0, 0, rows], dQ, TOL["grad"])
    assert torch.isfinite(dk).all() and torch.isfinite(dv).all()


# ------------------------------------------------------------- edge cases
def test_empty_inputs(gpu_lib):
    ta = gpu_lib
    dev = "cuda"
    z = torch.empty(0, 2, 128, 64, device=dev, dtype=torch.float16)
    o, lse = ta.attn_fwd(z, z, z)
    assert o.numel() == 0
    # M = 0: no output rows; backward writes dK = dV = 0
    q0 = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    k = torch.randn(1, 2, 130, 64, device=dev, dtype=torch.bfloat16)
    o, lse = ta.attn_fwd(q0, k, k)
    dq, dk, dv = ta.attn_bwd(q0, k, k, o, lse, q0)
    assert ta.sync_status() == "TA_OK"
    assert torch.all(dk == 0) and torch.all(dv == 0)
    # N = 0: every row sees no key -> O = 0, L = -inf, dQ = 0
    q = torch.randn(1, 2, 70, 64, device=dev, dtype=torch.bfloat16)
    k0 = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    o, lse = ta.attn_fwd(q, k0, k0)
    dq, dk, dv = ta.attn_bwd(q, k0, k0, o, lse, q)
    assert ta.sync_status() == "TA_OK"
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse)) and torch.all(dq == 0)


def test_bounded_wait_times_out_and_context_survives(gpu_lib):
    ta = gpu_lib
    assert ta.selftest_wait_timeout(20) == "TA_ERR_TIMEOUT"
    assert ta.sync_status() == "TA_OK"  # the word was cleared; the context still works
    _fwd_check(1, 1, 128, 128, 64, "f16", False, workload=31)


# ---------------------------------------------------------------- fp32 mode
F32_TOL = 1e-4


@pytest.mark.parametrize("B,H,M,N,D,causal", [(1, 2, 128, 128, 64, False), (1, 2, 200, 333, 128, True),
                                              (1, 1, 333, 200, 64, True), (2, 1, 96, 96, 128, False),
                                              (1, 2, 150, 150, 32, True), (1, 1, 100, 170, 16, False)])
def test_fp32_mode_fwd_bwd_jvp(gpu_lib, B, H, M, N, D, causal):
    ta = gpu_lib
    names = ("q", "k", "v", "do", "tq", "tk", "tv")
    cpu = {}
    for idx, n in enumerate(names):
        import synth_inputs as si
        rows = M if n in ("q", "do", "tq") else N
        cpu[n] = si.randn((B, H, rows, D), "f32", si.seed_for(15, idx))
    g = {n: t.cuda() for n, t in cpu.items()}
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    o2, lse2, to, tlse = ta.attn_fwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], causal=causal,
                                         with_tlse=True)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.attention_fwd_bhsd(cpu["q"], cpu["k"], cpu["v"], causal)
    dQ, dK, dV = oracle.attention_bwd_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["do"], causal)
    _, _, tO = oracle.attention_jvp_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["tq"], cpu["tk"], cpu["tv"], causal)
    tL = oracle.attention_jvp_tl_bhsd(cpu["q"], cpu["k"], cpu["tq"], cpu["tk"], causal)
    for name, got, ref in (("O", o, O), ("L", lse, L), ("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV),
                           ("O(jvp)", o2, O), ("tO", to, tO), ("tL", tlse, tL)):
        compare(name, got, ref, F32_TOL)


@pytest.mark.parametrize("D,w", [(64, 100), (128, 40), (64, -20), (32, 0), (16, 50)])
def test_fp32_mode_piecewise(gpu_lib, D, w):
    import synth_inputs as si
    ta = gpu_lib
    B, H, M, N = 1, 2, 256, 256
    names = ("q1", "k1", "q2", "k2", "v", "do")
    cpu = {n: si.randn((B, H, M if n in ("q1", "q2", "do") else N, D), "f32", si.seed_for(16, i))
           for i, n in enumerate(names)}
    g = {n: t.cuda() for n, t in cpu.items()}
    o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w, True)
    grads = ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], w, True)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.piecewise_fwd_bhsd(*(cpu[n] for n in names[:5]), True, None, w)
    ref = oracle.piecewise_bwd_bhsd(*(cpu[n] for n in names), True, None, w)
    compare("O", o, O, F32_TOL)
    compare("L", lse, L, F32_TOL)
    for name, got, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), grads, ref):
        compare(name, got, r, F32_TOL)


# ------------------------------------------------------- wide score range
@pytest.mark.parametrize("M,N,D,dtype,causal,scale", [(512, 512, 128, "bf16", True, 1.0),
                                                      (384, 640, 64, "f16", False, 2.0),
                                                      (300, 300, 64, "bf16", True, 2.0)])
def test_large_scores_exercise_the_rescale(gpu_lib, M, N, D, dtype, causal, scale):
    """sm_scale 1 or 2 instead of 1/sqrt(D): scores spread over ~10-20 units,
    so the running maximum rises by more than 2^8 across key tiles again and
    again and the O correction runs (the lazy-rescale reading).  The forward
    outputs O and L are held element by element to the tolerance plus their
    own 16-bit rounding.  The gradients grow with the scores (|dQ| ~ 50 here)
    and carry the rounding of the 16-bit MMA operands P and dS at that size,
    so they are held to the scaled tolerance plus two roundings of the
    largest value (bf16 meets ~1.7 u of it); tO gets a per-element bound from
    the terms it is the difference of."""
    from _parity import ROUND_U
    ta = gpu_lib
    names = ("q", "k", "v", "do", "tq", "tk", "tv")
    cpu, g = inputs(1, 2, M, N, D, dtype, 91, names)
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal, scale)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal, scale)
    o2, lse2, to = ta.attn_fwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], causal, scale)
    assert ta.sync_status() == "TA_OK"
    u = ROUND_U[dtype]
    O, L = oracle.attention_fwd_bhsd(cpu["q"], cpu["k"], cpu["v"], causal, scale)
    compare("O", o, O, o_tol(dtype), u)
    compare("L", lse, L, TOL["L"] * scale * 4)  # L scales with the scores; fp32 at |L| ~ 100
    for name, got, r in zip(("dQ", "dK", "dV"), (dq, dk, dv),
                            oracle.attention_bwd_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["do"], causal, scale)):
        compare(name, got, r, TOL["grad"] * scale + 2 * u * float(np.abs(r).max()))
    _, _, tO = oracle.attention_jvp_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["tq"], cpu["tk"], cpu["tv"], causal,
                                         scale)
    compare("O(jvp)", o2, O, o_tol(dtype), u)
    # tO = (P o T) V - mu O + P tV is a difference of two large terms; each
    # carries ~u of its own size (P o T and P rounded before their products),
    # so the bound is taken element by element from those terms
    keep = oracle.allowed_mask(M, N, causal)
    got = to.float().cpu().double().numpy()
    for h in range(2):
        q, k, v, tq, tk = (cpu[n][0, h].double().numpy() for n in ("q", "k", "v", "tq", "tk"))
        S = np.where(keep, scale * q @ k.T, -np.inf)
        P = np.exp(S - L[0, h][:, None])
        T = np.where(keep, scale * (tq @ k.T + q @ tk.T), 0.0)
        mu = (P * T).sum(axis=1)
        tv = cpu["tv"][0, h].double().numpy()
        bound = TOL["tO"] + 2 * u * ((P * np.abs(T)) @ np.abs(v) + np.abs(mu)[:, None] * np.abs(O[0, h])
                                     + P @ np.abs(tv))
        err = np.abs(got[0, h] - tO[0, h])
        assert np.all(err <= bound), f"tO: head {h} exceeds its bound by {np.max(err - bound):.3e}"
