"""Closed forms checked on every element at the benchmark's full size, in the
launch configuration the benchmark times (B=1, H=32, M=N=8192, D=128, bf16,
causal), and at the same size non-causal and in fp16 at D = 64.

With q = 0 every visible score is 0, so row i attends uniformly to its n_i
visible keys (n_i = i + 1 causal, N otherwise; the softmax of a constant
row):
  O_i = (sum of the visible v_j) / n_i,   L_i = ln n_i,
and the backward gives dV_j = sum_{i sees j} dO_i / n_i (P^T dO with
P_ij = 1/n_i) and dK = s dS^T Q = 0 exactly.  With also tq = tk = 0 the
JVP's tangent score T is 0, so mu = tL = 0 exactly and tO_i is the same
running mean of tv.  These hold at any size, so they reach every row of
every head, where the oracle can only sample; dQ is compared with the
oracle's row-restricted definition on rows of two heads."""
import numpy as np
import pytest
import torch

import oracle
from _parity import ROUND_U, TOL, compare, inputs

pytestmark = pytest.mark.gpu

B, H, S = 1, 32, 8192


def _uniform(x, causal):
    """Row i of the result: the mean of x over row i's visible keys."""
    if causal:
        return x.cumsum(2) / torch.arange(1, S + 1, dtype=torch.float64)[:, None]
    return (x.sum(2, keepdim=True) / S).expand_as(x)


@pytest.mark.parametrize("causal,dtype,D", [(True, "bf16", 128), (False, "bf16", 128), (True, "f16", 64)])
def test_uniform_attention_every_element_full_size(gpu_lib, causal, dtype, D):
    ta = gpu_lib
    cpu, g = inputs(B, H, S, S, D, dtype, 89, ("k", "v", "do", "tv"))
    q = torch.zeros_like(g["k"])
    o, lse = ta.attn_fwd(q, g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd(q, g["k"], g["v"], o, lse, g["do"], causal)
    o2, lse2, to, tlse = ta.attn_fwd_jvp(q, g["k"], g["v"], q, q, g["tv"], causal=causal, with_tlse=True)
    assert ta.sync_status() == "TA_OK"

    u = ROUND_U[dtype]
    n = np.arange(1, S + 1, dtype=np.float64) if causal else np.full(S, float(S))
    O = _uniform(cpu["v"].double(), causal).numpy()
    L = np.broadcast_to(np.log(n), (B, H, S))
    # p = 2^0 = 1 for every visible key, so the weights are exact: fp32 sums
    # and one rounding of the stored result
    compare("O", o, O, 1e-5, u)
    compare("L", lse, L, 1e-5)
    compare("O(jvp)", o2, O, 1e-5, u)
    compare("L(jvp)", lse2, L, 1e-5)
    w = cpu["do"].double() / torch.from_numpy(n)[:, None]
    dV = (w.flip(2).cumsum(2).flip(2) if causal else w.sum(2, keepdim=True).expand_as(w)).numpy()
    compare("dV", dv, dV, TOL["grad"], u)
    assert torch.all(dk == 0), "dK must be exactly 0 when q = 0"
    tO = _uniform(cpu["tv"].double(), causal).numpy()
    compare("tO", to, tO, 1e-5, u)
    assert torch.all(tlse == 0), "tL must be exactly 0 when tq = tk = 0"
    rows = [0, 1, 127, 128, 129, 4095, 8190, 8191]
    for h in (0, H - 1):
        _, _, dQr = oracle.attention_rows(np.zeros((S, D)), cpu["k"][0, h], cpu["v"][0, h], cpu["do"][0, h], rows,
                                          causal)
        compare(f"dQ rows [head {h}]", dq[0, h, rows], dQr, TOL["grad"])


def test_piecewise_uniform_every_element_full_size(gpu_lib):
    """The piecewise workload's shape (B=2, H=16, M=N=4096, D=64, bf16,
    causal, w=512) with q1 = q2 = 0: the near and the far scores are both 0,
    so the closed forms above hold whatever the threshold, dk1 = dk2 = 0
    exactly, and dq1 / dq2 split dQ by distance (rows of two heads against
    the oracle)."""
    ta = gpu_lib
    Bp, Hp, Sp, Dp, w = 2, 16, 4096, 64, 512
    cpu, g = inputs(Bp, Hp, Sp, Sp, Dp, "bf16", 88, ("k1", "k2", "v", "do"))
    q = torch.zeros_like(g["k1"])
    o, lse = ta.piecewise_fwd(q, g["k1"], q, g["k2"], g["v"], w, True)
    dq1, dk1, dq2, dk2, dv = ta.piecewise_bwd(q, g["k1"], q, g["k2"], g["v"], o, lse, g["do"], w, True)
    assert ta.sync_status() == "TA_OK"
    u = ROUND_U["bf16"]
    n = torch.arange(1, Sp + 1, dtype=torch.float64)[:, None]
    compare("O", o, (cpu["v"].double().cumsum(2) / n).numpy(), 1e-5, u)
    compare("L", lse, np.broadcast_to(np.log(n[:, 0].numpy()), (Bp, Hp, Sp)), 1e-5)
    compare("dv", dv, (cpu["do"].double() / n).flip(2).cumsum(2).flip(2).numpy(), TOL["grad"], u)
    assert torch.all(dk1 == 0) and torch.all(dk2 == 0), "dk1, dk2 must be exactly 0 when q1 = q2 = 0"
    rows = [0, 511, 512, 513, 2047, 4095]
    zero = np.zeros((Sp, Dp))
    for b, h in ((0, 0), (Bp - 1, Hp - 1)):
        x = [zero, cpu["k1"][b, h], zero, cpu["k2"][b, h], cpu["v"][b, h], cpu["do"][b, h]]
        ref = oracle.piecewise_bwd(*x, True, None, w)
        compare(f"dq1 rows [{b},{h}]", dq1[b, h, rows], ref[0][rows], TOL["grad"])
        compare(f"dq2 rows [{b},{h}]", dq2[b, h, rows], ref[2][rows], TOL["grad"])


def test_fp8_forward_uniform_every_element_full_size(gpu_lib):
    """The e5m2 forward at the benchmark size (B=1, H=32, M=N=8192, D=128,
    causal) with q = 0: P = 1 is exact in e5m2, so O is the running mean of v
    up to the fp32 sums and the output's e5m2 rounding, and L = ln(i + 1)."""
    import synth_inputs as si
    ta = gpu_lib
    v = si.randn((B, H, S, 128), "e5m2", si.seed_for(87, 0))
    k = si.randn((B, H, S, 128), "e5m2", si.seed_for(87, 1))
    q = torch.zeros(B, H, S, 128, dtype=torch.uint8).view(torch.float8_e5m2)
    vt = v.view(torch.uint8).transpose(-1, -2).contiguous().view(torch.float8_e5m2)
    o, lse = ta.attn_fwd_fp8(q.cuda(), k.cuda(), vt.cuda(), True)
    assert ta.sync_status() == "TA_OK"
    n = torch.arange(1, S + 1, dtype=torch.float64)[:, None]
    O = (v.to(torch.float64).cumsum(2) / n).numpy()
    got = o.cpu().to(torch.float64).numpy()
    # one e5m2 rounding: 2^-3 relative, or half the subnormal spacing 2^-16
    # below the smallest normal 2^-14
    assert np.all(np.abs(got - O) <= 2.0 ** -3 * np.abs(O) + 2.0 ** -17), "O outside one e5m2 rounding of the mean"
    compare("L", lse, np.broadcast_to(np.log(n[:, 0].numpy()), (B, H, S)), 1e-5)


def test_merge_equal_lse_every_element_full_size(gpu_lib):
    """The merge at the benchmark's state size (B=1, H=32, M=8192, D=128,
    bf16): two states with equal L merge to O = (O1 + O2)/2 and L + ln 2,
    and with dL = 0 the backward gives dO1 = dO2 = dO/2 and dL1 = -dL2 =
    <dO, O1 - O2>/4; rows where both parts saw no key stay O = 0, L = -inf."""
    import synth_inputs as si
    ta = gpu_lib
    o1, o2, do = (si.randn((B, H, S, 128), "bf16", si.seed_for(86, i)) for i in range(3))
    lse = si.randn((B, H, S), "f32", si.seed_for(86, 3)) * 3
    lse[..., 5] = -float("inf")
    o1[..., 5, :] = 0
    o2[..., 5, :] = 0
    g = [t.cuda() for t in (o1, lse, o2, lse, do)]
    mo, ml = ta.merge_fwd(*g[:4])
    d1, l1, d2, l2 = ta.merge_bwd(*g, None)
    assert ta.sync_status() == "TA_OK"
    u = ROUND_U["bf16"]
    a, b, dd = (t.double() for t in (o1, o2, do))
    # the weights 1/2 come from exp(l - L) in fp32 (relative error ~2^-22),
    # then one rounding of the stored result
    compare("O", mo, ((a + b) / 2).numpy(), 1e-5, u)
    compare("L", ml, (lse.double() + np.log(2.0)).numpy(), 1e-5)
    half = (dd / 2).numpy()
    half[..., 5, :] = 0
    compare("dO1", d1, half, 1e-5, u)
    compare("dO2", d2, half, 1e-5, u)
    t = ((dd * (a - b)).sum(-1) / 4).numpy()
    t[..., 5] = 0
    compare("dL1", l1, t, 1e-4, 2.0 ** -20)
    compare("dL2", l2, -t, 1e-4, 2.0 ** -20)
