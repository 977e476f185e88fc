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
