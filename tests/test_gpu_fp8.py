"""GPU parity of the e5m2 forward (attn_fwd_fp8) against the fp64 oracle.

The oracle runs on the exact e5m2 values the GPU reads.  The kernel then
differs from it only by two roundings to e5m2 (2 mantissa bits, unit roundoff
u = 2^-3): P before the P V product and O on output; L is formed from the
unrounded fp32 P.  So, element by element,
    |O_gpu - O| <= u (1 + u) (P |V|) + u |O|,
with P the oracle's probabilities, and |L_gpu - L| stays at fp32 level.  The
mean error must also be far below that worst case, which assumes every
rounding goes the same way."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si

pytestmark = pytest.mark.gpu

U = 2.0 ** -3


def _run(ta, B, H, M, N, D, causal, workload):
    q = si.randn((B, H, M, D), "e5m2", si.seed_for(workload, 0))
    k = si.randn((B, H, N, D), "e5m2", si.seed_for(workload, 1))
    v = si.randn((B, H, N, D), "e5m2", si.seed_for(workload, 2))
    vt = v.transpose(-1, -2).contiguous()
    o, lse = ta.attn_fwd_fp8(q.cuda(), k.cuda(), vt.cuda(), causal)
    assert ta.sync_status() == "TA_OK"
    return q, k, v, o.cpu().to(torch.float64).numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("B,H,M,N,D,causal", [(1, 2, 256, 256, 128, True), (1, 2, 384, 384, 64, False),
                                              (2, 1, 200, 336, 128, True), (1, 1, 333, 208, 64, True),
                                              (1, 1, 130, 96, 128, False)])
def test_fp8_forward_within_e5m2_rounding_bound(gpu_lib, B, H, M, N, D, causal):
    q, k, v, o, lse = _run(gpu_lib, B, H, M, N, D, causal, 51)
    s = oracle.default_scale(D)
    qf, kf, vf = (t.to(torch.float64).numpy() for t in (q, k, v))
    for b in range(B):
        for h in range(H):
            O, L = oracle.attention_fwd(qf[b, h], kf[b, h], vf[b, h], causal)
            keep = oracle.allowed_mask(M, N, causal)
            S = np.where(keep, s * qf[b, h] @ kf[b, h].T, -np.inf)
            fin = np.isfinite(L)
            P = np.zeros_like(S)
            P[fin] = np.exp(S[fin] - L[fin, None])
            bound = U * (1 + U) * (P @ np.abs(vf[b, h])) + U * np.abs(O) + 1e-6
            err = np.abs(o[b, h] - O)
            assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e} at head {(b, h)}"
            assert err.mean() < 0.03, err.mean()
            np.testing.assert_array_equal(np.isneginf(lse[b, h]), ~fin)
            np.testing.assert_allclose(lse[b, h][fin], L[fin], atol=1e-3)
            assert np.all(o[b, h][~fin] == 0)


def test_fp8_rejects_unsupported_shapes(gpu_lib):
    ta = gpu_lib
    f8 = torch.float8_e5m2
    q = torch.zeros(1, 1, 128, 64, device="cuda", dtype=f8)
    k = torch.zeros(1, 1, 100, 64, device="cuda", dtype=f8)  # N not a multiple of 16
    vt = torch.zeros(1, 1, 64, 100, device="cuda", dtype=f8)
    with pytest.raises(ta.TAError):
        ta.attn_fwd_fp8(q, k, vt)
    q32 = torch.zeros(1, 1, 128, 32, device="cuda", dtype=f8)
    k32 = torch.zeros(1, 1, 128, 32, device="cuda", dtype=f8)
    with pytest.raises(ta.TAError):
        ta.attn_fwd_fp8(q32, k32, torch.zeros(1, 1, 32, 128, device="cuda", dtype=f8))


def test_fp8_forward_benchmark_shape_sampled_heads(gpu_lib):
    """B1 H32 M=N=8192 D128 causal, the shape and launch bench.py times:
    first and last heads against the rounding bound."""
    B, H, M, D = 1, 32, 8192, 128
    q, k, v, o, lse = _run(gpu_lib, B, H, M, M, D, True, 52)
    s = oracle.default_scale(D)
    keep = oracle.allowed_mask(M, M, True)
    for h in (0, H - 1):
        qf, kf, vf = (t[0, h].to(torch.float64).numpy() for t in (q, k, v))
        O, L = oracle.attention_fwd(qf, kf, vf, True)
        S = np.where(keep, s * qf @ kf.T, -np.inf)
        P = np.exp(S - L[:, None])
        bound = U * (1 + U) * (P @ np.abs(vf)) + U * np.abs(O) + 1e-6
        err = np.abs(o[0, h] - O)
        assert np.all(err <= bound), f"max excess {np.max(err - bound):.3e} at head {h}"
        assert err.mean() < 0.03, err.mean()
        np.testing.assert_allclose(lse[0, h], L, atol=1e-3)
