"""Piecewise attention at D = 64 with the distance threshold w moved across
and between 128-row tile edges ("FlagAttention piecewise.py",
_fwd_kernel / _bwd_kv_kernel / _bwd_q_kernel piecewise_mask).

The kernels sort each (query tile, key tile) pair into near, far or
straddling; a straddling pair runs both score products and splits dS by
distance, in the dQ pass (per key tile) and in the dK/dV pass (per query
tile).  These values of w put the boundary on a tile edge, one row to either
side of it and inside tiles, so that the straddling pair is the first, the
last or an inner tile of a CTA, and, non-causal, also at negative distances.
Every output is compared with the oracle."""
import pytest

import oracle
from _parity import TOL, compare, inputs, o_tol

pytestmark = pytest.mark.gpu

W_VALUES = [-300, -128, -127, -1, 1, 127, 128, 129, 255, 256, 383, 511, 640]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("w", W_VALUES)
def test_piecewise_tile_classes(gpu_lib, w, causal):
    ta = gpu_lib
    B, H, M, N, D = 1, 1, 512, 512, 64
    names = ("q1", "k1", "q2", "k2", "v", "do")
    cpu, g = inputs(B, H, M, N, D, "bf16", 120, names)
    o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w, causal)
    grads = ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], w, causal)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.piecewise_fwd_bhsd(cpu["q1"], cpu["k1"], cpu["q2"], cpu["k2"], cpu["v"], causal, None, w)
    compare("O", o, O, o_tol("bf16"))
    compare("L", lse, L, TOL["L"])
    ref = oracle.piecewise_bwd_bhsd(cpu["q1"], cpu["k1"], cpu["q2"], cpu["k2"], cpu["v"], cpu["do"], causal,
                                    None, w)
    for name, got, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), grads, ref):
        compare(name, got, r, TOL["grad"])


@pytest.mark.parametrize("w", [-64, 100, 300])
def test_piecewise_tile_classes_ragged(gpu_lib, w):
    """M > N and M < N with ragged tails (bottom-right causal alignment)."""
    ta = gpu_lib
    names = ("q1", "k1", "q2", "k2", "v", "do")
    for M, N in ((450, 300), (300, 450)):
        cpu, g = inputs(1, 2, M, N, 64, "f16", 121, names)
        o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w, True)
        grads = ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], w, True)
        assert ta.sync_status() == "TA_OK"
        O, L = oracle.piecewise_fwd_bhsd(cpu["q1"], cpu["k1"], cpu["q2"], cpu["k2"], cpu["v"], True, None, w)
        compare("O", o, O, o_tol("f16"))
        compare("L", lse, L, TOL["L"])
        ref = oracle.piecewise_bwd_bhsd(cpu["q1"], cpu["k1"], cpu["q2"], cpu["k2"], cpu["v"], cpu["do"], True,
                                        None, w)
        for name, got, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), grads, ref):
            compare(name, got, r, TOL["grad"])
