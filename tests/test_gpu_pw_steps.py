"""The piecewise backward at D = 128 (16-bit): the key side runs in one pass
with 64-query steps (dV, dK1 and dK2 together, csrc/bwd_pw_steps.cu).  Every
gradient is compared with the fp64 oracle at the gradient tolerance on
shapes chosen for the step classes: steps wholly near, wholly far and
straddling the distance w (small and large w, negative w, w past every
distance), ragged M and N, M > N (queries that see no key), a key tile no
query reaches, fp16 and bf16, causal and not."""
import pytest

import oracle
from _parity import TOL, compare, inputs, o_tol

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, M, N, D, dtype, causal, w
    (1, 2, 512, 512, 128, "bf16", True, 100),     # straddling steps near the diagonal band's edge
    (1, 1, 640, 640, 128, "f16", True, 1),        # w = 1: almost every step far
    (1, 1, 384, 384, 128, "bf16", False, -50),    # negative w: every pair far
    (1, 1, 300, 700, 128, "bf16", False, 10000),  # every pair near
    (2, 1, 200, 333, 128, "f16", True, 77),       # ragged, N > M
    (1, 1, 333, 200, 128, "bf16", True, 64),      # M > N: the first rows see no key
    (1, 2, 130, 900, 128, "f16", True, 300),      # few queries, many keys: key tiles no query reaches
    (1, 1, 1024, 1024, 128, "bf16", True, 512),   # the benchmark's w on a longer sequence
]


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal,w", CASES)
def test_piecewise_backward_d128_one_pass(gpu_lib, B, H, M, N, D, dtype, causal, w):
    ta = gpu_lib
    names = ("q1", "k1", "q2", "k2", "v", "do")
    cpu, g = inputs(B, H, M, N, D, dtype, 93, names)
    o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w, causal)
    grads = ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], w, causal)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.piecewise_fwd_bhsd(*(cpu[n] for n in names[:5]), causal, None, w)
    compare("O", o, O, o_tol(dtype))
    compare("L", lse, L, TOL["L"])
    ref = oracle.piecewise_bwd_bhsd(*(cpu[n] for n in names), causal, None, w)
    for name, got, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), grads, ref):
        compare(name, got, r, TOL["grad"])
