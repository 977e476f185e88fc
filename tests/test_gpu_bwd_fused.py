"""GPU parity of attn_bwd_fused, the one-pass five-matmul backward (D = 128):
dq, dk, dv against the fp64 oracle on the same seeded inputs, every head of
the small cases (ragged M and N, M > N with rows that see no key, causal and
not, both 16-bit types) and whole sampled heads of the benchmark workloads;
plus the two properties the fp32 dQ accumulator must keep: a second call
gives dq equal up to the last place (the atomics' order varies) and
bit-identical dk, dv, and the result matches attn_bwd within the gradients'
tolerance."""
import pytest
import torch

import oracle
from _parity import TOL, assert_same_up_to_summation_order, compare, heads_of, inputs

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, M, N, dtype, causal
    (1, 2, 64, 64, "bf16", True),
    (2, 3, 256, 256, "bf16", True),
    (1, 2, 384, 384, "f16", False),
    (1, 2, 200, 333, "bf16", True),
    (1, 2, 333, 200, "bf16", True),   # M > N: the first rows see no key
    (1, 1, 1, 1, "f16", True),
    (1, 1, 5, 700, "bf16", False),
    (1, 1, 700, 5, "f16", False),
    (2, 1, 129, 257, "bf16", True),
    (1, 1, 1000, 1000, "f16", True),
]


@pytest.mark.parametrize("B,H,M,N,dtype,causal", CASES)
def test_fused_bwd_small(gpu_lib, B, H, M, N, dtype, causal):
    ta = gpu_lib
    cpu, g = inputs(B, H, M, N, 128, dtype, 15, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd_fused(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    assert ta.sync_status() == "TA_OK"
    dQ, dK, dV = oracle.attention_bwd_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["do"], causal)
    compare("dQ", dq, dQ, TOL["grad"])
    compare("dK", dk, dK, TOL["grad"])
    compare("dV", dv, dV, TOL["grad"])


def test_fused_bwd_repeat_and_two_pass_agree(gpu_lib):
    ta = gpu_lib
    cpu, g = inputs(2, 4, 640, 640, 128, "bf16", 16, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True)
    a = [t.clone() for t in ta.attn_bwd_fused(g["q"], g["k"], g["v"], o, lse, g["do"], True)]
    b = ta.attn_bwd_fused(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    ref = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    assert ta.sync_status() == "TA_OK"
    assert_same_up_to_summation_order("dq (second call)", b[0], a[0])
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
    for name, x, y in zip(("dq", "dk", "dv"), a, ref):
        compare(name + " vs attn_bwd", x, y.double().cpu().numpy(), TOL["grad"])


@pytest.mark.parametrize("B,H,S,workload,heads", [
    (4, 16, 2048, 2, [(0, 0), (1, 7), (3, 15)]),
    (1, 32, 8192, 3, [(0, 0), (0, 31)]),
])
def test_fused_bwd_workloads(gpu_lib, B, H, S, workload, heads):
    """The bf16 causal benchmark workloads (B4 H16 S2048, B1 H32 S8192), in
    the launch configuration the benchmark times: whole sampled heads."""
    ta = gpu_lib
    cpu, g = inputs(B, H, S, S, 128, "bf16", workload, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True)
    dq, dk, dv = ta.attn_bwd_fused(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    assert ta.sync_status() == "TA_OK"
    dQ, dK, dV = oracle.attention_bwd_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["do"], True, heads=heads)
    for name, got, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV)):
        compare(name, heads_of(got, heads), heads_of(ref, heads), TOL["grad"])


def test_fused_bwd_refuses_other_head_sizes(gpu_lib):
    ta = gpu_lib
    cpu, g = inputs(1, 1, 128, 128, 64, "bf16", 17, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True)
    with pytest.raises(ta.TAError) as e:
        ta.attn_bwd_fused(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    assert e.value.status == "TA_ERR_UNSUPPORTED"
