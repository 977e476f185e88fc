"""GPU parity of the two-state attention merge (split-KV combine) and its
backward, through the C ABI, against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from _parity import TOL, compare, inputs, o_tol

pytestmark = pytest.mark.gpu

DT = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def _states(B, H, M, D, dtype, workload):
    """Two partial states: O1, O2 ~ N(0,1) in dtype, L1, L2 ~ 3 N(0,1) with a
    few rows where one part, or both, saw no key (L = -inf)."""
    o1 = si.randn((B, H, M, D), dtype, si.seed_for(workload, 0))
    o2 = si.randn((B, H, M, D), dtype, si.seed_for(workload, 1))
    l1 = si.randn((B, H, M), "f32", si.seed_for(workload, 2)) * 3
    l2 = si.randn((B, H, M), "f32", si.seed_for(workload, 3)) * 3
    l1[..., 0] = -float("inf")                        # only part 2 saw keys
    l2[..., 1] = -float("inf")                        # only part 1 saw keys
    l1[..., 2] = l2[..., 2] = -float("inf")           # neither part saw a key
    o1[..., 2, :] = 0
    o2[..., 2, :] = 0
    return o1, l1, o2, l2


@pytest.mark.parametrize("B,H,M,D,dtype", [(1, 2, 1000, 128, "bf16"), (2, 1, 333, 64, "f16"),
                                           (1, 3, 257, 16, "bf16"), (1, 1, 129, 32, "f32"),
                                           (2, 2, 77, 128, "f32")])
def test_merge_fwd_bwd(gpu_lib, B, H, M, D, dtype):
    ta = gpu_lib
    o1, l1, o2, l2 = _states(B, H, M, D, dtype, 41)
    do = si.randn((B, H, M, D), dtype, si.seed_for(41, 4))
    dl = si.randn((B, H, M), "f32", si.seed_for(41, 5))
    g = [t.cuda() for t in (o1, l1, o2, l2, do, dl)]
    o, lse = ta.merge_fwd(g[0], g[1], g[2], g[3])
    do1, dl1, do2, dl2 = ta.merge_bwd(g[0], g[1], g[2], g[3], g[4], g[5])
    do1n, dl1n, do2n, dl2n = ta.merge_bwd(g[0], g[1], g[2], g[3], g[4], None)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.lse_merge_fwd_bhsd(o1, l1, o2, l2)
    ref = oracle.lse_merge_bwd_bhsd(o1, l1, o2, l2, do, dl)
    refn = oracle.lse_merge_bwd_bhsd(o1, l1, o2, l2, do, None)
    otol = 1e-5 if dtype == "f32" else o_tol(dtype)
    gtol = 1e-5 if dtype == "f32" else TOL["grad"]
    compare("O", o, O, otol)
    compare("L", lse, L, 1e-5)
    for name, got, r in zip(("dO1", "dL1", "dO2", "dL2"), (do1, dl1, do2, dl2), ref):
        compare(name, got, r, gtol if name.startswith("dO") else 1e-4)
    for name, got, r in zip(("dO1", "dL1", "dO2", "dL2"), (do1n, dl1n, do2n, dl2n), refn):
        compare(name + "(no dL)", got, r, gtol if name.startswith("dO") else 1e-4)
    assert torch.all(o[..., 2, :] == 0) and torch.all(torch.isneginf(lse[..., 2]))


@pytest.mark.parametrize("M,N,split,D,dtype", [(300, 500, 200, 128, "bf16"), (128, 256, 128, 64, "f16"),
                                               (97, 130, 60, 32, "bf16")])
def test_split_kv_attention_merges_to_full_attention(gpu_lib, M, N, split, D, dtype):
    """attn_fwd over keys [0, split) and [split, N), merged with attn_merge_fwd,
    equals attention over all N keys (non-causal)."""
    ta = gpu_lib
    cpu, g = inputs(1, 2, M, N, D, dtype, 42, ("q", "k", "v"))
    k1, k2 = g["k"][:, :, :split].contiguous(), g["k"][:, :, split:].contiguous()
    v1, v2 = g["v"][:, :, :split].contiguous(), g["v"][:, :, split:].contiguous()
    o1, l1 = ta.attn_fwd(g["q"], k1, v1, False)
    o2, l2 = ta.attn_fwd(g["q"], k2, v2, False)
    o, lse = ta.merge_fwd(o1, l1, o2, l2)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.attention_fwd_bhsd(cpu["q"], cpu["k"], cpu["v"], False)
    compare("O", o, O, o_tol(dtype) * 1.5)  # two roundings of the partial outputs plus the merged one
    compare("L", lse, L, TOL["L"])


def test_merge_empty_and_bad_arguments(gpu_lib):
    ta = gpu_lib
    dev = torch.device("cuda")
    e = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    le = torch.empty(1, 2, 0, device=dev, dtype=torch.float32)
    o, lse = ta.merge_fwd(e, le, e, le)
    assert o.shape == e.shape and ta.sync_status() == "TA_OK"
    x = torch.zeros(1, 1, 8, 96, device=dev, dtype=torch.bfloat16)
    lx = torch.zeros(1, 1, 8, device=dev, dtype=torch.float32)
    with pytest.raises(ta.TAError):
        ta.merge_fwd(x, lx, x, lx)  # D = 96 is not supported


def test_merge_benchmark_shape(gpu_lib):
    """B1 H32 M8192 D128 bf16, the shape bench.py times: every element of the
    forward and the backward (with dL)."""
    ta = gpu_lib
    B, H, M, D = 1, 32, 8192, 128
    o1, l1, o2, l2 = _states(B, H, M, D, "bf16", 43)
    do = si.randn((B, H, M, D), "bf16", si.seed_for(43, 4))
    dl = si.randn((B, H, M), "f32", si.seed_for(43, 5))
    g = [t.cuda() for t in (o1, l1, o2, l2, do, dl)]
    o, lse = ta.merge_fwd(g[0], g[1], g[2], g[3])
    grads = ta.merge_bwd(*g)
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.lse_merge_fwd_bhsd(o1, l1, o2, l2)
    compare("O", o, O, o_tol("bf16"))
    compare("L", lse, L, 1e-5)
    for name, got, r in zip(("dO1", "dL1", "dO2", "dL2"), grads, oracle.lse_merge_bwd_bhsd(o1, l1, o2, l2, do, dl)):
        compare(name, got, r, TOL["grad"] if name.startswith("dO") else 1e-4)
