"""GPU parity with tensors of more than 2^31 elements: B=1, H=66000,
M=N=256, D=128 bf16 (2.16e9 elements, 4.3 GB per tensor, about 35 GB on the
device in all), causal and not, so the forward, delta, dK/dV and dQ kernels
all form element offsets past 2^31.

The heads repeat a block of 61 distinct seeded heads.  A 32-bit wrap of an
element offset would move an access by 2^31 elements = 65536 heads, which 61
does not divide, so an aliased read or write would meet another head's data
and show as a mismatch.  Head 65536 starts exactly at element 2^31; heads on
both sides of that boundary are compared with the oracle."""
import pytest
import torch

import oracle
from _parity import ROUND_U, TOL, compare, inputs, o_tol

pytestmark = pytest.mark.gpu

H, S, D, PERIOD = 66000, 256, 128, 61
CHECK = (0, 60, 65535, 65536, 65537, 65999)
NAMES = ("q", "k", "v", "do")


def _tile_heads(x):
    """[1, PERIOD, S, D] -> [1, H, S, D]: head h holds block head h % PERIOD."""
    reps = (H + PERIOD - 1) // PERIOD
    return x.repeat(1, reps, 1, 1)[:, :H].contiguous()


@pytest.mark.parametrize("causal", [False, True])
def test_more_than_2_31_elements(gpu_lib, causal):
    ta = gpu_lib
    free, _ = torch.cuda.mem_get_info()
    if free < (48 << 30):
        pytest.skip("needs about 40 GB of free device memory")
    cpu, blk = inputs(1, PERIOD, S, S, D, "bf16", 97, NAMES)
    g = {n: _tile_heads(t) for n, t in blk.items()}
    del blk
    assert g["q"].numel() > 2 ** 31 and g["q"].shape == (1, H, S, D)
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    assert ta.sync_status() == "TA_OK"
    u = ROUND_U["bf16"]
    for h in CHECK:
        x = [cpu[n][0, h % PERIOD] for n in NAMES]
        O, L = oracle.attention_fwd(x[0], x[1], x[2], causal)
        compare(f"O[{h}]", o[0, h], O, o_tol("bf16"), u)
        compare(f"L[{h}]", lse[0, h], L, TOL["L"])
        for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), oracle.attention_bwd(*x, causal)):
            compare(f"{name}[{h}]", got[0, h], ref, TOL["grad"], u)
    del g, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


def test_merge_more_than_2_31_elements(gpu_lib):
    """The two-state merge and its backward over the same tiled shape: two
    seeded partial states (O ~ N(0,1) bf16, L ~ 3 N(0,1)) and their cotangents,
    checked per head against the oracle on both sides of element 2^31."""
    import synth_inputs as si
    ta = gpu_lib
    free, _ = torch.cuda.mem_get_info()
    if free < (48 << 30):
        pytest.skip("needs about 40 GB of free device memory")
    blk = [si.randn((1, PERIOD, S, D), "bf16", si.seed_for(98, 0)),
           si.randn((1, PERIOD, S), "f32", si.seed_for(98, 1)) * 3,
           si.randn((1, PERIOD, S, D), "bf16", si.seed_for(98, 2)),
           si.randn((1, PERIOD, S), "f32", si.seed_for(98, 3)) * 3,
           si.randn((1, PERIOD, S, D), "bf16", si.seed_for(98, 4)),
           si.randn((1, PERIOD, S), "f32", si.seed_for(98, 5))]
    reps = (H + PERIOD - 1) // PERIOD
    g = [t.cuda().repeat((1, reps) + (1,) * (t.dim() - 2))[:, :H].contiguous() for t in blk]
    assert g[0].numel() > 2 ** 31
    o, lse = ta.merge_fwd(g[0], g[1], g[2], g[3])
    grads = ta.merge_bwd(*g)
    assert ta.sync_status() == "TA_OK"
    for h in CHECK:
        x = [t[0, h % PERIOD] for t in blk]
        O, L = oracle.lse_merge_fwd(*x[:4])
        compare(f"merge O[{h}]", o[0, h], O, o_tol("bf16"), ROUND_U["bf16"])
        compare(f"merge L[{h}]", lse[0, h], L, 1e-5)
        for name, got, ref in zip(("dO1", "dL1", "dO2", "dL2"), grads, oracle.lse_merge_bwd(*x)):
            dgrad = name.startswith("dO")
            compare(f"merge {name}[{h}]", got[0, h], ref, TOL["grad"] if dgrad else 1e-4,
                    ROUND_U["bf16"] if dgrad else 2.0 ** -24)
    del g, o, lse, grads
    torch.cuda.empty_cache()
