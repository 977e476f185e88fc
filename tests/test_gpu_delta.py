"""The backward preprocess delta = rowsum(dO o O) that the 16-bit backward
forms inside its dQ pass ("Triton fused attention tutorial, updated with JVP
support", _attn_bwd_preprocess; "FlagAttention piecewise.py",
_bwd_preprocess), read back from the workspace, whose first B*H*M floats hold
it, and compared with the oracle's definition on the same stored O and dO.

O is seeded input here, not a forward's output, so delta is checked on its
own; the rows that see no key get O = 0, as the forward writes them (a query
tile that sees no key stores delta = 0 without reading O).  The shapes cover
ragged M and N, M > N (whole tiles of rows that see no key), a single row and
D = 16 to 128, for attn_bwd and piecewise_bwd."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, M, N, D, dtype, causal
    (1, 2, 200, 333, 64, "f16", True),
    (1, 1, 333, 200, 128, "bf16", True),
    (2, 1, 1, 1, 64, "f16", False),
    (1, 1, 130, 190, 16, "bf16", False),
    (1, 2, 384, 384, 128, "bf16", True),
    (1, 1, 300, 100, 32, "f16", True),
]


def _inputs(B, H, M, N, D, dtype, causal, seed, names):
    cpu = si.attention_inputs(B, H, M, N, D, dtype, seed, names=names)
    o = si.randn((B, H, M, D), dtype, si.seed_for(seed, 50))
    empty = ~oracle.allowed_mask(M, N, causal).any(axis=1)
    o[:, :, torch.from_numpy(empty)] = 0
    cpu["o"] = o
    return cpu, {n: t.cuda() for n, t in cpu.items()}


def _check_delta(ws, cpu, B, H, M):
    got = ws[: B * H * M * 4].view(torch.float32).reshape(B, H, M).double().cpu().numpy()
    ref = oracle.bwd_delta_bhsd(cpu["o"], cpu["do"])
    # fp32 sums of D exact products of 16-bit values: at most D + 1 roundings
    D = cpu["o"].shape[-1]
    mag = np.abs(cpu["o"].double().numpy() * cpu["do"].double().numpy()).sum(axis=-1)
    bound = 1e-7 + (D + 2) * 2.0 ** -24 * mag
    err = np.abs(got - ref)
    assert (err <= bound).all(), f"delta: max error {err.max():.3e}"


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", CASES)
def test_attn_bwd_stores_delta(gpu_lib, B, H, M, N, D, dtype, causal):
    ta = gpu_lib
    cpu, g = _inputs(B, H, M, N, D, dtype, causal, 110, ("q", "k", "v", "do"))
    _, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    nws = int(ta.load().attn_bwd_workspace_bytes(B, H, M, N, D, 0 if dtype == "f16" else 1))
    ws = torch.full((max(nws, 16),), 0xFF, dtype=torch.uint8, device="cuda")  # NaN-filled
    ta.attn_bwd(g["q"], g["k"], g["v"], g["o"], lse, g["do"], causal, ws=ws)
    assert ta.sync_status() == "TA_OK"
    _check_delta(ws, cpu, B, H, M)


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", CASES)
def test_piecewise_bwd_stores_delta(gpu_lib, B, H, M, N, D, dtype, causal):
    ta = gpu_lib
    w = max(1, N // 3)
    cpu, g = _inputs(B, H, M, N, D, dtype, causal, 111, ("q1", "k1", "q2", "k2", "v", "do"))
    _, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w, causal)
    nws = int(ta.load().piecewise_bwd_workspace_bytes(B, H, M, N, D, 0 if dtype == "f16" else 1))
    ws = torch.full((max(nws, 16),), 0xFF, dtype=torch.uint8, device="cuda")
    ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], g["o"], lse, g["do"], w, causal, ws=ws)
    assert ta.sync_status() == "TA_OK"
    _check_delta(ws, cpu, B, H, M)
