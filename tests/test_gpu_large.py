"""GPU parity with tensors of more than 2^31 elements: B=1, H=66000,
M=N=256, D=128 (2.16e9 elements per tensor, 4.3 GB in bf16), through every
entry point (forward and backward causal and not, the JVP forward and its
backward, piecewise, the merge, the e5m2 forward, the fp32 mode), so every
kernel forms element offsets past 2^31.

The heads repeat a block of 61 distinct seeded heads.  A 32-bit wrap of an
element offset would move an access by 2^31 elements = 65536 heads, which 61
does not divide, so an aliased read or write would meet another head's data
and show as a mismatch.  Head 65536 starts exactly at element 2^31; heads on
both sides of that boundary are compared with the oracle."""
import pytest
import torch

import oracle
import synth_inputs as si
from _parity import ROUND_U, TOL, compare, compare_bounded, inputs, jvp_bwd_bounds, o_tol

pytestmark = pytest.mark.gpu

H, S, D, PERIOD = 66000, 256, 128, 61
CHECK = (0, 60, 65535, 65536, 65537, 65999)
NAMES = ("q", "k", "v", "do")


def _tile_heads(x):
    """[1, PERIOD, ...] -> [1, H, ...] on the device: head h holds block head
    h % PERIOD."""
    reps = (H + PERIOD - 1) // PERIOD
    return x.cuda().repeat((1, reps) + (1,) * (x.dim() - 2))[:, :H].contiguous()


def _need_memory(gb):
    free, _ = torch.cuda.mem_get_info()
    if free < (gb << 30):
        pytest.skip(f"needs about {gb} GB of free device memory")


@pytest.mark.parametrize("causal", [False, True])
def test_more_than_2_31_elements(gpu_lib, causal):
    ta = gpu_lib
    _need_memory(48)
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
    ta = gpu_lib
    _need_memory(48)
    blk = [si.randn((1, PERIOD, S, D), "bf16", si.seed_for(98, 0)),
           si.randn((1, PERIOD, S), "f32", si.seed_for(98, 1)) * 3,
           si.randn((1, PERIOD, S, D), "bf16", si.seed_for(98, 2)),
           si.randn((1, PERIOD, S), "f32", si.seed_for(98, 3)) * 3,
           si.randn((1, PERIOD, S, D), "bf16", si.seed_for(98, 4)),
           si.randn((1, PERIOD, S), "f32", si.seed_for(98, 5))]
    g = [_tile_heads(t) for t in blk]
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


JVP_NAMES = ("q", "k", "v", "tq", "tk", "tv", "do", "dto")
GRADS = ("dq", "dk", "dv", "dtq", "dtk", "dtv")


def test_jvp_fwd_bwd_more_than_2_31_elements(gpu_lib):
    """attn_fwd_jvp (tO and tL) and attn_bwd_jvp, fp16 causal, with the
    gradients held to the derived per-element bound as in the other JVP
    backward tests."""
    ta = gpu_lib
    _need_memory(96)
    cpu, _ = inputs(1, PERIOD, S, S, D, "f16", 96, JVP_NAMES)
    g = {n: _tile_heads(t) for n, t in cpu.items()}
    o, lse, to, tlse = ta.attn_fwd_jvp(*(g[n] for n in JVP_NAMES[:6]), causal=True, with_tlse=True)
    grads = ta.attn_bwd_jvp(*(g[n] for n in JVP_NAMES[:6]), o, lse, to, tlse, g["do"], g["dto"], causal=True)
    assert ta.sync_status() == "TA_OK"
    u = ROUND_U["f16"]
    for h in CHECK:
        one = {n: t[:, h % PERIOD:h % PERIOD + 1] for n, t in cpu.items()}
        x = [one[n][0, 0] for n in JVP_NAMES]
        O, L, tO = oracle.attention_jvp(*x[:6], True)
        compare(f"O[{h}]", o[0, h], O, o_tol("f16"), u)
        compare(f"L[{h}]", lse[0, h], L, TOL["L"])
        compare(f"tO[{h}]", to[0, h], tO, TOL["tO"], u)
        compare(f"tL[{h}]", tlse[0, h], oracle.attention_jvp_tl(x[0], x[1], x[3], x[4], True), TOL["L"])
        bounds = jvp_bwd_bounds(one, True, u)
        for name, got, ref in zip(GRADS, grads, oracle.attention_jvp_bwd(*x, True)):
            compare_bounded(f"{name}[{h}]", got[0, h], ref, TOL["grad"], bounds[name][0, 0])
    del g, o, lse, to, tlse, grads
    torch.cuda.empty_cache()


def test_piecewise_more_than_2_31_elements(gpu_lib):
    """piecewise_fwd / piecewise_bwd, bf16 causal, w = 100 (tiles of all three
    classes: near, far and straddling)."""
    ta = gpu_lib
    _need_memory(80)
    names = ("q1", "k1", "q2", "k2", "v", "do")
    cpu, _ = inputs(1, PERIOD, S, S, D, "bf16", 95, names)
    g = {n: _tile_heads(t) for n, t in cpu.items()}
    w = 100
    o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w, True)
    grads = ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], w, True)
    assert ta.sync_status() == "TA_OK"
    u = ROUND_U["bf16"]
    for h in CHECK:
        x = [cpu[n][0, h % PERIOD] for n in names]
        O, L = oracle.piecewise_fwd(*x[:5], True, None, w)
        compare(f"O[{h}]", o[0, h], O, o_tol("bf16"), u)
        compare(f"L[{h}]", lse[0, h], L, TOL["L"])
        for name, got, ref in zip(("dq1", "dk1", "dq2", "dk2", "dv"), grads, oracle.piecewise_bwd(*x, True, None, w)):
            compare(f"{name}[{h}]", got[0, h], ref, TOL["grad"], u)
    del g, o, lse, grads
    torch.cuda.empty_cache()


def test_fp8_forward_more_than_2_31_elements(gpu_lib):
    """attn_fwd_fp8 (e5m2, 2.16 GB per tensor), causal, within the e5m2
    rounding bound of the output."""
    import numpy as np
    ta = gpu_lib
    _need_memory(24)
    blk = [si.randn((1, PERIOD, S, D), "e5m2", si.seed_for(94, i)) for i in range(3)]
    q, k, v = (_tile_heads(t.view(torch.uint8)) for t in blk)  # bytes: no float8 copy kernels needed
    vt = v.transpose(-1, -2).contiguous().view(torch.float8_e5m2)
    q, k = q.view(torch.float8_e5m2), k.view(torch.float8_e5m2)
    del v
    o, lse = ta.attn_fwd_fp8(q, k, vt, True)
    assert ta.sync_status() == "TA_OK"
    U = 2.0 ** -3
    keep = oracle.allowed_mask(S, S, True)
    s = oracle.default_scale(D)
    for h in CHECK:
        qf, kf, vf = (t[0, h % PERIOD].to(torch.float64).numpy() for t in blk)
        O, L = oracle.attention_fwd(qf, kf, vf, True)
        P = np.where(keep, np.exp(np.where(keep, s * qf @ kf.T, -np.inf) - L[:, None]), 0.0)
        bound = U * (1 + U) * (P @ np.abs(vf)) + U * np.abs(O) + 1e-6
        got = o[0, h].cpu().to(torch.float64).numpy()
        assert np.all(np.abs(got - O) <= bound), f"O[{h}] outside the e5m2 bound"
        compare(f"L[{h}]", lse[0, h], L, TOL["L"])
    del q, k, vt, o, lse
    torch.cuda.empty_cache()


def test_fp32_mode_more_than_2_31_elements(gpu_lib):
    """The fp32 mode (8.6 GB per tensor), forward and backward, causal, at
    its 1e-4 tolerance."""
    ta = gpu_lib
    _need_memory(96)
    cpu = {n: si.randn((1, PERIOD, S, D), "f32", si.seed_for(93, i)) for i, n in enumerate(NAMES)}
    g = {n: _tile_heads(t) for n, t in cpu.items()}
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    assert ta.sync_status() == "TA_OK"
    for h in CHECK:
        x = [cpu[n][0, h % PERIOD] for n in NAMES]
        O, L = oracle.attention_fwd(*x[:3], True)
        compare(f"O[{h}]", o[0, h], O, 1e-4, 2.0 ** -24)
        compare(f"L[{h}]", lse[0, h], L, 1e-4)
        for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv), oracle.attention_bwd(*x, True)):
            compare(f"{name}[{h}]", got[0, h], ref, 1e-4, 2.0 ** -24)
    del g, o, lse, dq, dk, dv
    torch.cuda.empty_cache()
