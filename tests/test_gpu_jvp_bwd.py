"""GPU parity of the backward of the JVP (attn_bwd_jvp) through the C ABI
against the fp64 oracle: the gradients of <dO, O> + <dtO, tO> with respect to
q, k, v and the tangents.  16-bit cases compare every element against the
gradients' 5e-2 (unit-normal inputs) plus a bound derived element by element
from the roundings the kernels make (jvp_bwd_bounds: the row constants from
the stored O and tO, the 16-bit MMA operands, the output); the fp32 mode at
1e-4.
The forward outputs (o, lse, to, tlse) are the GPU's own attn_fwd_jvp."""
import numpy as np
import pytest
import torch

import oracle
import synth_inputs as si
from _parity import ROUND_U, TOL, compare, compare_bounded, inputs, jvp_bwd_bounds, sample_heads

pytestmark = pytest.mark.gpu

NAMES = ("q", "k", "v", "tq", "tk", "tv", "do", "dto")
GRADS = ("dq", "dk", "dv", "dtq", "dtk", "dtv")

CASES = [
    # B, H, M, N, D, dtype, causal
    (1, 2, 128, 128, 64, "f16", False),
    (1, 2, 256, 256, 64, "bf16", True),
    (2, 1, 256, 256, 128, "bf16", True),
    (1, 2, 200, 333, 64, "bf16", True),
    (1, 1, 333, 200, 128, "f16", True),    # M > N: the first rows see no key
    (2, 1, 129, 257, 128, "bf16", False),
    (1, 1, 1, 1, 64, "f16", True),
    (1, 1, 70, 500, 64, "f16", False),
    (1, 2, 150, 150, 32, "f16", True),     # D = 32, 16: the D = 64 kernels over zero-filled columns
    (1, 1, 100, 170, 16, "bf16", False),
]


def _run(ta, g, causal, ws=None):
    o, lse, to, tlse = ta.attn_fwd_jvp(*(g[n] for n in NAMES[:6]), causal=causal, with_tlse=True)
    grads = ta.attn_bwd_jvp(*(g[n] for n in NAMES[:6]), o, lse, to, tlse, g["do"], g["dto"], causal=causal, ws=ws)
    assert ta.sync_status() == "TA_OK"
    return grads


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", CASES)
def test_jvp_backward_small(gpu_lib, B, H, M, N, D, dtype, causal):
    cpu, g = inputs(B, H, M, N, D, dtype, 61, NAMES)
    grads = _run(gpu_lib, g, causal)
    ref = oracle.attention_jvp_bwd_bhsd(*(cpu[n] for n in NAMES), causal)
    bounds = jvp_bwd_bounds(cpu, causal, ROUND_U[dtype])
    for name, got, r in zip(GRADS, grads, ref):
        compare_bounded(name, got, r, TOL["grad"], bounds[name])


# Where no single key carries the whole softmax weight of a row (every
# P_ij < 1 - 1e-3), the exact gradients do not cancel and the derived bound
# must stay a modest addition to the flat 5e-2: at most half of it.
BOUND_CAP = 0.5 * TOL["grad"]


def _bound_stats(cpu, causal, heads, bounds):
    """Largest and median bound per gradient over the sampled heads, and the
    largest over the rows (dq, dtq) or keys (dk, dv, dtk, dtv) where every
    P < 1 - 1e-3."""
    x = {n: cpu[n].double().numpy() for n in ("q", "k")}
    M, N = x["q"].shape[2], x["k"].shape[2]
    s = oracle.default_scale(x["q"].shape[3], None)
    keep = oracle.allowed_mask(M, N, causal)
    stats = {}
    for name in GRADS:
        vals = np.stack([bounds[name][b, h] for b, h in heads])
        worst = 0.0
        for b, h in heads:
            S = np.where(keep, s * x["q"][b, h] @ x["k"][b, h].T, -np.inf)
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            ok = (P.max(axis=1) if name in ("dq", "dtq") else P.max(axis=0)) < 1 - 1e-3
            if ok.any():
                worst = max(worst, float(bounds[name][b, h][ok].max()))
        stats[name] = (float(vals.max()), float(np.median(vals)), worst)
    return stats


@pytest.mark.parametrize("causal", [False, True])
def test_jvp_backward_fp16_b2_h8_s1024_d64(gpu_lib, causal):
    """The JVP workload's shape ([2, 8, 1024, 64] fp16), sampled heads; prints
    how large the derived bound gets there and holds it under BOUND_CAP where
    the gradients do not cancel."""
    B, H, M, D = 2, 8, 1024, 64
    cpu, g = inputs(B, H, M, M, D, "f16", 62, NAMES)
    grads = _run(gpu_lib, g, causal)
    heads = sample_heads(B, H, 3)
    ref = oracle.attention_jvp_bwd_bhsd(*(cpu[n] for n in NAMES), causal, heads=heads)
    bounds = jvp_bwd_bounds(cpu, causal, ROUND_U["f16"], heads=heads)
    for name, (mx, med, worst) in _bound_stats(cpu, causal, heads, bounds).items():
        print(f"jvp backward bound, causal={causal}, {name}: max {mx:.2e}, median {med:.2e}, "
              f"max where every P < 1 - 1e-3: {worst:.2e}")
        assert worst <= BOUND_CAP, f"{name}: derived bound {worst:.2e} > {BOUND_CAP:.1e}"
    for name, got, r in zip(GRADS, grads, ref):
        compare_bounded(name, np.stack([got[b, h].float().cpu().numpy() for b, h in heads]),
                        np.stack([r[b, h] for b, h in heads]), TOL["grad"],
                        np.stack([bounds[name][b, h] for b, h in heads]))


@pytest.mark.parametrize("B,H,M,N,D,causal", [(1, 2, 128, 128, 64, False), (1, 1, 200, 333, 128, True),
                                              (1, 1, 333, 200, 64, True), (1, 2, 96, 150, 32, False),
                                              (1, 1, 100, 100, 16, True)])
def test_jvp_backward_fp32_mode(gpu_lib, B, H, M, N, D, causal):
    cpu = {n: si.randn((B, H, M if n in ("q", "tq", "do", "dto") else N, D), "f32", si.seed_for(63, i))
           for i, n in enumerate(NAMES)}
    g = {n: t.cuda() for n, t in cpu.items()}
    grads = _run(gpu_lib, g, causal)
    ref = oracle.attention_jvp_bwd_bhsd(*(cpu[n] for n in NAMES), causal)
    for name, got, r in zip(GRADS, grads, ref):
        compare(name, got, r, 1e-4)


def test_jvp_backward_empty_and_bad_arguments(gpu_lib):
    ta = gpu_lib
    dev = torch.device("cuda")
    # no query: every key-side gradient is zero
    cpu, g = inputs(1, 2, 0, 64, 64, "bf16", 64, NAMES)
    o = torch.empty(1, 2, 0, 64, device=dev, dtype=torch.bfloat16)
    l0 = torch.empty(1, 2, 0, device=dev, dtype=torch.float32)
    grads = ta.attn_bwd_jvp(*(g[n] for n in NAMES[:6]), o, l0, o, l0, g["do"], g["dto"], causal=True)
    assert ta.sync_status() == "TA_OK"
    for t in grads[1:3] + grads[4:6]:
        assert t.shape == (1, 2, 64, 64) and torch.all(t == 0)
    # no key: rows see nothing, every query-side gradient is zero
    cpu, g = inputs(1, 1, 64, 0, 64, "f16", 65, NAMES)
    o, lse, to, tlse = ta.attn_fwd_jvp(*(g[n] for n in NAMES[:6]), causal=False, with_tlse=True)
    grads = ta.attn_bwd_jvp(*(g[n] for n in NAMES[:6]), o, lse, to, tlse, g["do"], g["dto"])
    assert ta.sync_status() == "TA_OK"
    assert torch.all(grads[0] == 0) and torch.all(grads[3] == 0)
    # a workspace that is too small is refused before any launch
    cpu, g = inputs(1, 1, 128, 128, 64, "bf16", 66, NAMES)
    o, lse, to, tlse = ta.attn_fwd_jvp(*(g[n] for n in NAMES[:6]), with_tlse=True)
    small = torch.empty(16, device=dev, dtype=torch.uint8)
    with pytest.raises(ta.TAError):
        ta.attn_bwd_jvp(*(g[n] for n in NAMES[:6]), o, lse, to, tlse, g["do"], g["dto"], ws=small)
