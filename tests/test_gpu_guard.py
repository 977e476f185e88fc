"""The guard build: libtattn_guard.so, the same kernels with device-side
checks compiled in (TA_GUARD): every TMA load's shared-memory destination
and coordinates, every TMEM load and store's lane quadrant and columns, every
MMA batch's TMEM and shared-memory operands, the row stores' alignment and
each CTA's work decode.  A failed check skips its access and turns the next
ta_sync_status into TA_ERR_GUARD, naming the check's line.

Every entry point runs here on shapes chosen for their edges: ragged M and
N, M > N (rows that see no key), a single row, D = 16 to 128, causal and not,
the key split forced on and off, the one-pass backward, the e5m2 forward,
the merge, the fp32 mode and empty problems.
Each call must leave the status at TA_OK, and a few results are compared with
the oracle to show the guard build computes what the product build does.
The self-test shows the channel works: one thread fails a check on purpose,
without touching memory, and the status reads TA_ERR_GUARD."""
import ctypes

import pytest
import torch

import oracle
import synth_inputs as si
from _parity import TOL, compare, inputs, o_tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def guarded(gpu_lib):
    """The binding, pointed at the guard library for this module."""
    from tiled_attention_tcgen05_gb300 import build
    path = build.build(guard=True)
    ta = gpu_lib
    saved = ta._lib
    ta._lib = None
    lib = ta.load(path)
    assert lib.ta_guard_build() == 1
    yield ta
    ta.set_fwd_kv_split("auto")
    ta._lib = saved
    assert ta.load().ta_guard_build() == 0


def _ok(ta, what):
    st = ta.sync_status()
    assert st == "TA_OK", f"{what}: {st} at {ta.load().ta_guard_last().decode()}"


def test_guard_channel_reports_a_failed_check(guarded):
    ta = guarded
    assert ta.load().ta_selftest_guard(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == 0
    assert ta.sync_status() == "TA_ERR_GUARD"
    assert ta.load().ta_guard_last().decode().startswith("aux.cu:")
    _ok(ta, "status after the self-test")  # read and cleared


FB_CASES = [
    # B, H, M, N, D, dtype, causal
    (1, 2, 200, 333, 64, "f16", True),
    (1, 1, 333, 200, 128, "bf16", True),
    (2, 1, 1, 1, 64, "f16", False),
    (1, 1, 130, 190, 16, "bf16", False),
    (1, 2, 257, 129, 32, "f16", True),
    (1, 1, 384, 384, 128, "bf16", False),
]


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", FB_CASES)
def test_forward_and_backward_pass_every_check(guarded, B, H, M, N, D, dtype, causal):
    ta = guarded
    cpu, g = inputs(B, H, M, N, D, dtype, 95, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    _ok(ta, "attn_fwd + attn_bwd")
    O, L = oracle.attention_fwd_bhsd(cpu["q"], cpu["k"], cpu["v"], causal)
    compare("O", o, O, o_tol(dtype))
    compare("L", lse, L, TOL["L"])
    for name, got, ref in zip(("dQ", "dK", "dV"), (dq, dk, dv),
                              oracle.attention_bwd_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["do"], causal)):
        compare(name, got, ref, TOL["grad"])
    if D == 128:
        ta.attn_bwd_fused(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
        _ok(ta, "attn_bwd_fused")


@pytest.mark.parametrize("split", ["never", "always"])
@pytest.mark.parametrize("B,H,M,N,D,dtype,causal", [(1, 2, 200, 333, 64, "f16", True),
                                                     (1, 1, 333, 600, 128, "bf16", False),
                                                     (1, 1, 100, 100, 32, "f16", True)])
def test_jvp_pass_every_check(guarded, split, B, H, M, N, D, dtype, causal):
    ta = guarded
    ta.set_fwd_kv_split(split)
    names = ("q", "k", "v", "tq", "tk", "tv", "do", "dto")
    cpu, g = inputs(B, H, M, N, D, dtype, 96, names)
    o, lse, to, tlse = ta.attn_fwd_jvp(*(g[n] for n in names[:6]), causal=causal, with_tlse=True)
    ta.attn_bwd_jvp(*(g[n] for n in names[:6]), o, lse, to, tlse, g["do"], g["dto"], causal=causal)
    _ok(ta, f"attn_fwd_jvp ({split}) + attn_bwd_jvp")
    O, L, tO = oracle.attention_jvp_bhsd(*(cpu[n] for n in names[:6]), causal)
    compare("O", o, O, o_tol(dtype))
    compare("tO", to, tO, TOL["tO"])
    ta.set_fwd_kv_split("auto")


@pytest.mark.parametrize("split", ["never", "always"])
@pytest.mark.parametrize("B,H,M,N,D,dtype,causal,w", [(1, 2, 200, 333, 64, "bf16", True, 77),
                                                       (1, 1, 384, 256, 128, "f16", True, 0),
                                                       (1, 1, 300, 333, 128, "bf16", False, 40)])
def test_piecewise_pass_every_check(guarded, split, B, H, M, N, D, dtype, causal, w):
    ta = guarded
    ta.set_fwd_kv_split(split)
    names = ("q1", "k1", "q2", "k2", "v", "do")
    cpu, g = inputs(B, H, M, N, D, dtype, 97, names)
    o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w, causal)
    ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], w, causal)
    _ok(ta, f"piecewise ({split})")
    O, L = oracle.piecewise_fwd_bhsd(*(cpu[n] for n in names[:5]), causal, None, w)
    compare("O", o, O, o_tol(dtype))
    ta.set_fwd_kv_split("auto")


@pytest.mark.parametrize("B,H,M,N,D,causal", [(1, 2, 200, 336, 64, True), (1, 1, 300, 256, 128, False)])
def test_fp8_forward_passes_every_check(guarded, B, H, M, N, D, causal):
    ta = guarded
    q = si.randn((B, H, M, D), "e5m2", si.seed_for(98, 0)).cuda()
    k = si.randn((B, H, N, D), "e5m2", si.seed_for(98, 1)).cuda()
    vt = si.randn((B, H, D, N), "e5m2", si.seed_for(98, 2)).cuda()
    ta.attn_fwd_fp8(q, k, vt, causal)
    _ok(ta, "attn_fwd_fp8")


@pytest.mark.parametrize("D,dtype", [(64, "bf16"), (128, "f16"), (16, "bf16")])
def test_merge_passes_every_check(guarded, D, dtype):
    ta = guarded
    B, H, M = 1, 2, 300
    o1, o2, do = (si.randn((B, H, M, D), dtype, si.seed_for(99, i)).cuda() for i in range(3))
    l1, l2 = (si.randn((B, H, M), "f32", si.seed_for(99, 3 + i)).cuda() for i in range(2))
    ta.merge_fwd(o1, l1, o2, l2)
    ta.merge_bwd(o1, l1, o2, l2, do)
    _ok(ta, "merge")


def test_fp32_mode_and_empty_problems_pass_every_check(guarded):
    ta = guarded
    names = ("q", "k", "v", "tq", "tk", "tv", "do")
    g = {n: si.randn((1, 1, 150 if n in ("q", "tq", "do") else 90, 64), "f32", si.seed_for(100, i)).cuda()
         for i, n in enumerate(names)}
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True)
    ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    ta.attn_fwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], causal=True)
    _ok(ta, "fp32 mode")
    cpu, e = inputs(1, 2, 0, 64, 64, "bf16", 101, ("q", "k", "v"))
    ta.attn_fwd(e["q"], e["k"], e["v"], True)
    cpu, e = inputs(1, 2, 64, 0, 64, "bf16", 101, ("q", "k", "v"))
    ta.attn_fwd(e["q"], e["k"], e["v"], False)
    _ok(ta, "empty problems")
