"""The key split of the one-query-tile forward: attn_fwd_jvp (every D) and
piecewise_fwd at D = 128 give each 128-row query tile a cluster of two CTAs
that take half of its key tiles each; the second CTA's running max, sum and
unnormalised accumulators are merged into the first's over distributed
shared memory.  Each case runs with the split forced on and forced off
(ta_set_fwd_kv_split), checks both against the fp64 oracle at the usual
tolerances, and checks that L agrees between the two to fp32 rounding (the
merge is the online-softmax rescale, exact up to rounding)."""
import numpy as np
import pytest

import oracle
from _parity import TOL, compare, inputs, o_tol, to_np

pytestmark = pytest.mark.gpu

JVP_NAMES = ("q", "k", "v", "tq", "tk", "tv")

JVP_CASES = [
    # B, H, M, N, D, dtype, causal, kscale (keys in the second half of the
    # sequence multiplied by kscale: the halves' row maxima far apart)
    (1, 2, 1024, 1024, 64, "f16", True, 1.0),     # 1..8 key tiles: odd and even splits, diagonal in the second half
    (1, 1, 300, 700, 128, "bf16", False, 1.0),    # 6 key tiles, ragged N
    (1, 1, 333, 200, 64, "f16", True, 1.0),       # M > N: the first rows see no key
    (2, 1, 129, 257, 128, "bf16", False, 1.0),    # 3 key tiles: 2 + 1, ragged M
    (1, 1, 100, 100, 32, "f16", True, 1.0),       # one key tile: the second CTA has none
    (1, 1, 130, 900, 16, "bf16", True, 1.0),      # D = 16
    (1, 1, 256, 1024, 64, "f16", False, 3.0),
]


@pytest.fixture
def split_mode(gpu_lib):
    yield gpu_lib.set_fwd_kv_split
    gpu_lib.set_fwd_kv_split("auto")


def _jvp(ta, g, causal):
    out = ta.attn_fwd_jvp(*(g[n] for n in JVP_NAMES), causal=causal, with_tlse=True)
    assert ta.sync_status() == "TA_OK"
    return out


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal,kscale", JVP_CASES)
def test_jvp_forward_split_and_unsplit(gpu_lib, split_mode, B, H, M, N, D, dtype, causal, kscale):
    ta = gpu_lib
    cpu, g = inputs(B, H, M, N, D, dtype, 91, JVP_NAMES)
    if kscale != 1.0:
        cpu["k"][:, :, N // 2:] *= kscale  # rounded to the 16-bit type; the GPU gets the same values
        g["k"] = cpu["k"].to(g["k"].device)
    O, L, tO = oracle.attention_jvp_bhsd(*(cpu[n] for n in JVP_NAMES), causal)
    tL = oracle.attention_jvp_tl_bhsd(cpu["q"], cpu["k"], cpu["tq"], cpu["tk"], causal)
    res = {}
    for mode in ("never", "always"):
        split_mode(mode)
        o, lse, to, tlse = res[mode] = _jvp(ta, g, causal)
        compare(f"O ({mode})", o, O, o_tol(dtype))
        compare(f"L ({mode})", lse, L, TOL["L"])
        compare(f"tO ({mode})", to, tO, TOL["tO"])
        compare(f"tL ({mode})", tlse, tL, TOL["tO"])
    a, b = to_np(res["never"][1]), to_np(res["always"][1])
    fin = np.isfinite(a)
    assert np.array_equal(fin, np.isfinite(b)) and np.array_equal(a[~fin], b[~fin])
    assert np.abs(a[fin] - b[fin]).max(initial=0.0) <= 1e-5 * max(1.0, np.abs(a[fin]).max(initial=0.0))


PW_CASES = [
    # B, H, M, N, D, dtype, causal, w
    (1, 2, 1024, 1024, 128, "bf16", True, 300),
    (1, 1, 512, 700, 128, "f16", False, -50),
    (1, 1, 640, 640, 128, "bf16", True, 256),
    (1, 1, 384, 256, 128, "f16", True, 0),        # M > N
    (1, 1, 200, 1000, 128, "bf16", False, 10000), # every key near
]


@pytest.mark.parametrize("B,H,M,N,D,dtype,causal,w", PW_CASES)
def test_piecewise_forward_split_and_unsplit(gpu_lib, split_mode, B, H, M, N, D, dtype, causal, w):
    ta = gpu_lib
    names = ("q1", "k1", "q2", "k2", "v")
    cpu, g = inputs(B, H, M, N, D, dtype, 92, names)
    O, L = oracle.piecewise_fwd_bhsd(*(cpu[n] for n in names), causal, None, w)
    res = {}
    for mode in ("never", "always"):
        split_mode(mode)
        o, lse = res[mode] = ta.piecewise_fwd(*(g[n] for n in names), w, causal)
        assert ta.sync_status() == "TA_OK"
        compare(f"O ({mode})", o, O, o_tol(dtype))
        compare(f"L ({mode})", lse, L, TOL["L"])
    a, b = to_np(res["never"][1]), to_np(res["always"][1])
    fin = np.isfinite(a)
    assert np.array_equal(fin, np.isfinite(b))
    assert np.abs(a[fin] - b[fin]).max(initial=0.0) <= 1e-5 * max(1.0, np.abs(a[fin]).max(initial=0.0))


def test_the_estimate_on_this_gpu(gpu_lib):
    """On this GPU the library's estimate leaves the JVP workload
    [2, 8, 1024, 64] fp16 whole (its grid is nearly a wave already) and
    splits a long key range with few query tiles."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms < 128:
        pytest.skip("the estimate assumes a GPU with at least 128 SMs")
    for causal in (False, True):
        assert gpu_lib.fwd_kv_split("attn_fwd_jvp", 2, 8, 1024, 1024, 64, torch.float16, causal) == 1
    assert gpu_lib.fwd_kv_split("attn_fwd_jvp", 1, 4, 1024, 8192, 64, torch.float16, False) == 2
