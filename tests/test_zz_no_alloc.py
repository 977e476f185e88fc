"""attn_bwd_noalloc: the backward for callers that cannot allocate.

Some callers cannot give the library a workspace: a host framework that keeps
all device memory in its own pool and offers plug-ins no allocator, or a step
loop where a cudaMalloc (which synchronises the device) is not acceptable.
attn_bwd_noalloc keeps its scratch in a fixed array inside the library
instead.  This test calls it through the C ABI twice in a row (different
inputs, so a stale scratch would show) and checks each result against
attn_bwd with a caller-provided workspace, within the gradient tolerance the
other GPU tests use.  The file is named to run last in a session.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu

TOL = 5e-2


def _noalloc_fn(lib):
    fn = lib.attn_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp] * 9 + [i] * 7 + [ctypes.c_float, vp]
    fn.restype = i
    return fn


def _case(ta, fn, B, H, S, D, dtype, causal, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q, k, v, do = (torch.randn(B, H, S, D, device="cuda", dtype=dtype, generator=g) for _ in range(4))
    o, lse = ta.attn_fwd(q, k, v, causal)
    ref = ta.attn_bwd(q, k, v, o, lse, do, causal)
    out = [torch.full_like(q, float("nan")) for _ in range(3)]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = 1 if dtype == torch.bfloat16 else 0
    st = fn(ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse), ptr(do), ptr(out[0]), ptr(out[1]), ptr(out[2]),
            B, H, S, S, D, dt, int(causal), -1.0, stream)
    assert st == 0, ta.STATUS.get(st, st)
    assert ta.sync_status() == "TA_OK"
    for name, a, b in zip(("dq", "dk", "dv"), out, ref):
        err = (a.float() - b.float()).abs().max().item()
        assert err <= TOL, f"{name}: max_abs {err:.3e}"


def test_noalloc_backward_matches_workspace_backward_twice(gpu_lib):
    ta = gpu_lib
    fn = _noalloc_fn(ta.load())
    _case(ta, fn, 2, 4, 1024, 128, torch.bfloat16, True, 1)
    _case(ta, fn, 1, 3, 640, 64, torch.float16, False, 2)


def test_noalloc_rejects_problems_above_its_capacity(gpu_lib):
    fn = _noalloc_fn(gpu_lib.load())
    vp = ctypes.c_void_p
    p = [vp(256 * (i + 1)) for i in range(9)]
    st = fn(*p, 1, 1024, 4096, 4096, 128, 1, 1, -1.0, vp(0))  # B*H*M = 2^22 rows > 2^21
    assert gpu_lib.STATUS[st] == "TA_ERR_UNSUPPORTED"
