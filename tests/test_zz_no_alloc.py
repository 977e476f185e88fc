"""attn_bwd_noalloc: the backward for callers that cannot allocate.

Some callers cannot give the library a workspace: a host framework that keeps
all device memory in its own pool and offers plug-ins no allocator, or a step
loop where a cudaMalloc (which synchronises the device) is not acceptable.
attn_bwd_noalloc keeps its scratch in a fixed array inside the library
instead.  These tests call it through the C ABI on seeded inputs:

* twice in a row with different inputs (a stale scratch would show), each
  result against the fp64 oracle on whole heads and against attn_bwd with a
  caller-provided workspace, within the gradient tolerance the other GPU tests
  use;
* at exactly the array's capacity, B*H*M = 2^21 rows, with the heads at the
  end of the array checked against the oracle;
* one row past the capacity, which must be refused with TA_ERR_UNSUPPORTED.

The file is named to run last in a session.
"""
import ctypes

import pytest
import torch

import oracle
from _parity import TOL, compare, heads_of, inputs

pytestmark = pytest.mark.gpu

CAPACITY_ROWS = 1 << 21


def _noalloc_fn(lib):
    fn = lib.attn_bwd_noalloc
    vp, i = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp] * 9 + [i] * 7 + [ctypes.c_float, vp]
    fn.restype = i
    return fn


def _call(ta, fn, g, o, lse, causal):
    B, H, S, D = g["q"].shape
    out = [torch.full_like(g["q"], float("nan")) for _ in range(3)]
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = 1 if g["q"].dtype == torch.bfloat16 else 0
    st = fn(ptr(g["q"]), ptr(g["k"]), ptr(g["v"]), ptr(o), ptr(lse), ptr(g["do"]), ptr(out[0]), ptr(out[1]),
            ptr(out[2]), B, H, S, S, D, dt, int(causal), -1.0, stream)
    assert st == 0, ta.STATUS.get(st, st)
    assert ta.sync_status() == "TA_OK"
    return out


def _case(ta, fn, B, H, S, D, dtype, causal, workload, heads):
    cpu, g = inputs(B, H, S, S, D, dtype, workload, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal)
    out = _call(ta, fn, g, o, lse, causal)
    ref = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal)
    exact = oracle.attention_bwd_bhsd(cpu["q"], cpu["k"], cpu["v"], cpu["do"], causal, heads=heads)
    for name, a, b, x in zip(("dq", "dk", "dv"), out, ref, exact):
        compare(name + " vs attn_bwd", a, b.double().cpu().numpy(), TOL["grad"])
        compare(name + " vs oracle", heads_of(a, heads), heads_of(x, heads), TOL["grad"])


def test_noalloc_backward_twice_against_oracle_and_workspace_backward(gpu_lib):
    ta = gpu_lib
    fn = _noalloc_fn(ta.load())
    _case(ta, fn, 2, 4, 1024, 128, "bf16", True, 81, [(0, 0), (1, 3)])
    _case(ta, fn, 1, 3, 640, 64, "f16", False, 82, [(0, 0), (0, 2)])


def test_noalloc_at_exactly_its_capacity(gpu_lib):
    """B*H*M = 2^21 rows (B=1, H=2048, M=N=1024, D=64 fp16, causal): the
    heads repeat a block of 61 seeded heads; the last heads use the end of
    the scratch array and are checked against the oracle."""
    ta = gpu_lib
    fn = _noalloc_fn(ta.load())
    H, S, D, period = 2048, 1024, 64, 61
    assert H * S == CAPACITY_ROWS
    cpu, blk = inputs(1, period, S, S, D, "f16", 83, ("q", "k", "v", "do"))
    reps = (H + period - 1) // period
    g = {n: t.repeat(1, reps, 1, 1)[:, :H].contiguous() for n, t in blk.items()}
    del blk
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True)
    out = _call(ta, fn, g, o, lse, True)
    ref = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    for name, a, b in zip(("dq", "dk", "dv"), out, ref):
        assert (a.float() - b.float()).abs().max().item() <= TOL["grad"], name
    for h in (0, H - 2, H - 1):
        x = [cpu[n][0, h % period] for n in ("q", "k", "v", "do")]
        for name, got, exact in zip(("dq", "dk", "dv"), out, oracle.attention_bwd(*x, True)):
            compare(f"{name}[{h}]", got[0, h], exact, TOL["grad"])
    del g, o, lse, out, ref
    torch.cuda.empty_cache()


def test_noalloc_rejects_problems_above_its_capacity(gpu_lib):
    fn = _noalloc_fn(gpu_lib.load())
    vp = ctypes.c_void_p
    p = [vp(256 * (i + 1)) for i in range(9)]
    st = fn(*p, 1, 1024, 4096, 4096, 128, 1, 1, -1.0, vp(0))  # B*H*M = 2^22 rows
    assert gpu_lib.STATUS[st] == "TA_ERR_UNSUPPORTED"
    st = fn(*p, 1, 1, CAPACITY_ROWS + 1, CAPACITY_ROWS + 1, 64, 0, 0, -1.0, vp(0))  # one row past it
    assert gpu_lib.STATUS[st] == "TA_ERR_UNSUPPORTED"
    st = fn(*p, 1 << 20, 1 << 20, 1, 1, 64, 0, 0, -1.0, vp(0))  # B*H past 2^31: no overflow in the check
    assert gpu_lib.STATUS[st] == "TA_ERR_INVALID_ARG"
