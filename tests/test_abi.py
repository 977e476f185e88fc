"""The C ABI without a GPU: libtattn.so builds, loads, exports every function
include/tattn.h declares, and rejects bad arguments with the documented
status codes before any CUDA call is made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tattn.h")

OK, INVALID, UNSUPPORTED, ALIGNMENT = 0, 1, 2, 3
F16, BF16, F32 = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    from tiled_attention_tcgen05_gb300 import build
    path = build.build()
    import tiled_attention_tcgen05_gb300 as ta
    return ta.load(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "extern")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_bytes", "attn_fwd_jvp", "piecewise_fwd",
              "piecewise_bwd", "ta_sync_status", "ta_status_str"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in tattn.h but not exported"


def test_status_strings(lib):
    assert lib.ta_status_str(0) == b"TA_OK"
    assert lib.ta_status_str(5) == b"TA_ERR_TIMEOUT"


def _fwd(lib, q=16, k=32, v=48, o=64, lse=80, B=1, H=1, M=128, N=128, D=64, dt=BF16):
    vp = ctypes.c_void_p
    return lib.attn_fwd(vp(q), vp(k), vp(v), vp(o), vp(lse), B, H, M, N, D, dt, 0, -1.0, vp(0))


def test_validation_codes(lib):
    assert _fwd(lib, D=96) == UNSUPPORTED
    assert _fwd(lib, D=256) == UNSUPPORTED
    assert _fwd(lib, dt=F32, D=96) == UNSUPPORTED
    assert _fwd(lib, dt=7) == UNSUPPORTED
    assert _fwd(lib, dt=F32, k=0x1004) == ALIGNMENT
    assert _fwd(lib, B=-1) == INVALID
    assert _fwd(lib, M=-5) == INVALID
    assert _fwd(lib, q=0) == INVALID
    assert _fwd(lib, lse=0) == INVALID
    assert _fwd(lib, k=0x1008) == ALIGNMENT
    assert _fwd(lib, o=0x1004) == ALIGNMENT
    assert _fwd(lib, B=0) == OK          # empty: no work, no launch
    assert _fwd(lib, M=0) == OK
    assert _fwd(lib, M=128 * 65536) == UNSUPPORTED  # more query tiles than the grid allows


def test_backward_workspace_and_validation(lib):
    vp = ctypes.c_void_p
    assert lib.attn_bwd_workspace_bytes(1, 32, 8192, 8192, 128, BF16) == 32 * 8192 * 4
    assert lib.attn_bwd_workspace_bytes(1, 1, 3, 3, 64, F16) == 256
    # the fused backward: delta, then the fp32 dQ accumulator (D = 128, 16-bit)
    assert lib.attn_bwd_fused_workspace_bytes(1, 32, 8192, 8192, 128, BF16) == 32 * 8192 * 4 + 32 * 8192 * 128 * 4
    assert lib.attn_bwd_fused_workspace_bytes(1, 1, 3, 3, 128, F16) == 256 + 3 * 128 * 4
    assert lib.attn_bwd_fused_workspace_bytes(1, 1, 3, 3, 128, F32) == 256
    assert lib.attn_bwd_fused_workspace_bytes(0, 1, 3, 3, 128, F16) == 0
    assert lib.attn_bwd_workspace_bytes(0, 1, 3, 3, 64, F16) == 0
    p = [vp(16 * (i + 1)) for i in range(10)]
    st = lib.attn_bwd(*p[:9], vp(0), 1024, 1, 1, 128, 128, 64, BF16, 1, -1.0, vp(0))
    assert st == INVALID  # null workspace
    st = lib.attn_bwd(*p[:9], vp(0x2008), 1024, 1, 1, 128, 128, 64, BF16, 1, -1.0, vp(0))
    assert st == ALIGNMENT
    # attn_bwd_fused: a workspace with room for delta alone is refused before any
    # launch; head sizes other than 128 and the fp32 mode are not supported
    st = lib.attn_bwd_fused(*p[:9], vp(0x4000), 512, 1, 1, 128, 128, 128, BF16, 1, -1.0, vp(0))
    assert st == INVALID
    st = lib.attn_bwd_fused(*p[:9], vp(0x4000), 1 << 20, 1, 1, 128, 128, 64, BF16, 1, -1.0, vp(0))
    assert st == UNSUPPORTED
    st = lib.attn_bwd_fused(*p[:9], vp(0x4000), 1 << 20, 1, 1, 128, 128, 128, F32, 1, -1.0, vp(0))
    assert st == UNSUPPORTED
    st = lib.attn_bwd_fused(*p[:9], vp(0x4008), 1 << 20, 1, 1, 128, 128, 128, BF16, 1, -1.0, vp(0))
    assert st == ALIGNMENT
    # a head size outside {16, 32, 64, 128} is refused before any launch
    q = [vp(16 * (i + 1)) for i in range(14)]
    st = lib.piecewise_bwd(*q, 1 << 20, 1, 1, 128, 128, 96, BF16, 1, -1.0, 64, vp(0))
    assert st == UNSUPPORTED


def test_binding_fails_loudly_without_library(tmp_path):
    import tiled_attention_tcgen05_gb300 as ta
    saved = ta._lib
    try:
        ta._lib = None
        with pytest.raises(RuntimeError, match="not built"):
            ta.load(str(tmp_path / "missing.so"))
    finally:
        ta._lib = saved


def test_jvp_backward_workspace_and_validation(lib):
    """attn_bwd_jvp: workspace size (eps and delta2 rows) and the argument
    checks that run before any launch."""
    vp = ctypes.c_void_p
    assert lib.attn_bwd_jvp_workspace_bytes(2, 8, 1024, 1024, 64, F16) == 2 * 16 * 1024 * 4
    assert lib.attn_bwd_jvp_workspace_bytes(1, 1, 3, 3, 64, F16) == 512
    assert lib.attn_bwd_jvp_workspace_bytes(0, 1, 3, 3, 64, F16) == 0
    p = [vp(16 * (i + 1)) for i in range(18)]

    def call(ptrs, ws, nbytes, D=64, dt=F16, M=128, N=128):
        return lib.attn_bwd_jvp(*ptrs, ws, nbytes, 1, 1, M, N, D, dt, 1, -1.0, vp(0))

    nws = 1 << 20
    assert call(p, vp(0x4000), nws, D=96) == UNSUPPORTED
    assert call(p, vp(0x4000), nws, dt=5) == UNSUPPORTED
    assert call(p, vp(0), nws) == INVALID                  # null workspace
    assert call(p, vp(0x4000), 16) == INVALID              # workspace too small
    no_tl = list(p)
    no_tl[9] = vp(0)                                        # tlse is required
    assert call(no_tl, vp(0x4000), nws) == INVALID
    misaligned = list(p)
    misaligned[11] = vp(0x2008)                             # dtO
    assert call(misaligned, vp(0x4000), nws) == ALIGNMENT
    assert lib.attn_bwd_jvp(*p, vp(0x4000), nws, 0, 1, 128, 128, 64, F16, 1, -1.0, vp(0)) == OK  # B = 0


def test_forward_key_split_choice(lib):
    """Which problems the one-query-tile forward splits (host logic only: the
    SM count is passed in, so no CUDA call is made)."""
    f = lib.ta_fwd_kv_split
    STD, PW, JVP = 0, 1, 2
    # the JVP workload [2, 8, 1024, 64] fp16 on 152 SMs: 128 CTAs, under one
    # wave.  Split, they would be 256 CTAs in two waves: the second wave's
    # set-up and epilogue cost what the shorter key ranges save -> no split,
    # causal or not.
    assert f(JVP, 2, 8, 1024, 1024, 64, F16, 1, 152) == 1
    assert f(JVP, 2, 8, 1024, 1024, 64, F16, 0, 152) == 1
    # one head: 8 CTAs; split, 16 CTAs in one wave with half the key tiles each
    assert f(JVP, 1, 1, 1024, 1024, 64, F16, 1, 152) == 2
    # more query tiles than SMs: the grid already balances itself
    assert f(JVP, 1, 32, 8192, 8192, 128, BF16, 1, 152) == 1
    # one key tile per query tile: nothing to share
    assert f(JVP, 1, 4, 128, 128, 64, F16, 0, 152) == 1
    # a few long rows: split
    assert f(JVP, 1, 1, 1024, 4096, 128, BF16, 0, 152) == 2
    # piecewise: the D = 128 forward (one query tile per CTA) splits, the D = 64
    # two-tile forward and the standard forward never do
    assert f(PW, 1, 1, 4096, 4096, 128, BF16, 1, 152) == 2
    assert f(PW, 1, 1, 4096, 4096, 64, BF16, 1, 152) == 1
    assert f(STD, 1, 1, 4096, 4096, 128, BF16, 1, 152) == 1
    # the fp32 mode runs SIMT kernels
    assert f(JVP, 1, 1, 1024, 4096, 64, F32, 0, 152) == 1
    # invalid arguments
    assert f(JVP, 1, 1, 1024, 1024, 96, F16, 0, 152) == 0
    assert f(3, 1, 1, 1024, 1024, 64, F16, 0, 152) == 0
    assert f(JVP, 0, 1, 1024, 1024, 64, F16, 0, 152) == 0
    # the process-wide setting overrides the estimate
    try:
        lib.ta_set_fwd_kv_split(1)
        assert f(JVP, 1, 1, 1024, 1024, 64, F16, 1, 152) == 1
        lib.ta_set_fwd_kv_split(2)
        assert f(JVP, 2, 8, 1024, 1024, 64, F16, 0, 152) == 2
        assert f(JVP, 1, 32, 8192, 8192, 128, BF16, 1, 152) == 2
        assert f(STD, 1, 1, 4096, 4096, 128, BF16, 1, 152) == 1  # no split kernel there
    finally:
        lib.ta_set_fwd_kv_split(0)
    assert f(JVP, 2, 8, 1024, 1024, 64, F16, 0, 152) == 1


def test_guard_build_flag(lib):
    """libtattn.so compiles the device-side checks out; libtattn_guard.so (the
    test build, csrc/guard.cuh) has them and exports the same functions."""
    assert lib.ta_guard_build() == 0
    assert lib.ta_guard_last() == b""
    from tiled_attention_tcgen05_gb300 import build
    g = ctypes.CDLL(build.build(guard=True))
    g.ta_guard_build.restype = ctypes.c_int
    assert g.ta_guard_build() == 1
    for n in declared_functions():
        assert hasattr(g, n), f"{n} declared in tattn.h but not exported by the guard build"
