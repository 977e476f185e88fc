"""Python binding of libtattn.so (fused attention for GB300 / sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI declared in include/tattn.h.  PyTorch provides the
device memory and the current stream.  There is no CPU fallback: if the
library is missing or fails to load, every call raises.

Entry points (same names as the C ABI):
  attn_fwd(q, k, v, causal, sm_scale)                -> (o, lse)
  attn_bwd(q, k, v, o, lse, do, causal, sm_scale)    -> (dq, dk, dv)
  attn_bwd_fused(q, k, v, o, lse, do, causal, sm_scale) -> (dq, dk, dv)  [D = 128]
  attn_fwd_jvp(q, k, v, tq, tk, tv, causal, sm_scale, with_tlse) -> (o, lse, to[, tlse])
  attn_bwd_jvp(q, k, v, tq, tk, tv, o, lse, to, tlse, do, dto, causal, sm_scale)
                                                     -> (dq, dk, dv, dtq, dtk, dtv)
  piecewise_fwd(q1, k1, q2, k2, v, w, causal, sm_scale) -> (o, lse)
  piecewise_bwd(q1, k1, q2, k2, v, o, lse, do, w, causal, sm_scale)
                                                     -> (dq1, dk1, dq2, dk2, dv)
Tensors are contiguous [B, H, S, D] float16/bfloat16 CUDA tensors; lse is
float32 [B, H, M].  sm_scale None means 1/sqrt(D).
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = ["load", "lib_path", "attn_fwd", "attn_bwd", "attn_bwd_fused", "attn_fwd_jvp", "attn_bwd_jvp", "piecewise_fwd", "piecewise_bwd", "merge_fwd", "merge_bwd", "attn_fwd_fp8",
           "attn_bwd_workspace_bytes", "attn_bwd_fused_workspace_bytes", "sync_status", "selftest_wait_timeout", "profile_enable",
           "profile_read", "set_wait_timeout_ms", "fwd_kv_split", "set_fwd_kv_split", "TAError", "STATUS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libtattn.so")
_lib = None

STATUS = {0: "TA_OK", 1: "TA_ERR_INVALID_ARG", 2: "TA_ERR_UNSUPPORTED", 3: "TA_ERR_ALIGNMENT",
          4: "TA_ERR_CUDA", 5: "TA_ERR_TIMEOUT", 6: "TA_ERR_GUARD"}
_DT = {torch.float16: 0, torch.bfloat16: 1, torch.float32: 2}

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "attn_fwd": ([_vp] * 5 + [_i] * 7 + [_f, _vp], _i),
    "attn_bwd_workspace_bytes": ([_i] * 6, _sz),
    "attn_bwd": ([_vp] * 10 + [_sz] + [_i] * 7 + [_f, _vp], _i),
    "attn_bwd_fused_workspace_bytes": ([_i] * 6, _sz),
    "attn_bwd_fused": ([_vp] * 10 + [_sz] + [_i] * 7 + [_f, _vp], _i),
    "attn_fwd_jvp": ([_vp] * 10 + [_i] * 7 + [_f, _vp], _i),
    "attn_bwd_jvp_workspace_bytes": ([_i] * 6, _sz),
    "attn_bwd_jvp": ([_vp] * 19 + [_sz] + [_i] * 7 + [_f, _vp], _i),
    "piecewise_fwd": ([_vp] * 7 + [_i] * 7 + [_f, _i, _vp], _i),
    "piecewise_bwd_workspace_bytes": ([_i] * 6, _sz),
    "piecewise_bwd": ([_vp] * 14 + [_sz] + [_i] * 7 + [_f, _i, _vp], _i),
    "attn_merge_fwd": ([_vp] * 6 + [_i] * 5 + [_vp], _i),
    "attn_fwd_fp8": ([_vp] * 5 + [_i] * 6 + [_f, _vp], _i),
    "attn_merge_bwd": ([_vp] * 10 + [_i] * 5 + [_vp], _i),
    "ta_sync_status": ([_vp], _i),
    "ta_status_str": ([_i], ctypes.c_char_p),
    "ta_selftest_wait_timeout": ([_i, _vp], _i),
    "ta_profile_enable": ([_i], _i),
    "ta_profile_read": ([ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(_i), ctypes.POINTER(ctypes.c_double),
                         _i], _i),
    "ta_set_wait_timeout_ms": ([_i], None),
    "ta_fwd_kv_split": ([_i] * 9, _i),
    "ta_set_fwd_kv_split": ([_i], None),
    "ta_guard_build": ([], _i),
    "ta_guard_last": ([], ctypes.c_char_p),
    "ta_selftest_guard": ([_vp], _i),
}


class TAError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code
        self.status = STATUS.get(code, str(code))


def lib_path() -> str:
    return _LIB_PATH


def load(path: str | None = None):
    """Loads libtattn.so (built by __graft_entry__.build()); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libtattn.so not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)  # AttributeError if the symbol is missing
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, code: int):
    if code != 0:
        raise TAError(fn, code)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _prep(tensors, M_names, N_names):
    """Validates [B,H,S,D] CUDA tensors and returns (B, H, M, N, D, dtype code)."""
    first = tensors[M_names[0]]
    if first.dim() != 4:
        raise ValueError("tensors must be [B, H, S, D]")
    B, H, M, D = first.shape
    N = tensors[N_names[0]].shape[2]
    dt = first.dtype
    for name, t in tensors.items():
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dtype != dt:
            raise ValueError(f"{name} has dtype {t.dtype}, expected {dt}")
        rows = M if name in M_names else N
        if tuple(t.shape) != (B, H, rows, D):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {(B, H, rows, D)}")
    if dt not in _DT:
        raise ValueError(f"unsupported dtype {dt}")
    return B, H, M, N, D, _DT[dt]


def _scale(sm_scale):
    return -1.0 if sm_scale is None else float(sm_scale)


def attn_bwd_workspace_bytes(B, H, M, N, D, dtype=torch.bfloat16) -> int:
    return int(load().attn_bwd_workspace_bytes(B, H, M, N, D, _DT[dtype]))


def attn_bwd_fused_workspace_bytes(B, H, M, N, D, dtype=torch.bfloat16) -> int:
    return int(load().attn_bwd_fused_workspace_bytes(B, H, M, N, D, _DT[dtype]))


def attn_fwd(q, k, v, causal=False, sm_scale=None, o=None, lse=None, stream=None):
    lib = load()
    B, H, M, N, D, dt = _prep({"q": q, "k": k, "v": v}, ("q",), ("k", "v"))
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, M), device=q.device, dtype=torch.float32) if lse is None else lse
    _check("attn_fwd", lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, M, N, D, dt,
                                    int(bool(causal)), _scale(sm_scale), _stream(stream)))
    return o, lse


def attn_bwd(q, k, v, o, lse, do, causal=False, sm_scale=None, dq=None, dk=None, dv=None, ws=None,
             stream=None):
    lib = load()
    B, H, M, N, D, dt = _prep({"q": q, "k": k, "v": v, "o": o, "do": do}, ("q", "o", "do"), ("k", "v"))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nws = int(lib.attn_bwd_workspace_bytes(B, H, M, N, D, dt))
    if ws is None:
        ws = torch.empty(max(nws, 16), device=q.device, dtype=torch.uint8)
    _check("attn_bwd", lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do), _ptr(dq),
                                    _ptr(dk), _ptr(dv), _ptr(ws), ws.numel() * ws.element_size(), B, H, M, N,
                                    D, dt, int(bool(causal)), _scale(sm_scale), _stream(stream)))
    return dq, dk, dv


def attn_bwd_fused(q, k, v, o, lse, do, causal=False, sm_scale=None, dq=None, dk=None, dv=None, ws=None,
                   stream=None):
    """attn_bwd in one key-stationary pass (five matmuls per block pair; dq
    summed in fp32 with atomics).  D = 128, float16/bfloat16."""
    lib = load()
    B, H, M, N, D, dt = _prep({"q": q, "k": k, "v": v, "o": o, "do": do}, ("q", "o", "do"), ("k", "v"))
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nws = int(lib.attn_bwd_fused_workspace_bytes(B, H, M, N, D, dt))
    if ws is None:
        ws = torch.empty(max(nws, 16), device=q.device, dtype=torch.uint8)
    _check("attn_bwd_fused", lib.attn_bwd_fused(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(do),
                                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws),
                                                ws.numel() * ws.element_size(), B, H, M, N, D, dt,
                                                int(bool(causal)), _scale(sm_scale), _stream(stream)))
    return dq, dk, dv


def attn_fwd_jvp(q, k, v, tq, tk, tv, causal=False, sm_scale=None, with_tlse=False, stream=None):
    """Returns (o, lse, to), or (o, lse, to, tlse) with with_tlse=True (tlse =
    the tangent of lse along (tq, tk))."""
    lib = load()
    B, H, M, N, D, dt = _prep({"q": q, "k": k, "v": v, "tq": tq, "tk": tk, "tv": tv}, ("q", "tq"),
                              ("k", "v", "tk", "tv"))
    o = torch.empty_like(q)
    to = torch.empty_like(q)
    lse = torch.empty((B, H, M), device=q.device, dtype=torch.float32)
    tlse = torch.empty_like(lse) if with_tlse else None
    _check("attn_fwd_jvp", lib.attn_fwd_jvp(_ptr(q), _ptr(k), _ptr(v), _ptr(tq), _ptr(tk), _ptr(tv), _ptr(o),
                                            _ptr(lse), _ptr(to), _ptr(tlse), B, H, M, N, D, dt,
                                            int(bool(causal)), _scale(sm_scale), _stream(stream)))
    return (o, lse, to, tlse) if with_tlse else (o, lse, to)


def attn_bwd_jvp(q, k, v, tq, tk, tv, o, lse, to, tlse, do, dto, causal=False, sm_scale=None, ws=None,
                 stream=None):
    """Backward of attn_fwd_jvp: gradients of <do, o> + <dto, to> with respect
    to (q, k, v, tq, tk, tv); o, lse, to, tlse are attn_fwd_jvp's outputs
    (with_tlse=True)."""
    lib = load()
    B, H, M, N, D, dt = _prep({"q": q, "k": k, "v": v, "tq": tq, "tk": tk, "tv": tv, "o": o, "to": to, "do": do,
                               "dto": dto}, ("q", "tq", "o", "to", "do", "dto"), ("k", "v", "tk", "tv"))
    _lse_of("lse", lse, B, H, M, q.device)
    _lse_of("tlse", tlse, B, H, M, q.device)
    grads = [torch.empty_like(x) for x in (q, k, v, tq, tk, tv)]
    nws = int(lib.attn_bwd_jvp_workspace_bytes(B, H, M, N, D, dt))
    if ws is None:
        ws = torch.empty(max(nws, 16), device=q.device, dtype=torch.uint8)
    _check("attn_bwd_jvp", lib.attn_bwd_jvp(*(_ptr(x) for x in (q, k, v, tq, tk, tv, o, lse, to, tlse, do, dto)),
                                            *(_ptr(g) for g in grads), _ptr(ws), ws.numel() * ws.element_size(),
                                            B, H, M, N, D, dt, int(bool(causal)), _scale(sm_scale),
                                            _stream(stream)))
    return tuple(grads)


def piecewise_fwd(q1, k1, q2, k2, v, w, causal=False, sm_scale=None, stream=None):
    lib = load()
    B, H, M, N, D, dt = _prep({"q1": q1, "k1": k1, "q2": q2, "k2": k2, "v": v}, ("q1", "q2"), ("k1", "k2", "v"))
    o = torch.empty_like(q1)
    lse = torch.empty((B, H, M), device=q1.device, dtype=torch.float32)
    _check("piecewise_fwd", lib.piecewise_fwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), _ptr(o),
                                              _ptr(lse), B, H, M, N, D, dt, int(bool(causal)),
                                              _scale(sm_scale), int(w), _stream(stream)))
    return o, lse


def piecewise_bwd(q1, k1, q2, k2, v, o, lse, do, w, causal=False, sm_scale=None, ws=None, stream=None):
    lib = load()
    B, H, M, N, D, dt = _prep({"q1": q1, "k1": k1, "q2": q2, "k2": k2, "v": v, "o": o, "do": do},
                              ("q1", "q2", "o", "do"), ("k1", "k2", "v"))
    dq1, dq2 = torch.empty_like(q1), torch.empty_like(q2)
    dk1, dk2, dv = torch.empty_like(k1), torch.empty_like(k2), torch.empty_like(v)
    nws = int(lib.piecewise_bwd_workspace_bytes(B, H, M, N, D, dt))
    if ws is None:
        ws = torch.empty(max(nws, 16), device=q1.device, dtype=torch.uint8)
    _check("piecewise_bwd", lib.piecewise_bwd(_ptr(q1), _ptr(k1), _ptr(q2), _ptr(k2), _ptr(v), _ptr(o),
                                              _ptr(lse), _ptr(do), _ptr(dq1), _ptr(dk1), _ptr(dq2), _ptr(dk2),
                                              _ptr(dv), _ptr(ws), ws.numel() * ws.element_size(), B, H, M, N,
                                              D, dt, int(bool(causal)), _scale(sm_scale), int(w),
                                              _stream(stream)))
    return dq1, dk1, dq2, dk2, dv


def attn_fwd_fp8(q, k, vt, causal=False, sm_scale=None, stream=None):
    """e5m2 forward: q [B,H,M,D], k [B,H,N,D], vt = V transposed [B,H,D,N], all
    torch.float8_e5m2 CUDA tensors; returns (o [B,H,M,D] e5m2, lse fp32)."""
    lib = load()
    f8 = torch.float8_e5m2
    for name, t in (("q", q), ("k", k), ("vt", vt)):
        if t.dtype != f8 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D float8_e5m2 CUDA tensor")
    B, H, M, D = q.shape
    N = k.shape[2]
    if tuple(k.shape) != (B, H, N, D) or tuple(vt.shape) != (B, H, D, N):
        raise ValueError("expected k [B,H,N,D] and vt [B,H,D,N]")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, M), device=q.device, dtype=torch.float32)
    _check("attn_fwd_fp8", lib.attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(vt), _ptr(o), _ptr(lse), B, H, M, N, D,
                                            int(bool(causal)), _scale(sm_scale), _stream(stream)))
    return o, lse


def _lse_of(name, t, B, H, M, dev):
    if t.dtype != torch.float32 or tuple(t.shape) != (B, H, M) or not t.is_contiguous() or t.device != dev:
        raise ValueError(f"{name} must be a contiguous float32 [B, H, M] tensor on {dev}")


def merge_fwd(o1, lse1, o2, lse2, o=None, lse=None, stream=None):
    """Merge of two partial attention states over disjoint key sets:
    returns (o, lse) with O = (e^L1 O1 + e^L2 O2) / e^L, L = ln(e^L1 + e^L2)."""
    lib = load()
    B, H, M, _, D, dt = _prep({"o1": o1, "o2": o2}, ("o1", "o2"), ("o1",))
    _lse_of("lse1", lse1, B, H, M, o1.device)
    _lse_of("lse2", lse2, B, H, M, o1.device)
    o = torch.empty_like(o1) if o is None else o
    lse = torch.empty_like(lse1) if lse is None else lse
    _check("attn_merge_fwd", lib.attn_merge_fwd(_ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2), _ptr(o), _ptr(lse),
                                                B, H, M, D, dt, _stream(stream)))
    return o, lse


def merge_bwd(o1, lse1, o2, lse2, do, dlse=None, stream=None):
    """Backward of merge_fwd: returns (do1, dlse1, do2, dlse2); dlse None = 0."""
    lib = load()
    B, H, M, _, D, dt = _prep({"o1": o1, "o2": o2, "do": do}, ("o1", "o2", "do"), ("o1",))
    _lse_of("lse1", lse1, B, H, M, o1.device)
    _lse_of("lse2", lse2, B, H, M, o1.device)
    if dlse is not None:
        _lse_of("dlse", dlse, B, H, M, o1.device)
    do1, do2 = torch.empty_like(o1), torch.empty_like(o2)
    dl1, dl2 = torch.empty_like(lse1), torch.empty_like(lse2)
    _check("attn_merge_bwd", lib.attn_merge_bwd(_ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2), _ptr(do), _ptr(dlse),
                                                _ptr(do1), _ptr(dl1), _ptr(do2), _ptr(dl2), B, H, M, D, dt,
                                                _stream(stream)))
    return do1, dl1, do2, dl2


def sync_status(stream=None) -> str:
    """Synchronises the stream and returns the device error status name."""
    return STATUS.get(int(load().ta_sync_status(_stream(stream))), "?")


def selftest_wait_timeout(timeout_ms: int = 20, stream=None) -> str:
    _check("ta_selftest_wait_timeout", load().ta_selftest_wait_timeout(int(timeout_ms), _stream(stream)))
    return sync_status(stream)


def set_wait_timeout_ms(ms: int):
    load().ta_set_wait_timeout_ms(int(ms))


_ENTRY = {"attn_fwd": 0, "piecewise_fwd": 1, "attn_fwd_jvp": 2}
_SPLIT_MODE = {"auto": 0, "never": 1, "always": 2}


def fwd_kv_split(entry: str, B: int, H: int, M: int, N: int, D: int, dtype, causal: bool, num_sms: int = 0) -> int:
    """CTAs per 128-row query tile that forward entry point `entry` launches
    for this problem (2: key split into a two-CTA cluster, 1: not split) on a
    GPU with `num_sms` SMs (0: the current device's)."""
    r = load().ta_fwd_kv_split(_ENTRY[entry], B, H, M, N, D, _DT[dtype], int(bool(causal)), int(num_sms))
    if r == 0:
        raise ValueError("invalid problem for ta_fwd_kv_split")
    return r


def set_fwd_kv_split(mode: str):
    """Process-wide key-split choice of the one-query-tile forward: "auto"
    (the library's estimate, the default), "never" or "always"."""
    load().ta_set_fwd_kv_split(_SPLIT_MODE[mode])


def profile_enable(on: bool = True):
    load().ta_profile_enable(int(bool(on)))


def profile_read() -> dict:
    """{kernel name: (launches, total_ms)} for launches since profile_enable(True)."""
    lib = load()
    cap = 32
    names = (ctypes.c_char_p * cap)()
    launches = (ctypes.c_int * cap)()
    ms = (ctypes.c_double * cap)()
    n = lib.ta_profile_read(names, launches, ms, cap)
    if n < 0:
        raise TAError("ta_profile_read", 4)
    return {names[i].decode(): (launches[i], ms[i]) for i in range(min(n, cap))}
