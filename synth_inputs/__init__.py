"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no attention arithmetic: it only turns (seed, shape, dtype)
into tensors of i.i.d. standard-normal values, so that the GPU path and the
fp64 oracle consume exactly the same dtype-rounded bits.

Generator (published definitions, restated):
  * SplitMix64 (S. Vigna, "Further scramblings of Marsaglia's xorshift
    generators", 2014/2017): a counter-based 64-bit mixer.  Element counter
    c gives z = mix64(seed + (c + 1) * 0x9E3779B97F4A7C15).
  * Box-Muller transform (G. Box, M. Muller, Ann. Math. Stat. 29, 1958): two
    uniforms u1 in (0, 1], u2 in [0, 1) give two independent N(0, 1) values
    r cos(2 pi u2), r sin(2 pi u2) with r = sqrt(-2 ln u1).
The fp64 normals are rounded to the requested dtype by torch's CPU
conversion (round-to-nearest-even through fp32); both sides then read that
one rounded tensor.

Seed convention: tensor index t of workload w gets seed 1000 * w + t, in the
style of the JVP test script of "Triton fused attention tutorial, updated
with JVP support" (one seed per tensor, ``seed + ix``).
"""
from __future__ import annotations

import numpy as np
import torch

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

DTYPES = {
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "f32": torch.float32,
    "f64": torch.float64,
    "e5m2": torch.float8_e5m2,
}


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs number start .. start+count-1 of the SplitMix64 stream of `seed`."""
    ctr = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + ctr * _GOLDEN
        return _mix64(state)


def normal_f64(seed: int, n: int) -> np.ndarray:
    """n i.i.d. N(0,1) doubles from the counter-based stream of `seed`."""
    out = np.empty(n, dtype=np.float64)
    npairs = (n + 1) // 2
    two53 = np.float64(2.0 ** -53)
    for p0 in range(0, npairs, _CHUNK):
        cnt = min(_CHUNK, npairs - p0)
        z = splitmix64(seed, 2 * p0, 2 * cnt)
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * two53
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * two53
        r = np.sqrt(-2.0 * np.log(u1))
        ang = 2.0 * np.pi * u2
        pair = np.empty(2 * cnt, dtype=np.float64)
        pair[0::2] = r * np.cos(ang)
        pair[1::2] = r * np.sin(ang)
        lo = 2 * p0
        hi = min(n, lo + 2 * cnt)
        out[lo:hi] = pair[: hi - lo]
    return out


def randn(shape, dtype: str, seed: int) -> torch.Tensor:
    """CPU tensor of the given shape, N(0,1) entries rounded to `dtype`."""
    n = int(np.prod(shape)) if len(shape) else 1
    x = torch.from_numpy(normal_f64(seed, n)).reshape(tuple(shape))
    if dtype in ("f16", "bf16", "e5m2"):  # through fp32, round to nearest even
        return x.to(torch.float32).to(DTYPES[dtype]).contiguous()
    return x.to(DTYPES[dtype]).contiguous()


def seed_for(workload: int, index: int) -> int:
    return 1000 * workload + index


# Workloads with the shapes of the benchmark configurations: (B, H, M, N, D),
# dtype, causal, mode, piecewise threshold w.
WORKLOADS = {
    1: dict(name="fwd+bwd fp16 non-causal B1 H2 S128 D64", B=1, H=2, M=128, N=128, D=64,
            dtype="f16", causal=False, mode="fwdbwd", w=None),
    2: dict(name="fwd+bwd bf16 causal B4 H16 S2048 D128", B=4, H=16, M=2048, N=2048, D=128,
            dtype="bf16", causal=True, mode="fwdbwd", w=None),
    3: dict(name="fwd+bwd bf16 causal B1 H32 S8192 D128", B=1, H=32, M=8192, N=8192, D=128,
            dtype="bf16", causal=True, mode="fwdbwd", w=None),
    4: dict(name="fwd+jvp fp16 B2 H8 S1024 D64", B=2, H=8, M=1024, N=1024, D=64,
            dtype="f16", causal=None, mode="jvp", w=None),
    5: dict(name="piecewise fwd+bwd bf16 causal B2 H16 S4096 D64 w512", B=2, H=16, M=4096, N=4096,
            D=64, dtype="bf16", causal=True, mode="piecewise", w=512),
}


def attention_inputs(B, H, M, N, D, dtype, workload, names=("q", "k", "v", "do")):
    """Dict of named CPU tensors; rows of q/do have length M, of k/v length N."""
    out = {}
    for idx, name in enumerate(names):
        rows = M if name in ("q", "do", "tq", "dto", "q1", "q2") else N
        out[name] = randn((B, H, rows, D), dtype, seed_for(workload, idx))
    return out
