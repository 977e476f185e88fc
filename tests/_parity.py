"""Helpers shared by the GPU parity tests: seeded inputs, oracle calls and the
tolerance checks (max_abs against the fp64 oracle, max_rel against max|ref|
reported alongside)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth_inputs as si

# max_abs tolerances for unit-normal inputs
TOL = {"O_f16": 1e-2, "O_bf16": 2e-2, "L": 1e-3, "grad": 5e-2, "tO": 5e-2}


def o_tol(dtype: str) -> float:
    return TOL["O_bf16"] if dtype == "bf16" else TOL["O_f16"]


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def compare(name, got, ref, tol):
    """Asserts max|got - ref| <= tol (same shapes; non-finite entries must match)."""
    g = to_np(got) if hasattr(got, "detach") else np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    fin_r = np.isfinite(r)
    assert np.array_equal(fin_r, np.isfinite(g)), f"{name}: non-finite pattern differs"
    if not fin_r.any():
        return 0.0, 0.0
    assert np.array_equal(g[~fin_r], r[~fin_r]), f"{name}: infinities differ"
    max_abs = float(np.abs(g[fin_r] - r[fin_r]).max())
    scale = float(np.abs(r[fin_r]).max())
    max_rel = max_abs / scale if scale > 0 else max_abs
    assert max_abs <= tol, f"{name}: max_abs {max_abs:.3e} > {tol:.1e} (max_rel {max_rel:.3e})"
    return max_abs, max_rel


def heads_of(x, heads):
    """Stack the selected (b, h) slices of a [B, H, ...] array/tensor."""
    a = to_np(x) if hasattr(x, "detach") else np.asarray(x)
    return np.stack([a[b, h] for (b, h) in heads])


def inputs(B, H, M, N, D, dtype, workload, names):
    cpu = si.attention_inputs(B, H, M, N, D, dtype, workload, names=names)
    return cpu, {k: v.cuda() for k, v in cpu.items()}


def all_heads(B, H):
    return [(b, h) for b in range(B) for h in range(H)]


def sample_heads(B, H, n=2):
    hs = all_heads(B, H)
    if len(hs) <= n:
        return hs
    pick = [hs[0], hs[-1]] + [hs[len(hs) // 2]][: max(0, n - 2)]
    return pick[:n]
