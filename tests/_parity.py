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


def jvp_grad_tol(dtype: str) -> float:
    """Gradients of the backward of the JVP.  Its row constants
    delta2 = <dO, O> + <dtO, tO> and eps = <dtO, O> are formed from the two
    stored, rounded outputs O and tO (as the plain backward forms delta from
    the stored O), so where the exact dS and dT cancel (one visible key: P = 1)
    the rounding of both outputs remains: about u sqrt(D) s max|K| per term,
    u the unit roundoff.  Twice the plain gradients' 5e-2 for bf16 (u = 2^-8);
    fp16 (u = 2^-11) keeps 5e-2."""
    return 1e-1 if dtype == "bf16" else TOL["grad"]


def to_np(t) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


# unit roundoff of the 16-bit output types (round to nearest even)
ROUND_U = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}


def compare(name, got, ref, tol, round_u=0.0):
    """Asserts |got - ref| <= tol + round_u |ref| element by element (same
    shapes; non-finite entries must match).  round_u > 0 adds the rounding of
    the stored result to its 16-bit type, which no implementation can avoid
    once |ref| is large (a sum over many rows); max_abs and max_rel are
    reported either way."""
    g = to_np(got) if hasattr(got, "detach") else np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    fin_r = np.isfinite(r)
    assert np.array_equal(fin_r, np.isfinite(g)), f"{name}: non-finite pattern differs"
    if not fin_r.any():
        return 0.0, 0.0
    assert np.array_equal(g[~fin_r], r[~fin_r]), f"{name}: infinities differ"
    err = np.abs(g[fin_r] - r[fin_r])
    max_abs = float(err.max())
    scale = float(np.abs(r[fin_r]).max())
    max_rel = max_abs / scale if scale > 0 else max_abs
    if round_u > 0:
        excess = float((err - tol - round_u * np.abs(r[fin_r])).max())
        assert excess <= 0, (f"{name}: error exceeds {tol:.1e} + {round_u:.2e} |ref| by {excess:.3e} "
                             f"(max_abs {max_abs:.3e}, max_rel {max_rel:.3e})")
    else:
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
