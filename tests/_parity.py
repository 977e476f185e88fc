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


def assert_same_up_to_summation_order(name, got, ref):
    """Two results of the same call that may differ only in the order of an
    fp32 sum (the fused backward adds dQ's per-key-tile contributions with
    atomics): equal up to one unit in the last place of their 16-bit type,
    i.e. |got - ref| <= 2 u |ref| (u the unit roundoff) plus 2^-20 for
    values near zero, where the fp32 sums' own difference shows."""
    u = {torch.bfloat16: ROUND_U["bf16"], torch.float16: ROUND_U["f16"], torch.float32: 2.0 ** -24}[got.dtype]
    a, b = got.detach().double(), ref.detach().double()
    assert a.shape == b.shape, f"{name}: shape {tuple(a.shape)} vs {tuple(b.shape)}"
    excess = float(((a - b).abs() - 2 * u * b.abs() - 2.0 ** -20).max()) if a.numel() else 0.0
    assert excess <= 0, f"{name}: differs by more than the last place (excess {excess:.3e})"


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


def jvp_bwd_bounds(cpu, causal, u, sm_scale=None, heads=None):
    """Element-wise error bounds for the backward of the JVP (beyond a flat
    unit-scale tolerance), per head, from the quantities the kernels round:

    * the row constants delta2 = <dO,O> + <dtO,tO> and eps = <dtO,O> are
      formed from the stored 16-bit O and tO, and tO already carries the
      rounding of P o T before its product with V: over the D terms of each
      row, r_d2 = u rms-sum(dO O, dtO tO, dtO (P o |T|) |V|) and
      r_e = u rms-sum(dtO O), so dS moves by P (r_d2 + |T - mu| r_e) and dT by
      P r_e, and every gradient sums those moves over its keys or queries;
    * P, tP, dS and dT are rounded to 16 bits before the gradient MMAs (u of
      each term) and every result once more on output.
    The roundings are independent, so sums combine as the root of the summed
    squares; the bound is 4 times that (a 4-sigma allowance).  It matters
    where the exact gradients cancel (one key: P = 1) and the key-side
    gradients sum the rows' rounding over every query.
    Returns {name: [B, H, ...] bound} for dq, dk, dv, dtq, dtk, dtv (heads not
    listed stay 0)."""
    import oracle
    x = {n: cpu[n].double().numpy() for n in ("q", "k", "v", "tq", "tk", "tv", "do", "dto")}
    B, H, M, D = x["q"].shape
    N = x["k"].shape[2]
    s = oracle.default_scale(D, sm_scale)
    keep = oracle.allowed_mask(M, N, causal)
    out = {n: np.zeros((B, H) + (M if n in ("dq", "dtq") else N, D)) for n in ("dq", "dk", "dv", "dtq", "dtk", "dtv")}
    for b in range(B):
        for h in range(H):
            if heads is not None and (b, h) not in heads:
                continue
            q, k, v, tq, tk, tv, do, dto = (x[n][b, h] for n in ("q", "k", "v", "tq", "tk", "tv", "do", "dto"))
            O, L, tO = oracle.attention_jvp(q, k, v, tq, tk, tv, causal, sm_scale)
            fin = np.isfinite(L)
            S = np.where(keep, s * q @ k.T, -np.inf)
            P = np.zeros_like(S)
            P[fin] = np.exp(S[fin] - L[fin, None])
            T = np.where(keep, s * (tq @ k.T + q @ tk.T), 0.0)
            mu = (P * T).sum(axis=1)
            tP = P * (T - mu[:, None])
            dT = P * (dto @ v.T - (dto * O).sum(axis=1)[:, None])
            dS = P * (do @ v.T + dto @ tv.T - ((do * O).sum(axis=1) + (dto * tO).sum(axis=1))[:, None]) \
                + (T - mu[:, None]) * dT
            r_d2 = u * np.sqrt(((do * O) ** 2 + (dto * tO) ** 2 + (dto * ((P * np.abs(T)) @ np.abs(v))) ** 2)
                               .sum(axis=1))
            r_e = u * np.sqrt(((dto * O) ** 2).sum(axis=1))
            mdS = P * (r_d2[:, None] + np.abs(T - mu[:, None]) * r_e[:, None]) + u * np.abs(dS)
            mdT = P * r_e[:, None] + u * np.abs(dT)
            g = oracle.attention_jvp_bwd(q, k, v, tq, tk, tv, do, dto, causal, sm_scale)
            # independent roundings add in quadrature over the summed keys or
            # queries: a 4-sigma allowance on the root of the summed squares
            rs = lambda a, bb: 4.0 * np.sqrt(a ** 2 @ bb ** 2)
            out["dq"][b, h] = s * (rs(mdS, k) + rs(mdT, tk)) + u * np.abs(g[0])
            out["dk"][b, h] = s * (rs(mdS.T, q) + rs(mdT.T, tq)) + u * np.abs(g[1])
            out["dv"][b, h] = u * (rs(P.T, do) + rs(np.abs(tP).T, dto)) + u * np.abs(g[2])
            out["dtq"][b, h] = s * rs(mdT, k) + u * np.abs(g[3])
            out["dtk"][b, h] = s * rs(mdT.T, q) + u * np.abs(g[4])
            out["dtv"][b, h] = u * rs(P.T, dto) + u * np.abs(g[5])
    return out


def compare_bounded(name, got, ref, tol, bound):
    """Asserts |got - ref| <= tol + bound element by element (same shapes)."""
    g = to_np(got) if hasattr(got, "detach") else np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    excess = float((np.abs(g - r) - tol - bound).max())
    assert excess <= 0, f"{name}: error exceeds {tol:.1e} + its bound by {excess:.3e}"
