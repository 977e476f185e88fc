"""The oracle still reproduces its committed tiny-problem outputs
(tests/golden/oracle_tiny.json, written by tests/golden/make_golden.py)."""
import json
import os

import numpy as np

import oracle
import synth_inputs as si

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_tiny.json")


def test_oracle_matches_golden_tiny_problems():
    g = json.load(open(GOLD))
    s = g["standard"]
    x = si.attention_inputs(1, 1, s["M"], s["N"], s["D"], "f64", s["workload_seed_base"], names=("q", "k", "v", "do"))
    q, k, v, do = (x[n][0, 0].numpy() for n in ("q", "k", "v", "do"))
    O, L = oracle.attention_fwd(q, k, v, s["causal"], s["sm_scale"])
    np.testing.assert_allclose(O, s["O"], atol=1e-14)
    np.testing.assert_allclose(L, s["L"], atol=1e-14)
    for got, name in zip(oracle.attention_bwd(q, k, v, do, s["causal"], s["sm_scale"]), ("dq", "dk", "dv")):
        np.testing.assert_allclose(got, s[name], atol=1e-14)
    p = g["piecewise"]
    y = si.attention_inputs(1, 1, p["M"], p["N"], p["D"], "f64", p["workload_seed_base"],
                            names=("q1", "k1", "q2", "k2", "v", "do"))
    a = [y[n][0, 0].numpy() for n in ("q1", "k1", "q2", "k2", "v", "do")]
    Op, Lp = oracle.piecewise_fwd(*a[:5], p["causal"], p["sm_scale"], p["w"])
    np.testing.assert_allclose(Op, p["O"], atol=1e-14)
    for got, ref in zip(oracle.piecewise_bwd(*a, p["causal"], p["sm_scale"], p["w"]), p["grads"]):
        np.testing.assert_allclose(got, ref, atol=1e-14)


def _num(x):
    return np.array([float("-inf") if v == "-inf" else v for v in np.ravel(x)], dtype=np.float64)


def test_oracle_matches_golden_jvp_and_merge():
    g = json.load(open(GOLD))
    j = g["jvp"]
    names = ("q", "k", "v", "tq", "tk", "tv", "do", "dto")
    z = si.attention_inputs(1, 1, j["M"], j["N"], j["D"], "f64", j["workload_seed_base"], names=names)
    a = [z[n][0, 0].numpy() for n in names]
    O, L, tO = oracle.attention_jvp(*a[:6], j["causal"], j["sm_scale"])
    tL = oracle.attention_jvp_tl(a[0], a[1], a[3], a[4], j["causal"], j["sm_scale"])
    for got, ref in ((O, j["O"]), (L, j["L"]), (tO, j["tO"]), (tL, j["tL"])):
        np.testing.assert_allclose(got, ref, atol=1e-14)
    for got, ref in zip(oracle.attention_jvp_bwd(*a, j["causal"], j["sm_scale"]), j["grads"]):
        np.testing.assert_allclose(got, ref, atol=1e-13)
    m = g["merge"]
    mo = si.attention_inputs(1, 1, m["M"], m["M"], m["D"], "f64", m["workload_seed_base"][0], names=("q", "k", "do"))
    o1, o2, do = (mo[n][0, 0].numpy() for n in ("q", "k", "do"))
    ml = si.attention_inputs(1, 1, m["M"], m["M"], 2, "f64", m["workload_seed_base"][1], names=("q", "k"))
    l1, l2 = (ml[n][0, 0].numpy()[:, 0].copy() for n in ("q", "k"))
    l1[0] = -np.inf
    Om, Lm = oracle.lse_merge_fwd(o1, l1, o2, l2)
    np.testing.assert_allclose(Om, m["O"], atol=1e-14)
    np.testing.assert_allclose(Lm, _num(m["L"]), atol=1e-14)
    for got, ref in zip(oracle.lse_merge_bwd(o1, l1, o2, l2, do, l2 * 0.5), m["grads"]):
        np.testing.assert_allclose(np.ravel(got), _num(ref), atol=1e-14)
