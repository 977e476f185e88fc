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
