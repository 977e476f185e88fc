"""Writes tests/golden/oracle_tiny.json: the oracle's outputs on tiny seeded
problems (standard causal, piecewise, the JVP with tL and its backward, and
the two-state merge with its backward), so that any later change to the
oracle's arithmetic shows up as a diff of this file.

It calls only the oracle and the seeded input generator.  The pages print no
attention values (their printed numbers depend on torch's CUDA RNG), so these
are regression values, not page values.  Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth_inputs as si  # noqa: E402


def main():
    x = si.attention_inputs(1, 1, 5, 7, 4, "f64", 90, names=("q", "k", "v", "do"))
    q, k, v, do = (x[n][0, 0].numpy() for n in ("q", "k", "v", "do"))
    O, L = oracle.attention_fwd(q, k, v, True, 0.5)
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, True, 0.5)
    y = si.attention_inputs(1, 1, 6, 6, 4, "f64", 91, names=("q1", "k1", "q2", "k2", "v", "do"))
    a = [y[n][0, 0].numpy() for n in ("q1", "k1", "q2", "k2", "v", "do")]
    Op, Lp = oracle.piecewise_fwd(*a[:5], True, 0.5, 2)
    gp = oracle.piecewise_bwd(*a, True, 0.5, 2)
    names = ("q", "k", "v", "tq", "tk", "tv", "do", "dto")
    z = si.attention_inputs(1, 1, 6, 5, 4, "f64", 92, names=names)
    j = [z[n][0, 0].numpy() for n in names]
    Oj, Lj, tO = oracle.attention_jvp(*j[:6], True, 0.5)
    tL = oracle.attention_jvp_tl(j[0], j[1], j[3], j[4], True, 0.5)
    gj = oracle.attention_jvp_bwd(*j, True, 0.5)
    mo = si.attention_inputs(1, 1, 6, 6, 4, "f64", 93, names=("q", "k", "do"))
    o1, o2, dom = (mo[n][0, 0].numpy() for n in ("q", "k", "do"))
    ml = si.attention_inputs(1, 1, 6, 6, 2, "f64", 94, names=("q", "k"))
    l1, l2 = (ml[n][0, 0].numpy()[:, 0] for n in ("q", "k"))
    l1[0] = -float("inf")  # a row whose first part saw no key
    Om, Lm = oracle.lse_merge_fwd(o1, l1, o2, l2)
    gm = oracle.lse_merge_bwd(o1, l1, o2, l2, dom, l2 * 0.5)
    out = {
        "standard": {"M": 5, "N": 7, "D": 4, "causal": True, "sm_scale": 0.5, "workload_seed_base": 90,
                     "O": O.tolist(), "L": L.tolist(), "dq": dq.tolist(), "dk": dk.tolist(), "dv": dv.tolist()},
        "piecewise": {"M": 6, "N": 6, "D": 4, "causal": True, "sm_scale": 0.5, "w": 2, "workload_seed_base": 91,
                      "O": Op.tolist(), "L": Lp.tolist(),
                      "grads": [g.tolist() for g in gp]},
        "jvp": {"M": 6, "N": 5, "D": 4, "causal": True, "sm_scale": 0.5, "workload_seed_base": 92,
                "O": Oj.tolist(), "L": Lj.tolist(), "tO": tO.tolist(), "tL": tL.tolist(),
                "grads": [g.tolist() for g in gj]},
        "merge": {"M": 6, "D": 4, "workload_seed_base": [93, 94], "l1_row0": "-inf", "dl": "0.5 * l2",
                  "O": Om.tolist(), "L": [x if x != float("-inf") else "-inf" for x in Lm.tolist()],
                  "grads": [[x if x != float("-inf") else "-inf" for x in (g.ravel().tolist())] for g in gm]},
    }
    with open(os.path.join(HERE, "oracle_tiny.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
