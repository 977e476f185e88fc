"""Runs the library's entry points on one of the synthetic workloads for a
number of steps: the command line used for profiling (ncu) and timing runs.

  python -m tiled_attention_tcgen05_gb300.run_workload --workload 3 --steps 2 --warmup 1

Workloads (synth_inputs.WORKLOADS): 1 fwd+bwd fp16 B1 H2 S128 D64 non-causal;
2 fwd+bwd bf16 causal B4 H16 S2048 D128; 3 fwd+bwd bf16 causal B1 H32 S8192
D128; 4 JVP forward (with tL) and the backward of the JVP, fp16 B2 H8 S1024
D64 (--causal 0/1); 5 piecewise fwd+bwd bf16 causal B2 H16 S4096 D64 w=512.
--shape B,H,S,D replaces the workload's sizes; --op merge / --op fp8 runs the
merge (forward and backward) or the e5m2 forward instead; --kv-split sets
the key split of the one-query-tile forward.  Prints the mean milliseconds per
step.
"""
from __future__ import annotations

import argparse
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch  # noqa: E402

import synth_inputs as si  # noqa: E402
import tiled_attention_tcgen05_gb300 as ta  # noqa: E402


def make_op_step(op: str, shape=None):
    """Steps of the entry points that are not a fwd+bwd workload, on the
    benchmark's shape (B1 H32 S8192 D128) unless `shape` is given:
    merge (attn_merge_fwd + attn_merge_bwd, bf16) and fp8 (attn_fwd_fp8,
    e5m2, causal)."""
    B, H, S, D = shape if shape is not None else (1, 32, 8192, 128)
    if op == "merge":
        o1, o2, do = (si.randn((B, H, S, D), "bf16", si.seed_for(6, i)).cuda() for i in range(3))
        l1, l2 = (si.randn((B, H, S), "f32", si.seed_for(6, 3 + i)).cuda() * 3 for i in range(2))

        def step():
            ta.merge_fwd(o1, l1, o2, l2)
            ta.merge_bwd(o1, l1, o2, l2, do)
        return step
    if op == "fp8":
        q = si.randn((B, H, S, D), "e5m2", si.seed_for(7, 0)).cuda()
        k = si.randn((B, H, S, D), "e5m2", si.seed_for(7, 1)).cuda()
        vt = si.randn((B, H, D, S), "e5m2", si.seed_for(7, 2)).cuda()
        return lambda: ta.attn_fwd_fp8(q, k, vt, True)
    raise ValueError(f"unknown op {op}")


def make_step(wid: int, causal_override=None, shape=None):
    w = si.WORKLOADS[wid]
    B, H, M, N, D, dt = w["B"], w["H"], w["M"], w["N"], w["D"], w["dtype"]
    causal = w["causal"] if causal_override is None else bool(causal_override)
    if shape is not None:
        B, H, M, D = shape
        N = M
    if w["mode"] == "jvp":
        names = ("q", "k", "v", "tq", "tk", "tv", "do", "dto")
    elif w["mode"] == "piecewise":
        names = ("q1", "k1", "q2", "k2", "v", "do")
    else:
        names = ("q", "k", "v", "do")
    x = {n: t.cuda() for n, t in si.attention_inputs(B, H, M, N, D, dt, wid, names=names).items()}
    if w["mode"] == "jvp":
        def jvp_step():
            o, lse, to, tlse = ta.attn_fwd_jvp(*(x[n] for n in names[:6]), causal=bool(causal), with_tlse=True)
            ta.attn_bwd_jvp(*(x[n] for n in names[:6]), o, lse, to, tlse, x["do"], x["dto"], causal=bool(causal))
        return jvp_step
    if w["mode"] == "piecewise":
        def step():
            o, lse = ta.piecewise_fwd(x["q1"], x["k1"], x["q2"], x["k2"], x["v"], w["w"], causal)
            ta.piecewise_bwd(x["q1"], x["k1"], x["q2"], x["k2"], x["v"], o, lse, x["do"], w["w"], causal)
        return step

    def step():
        o, lse = ta.attn_fwd(x["q"], x["k"], x["v"], causal)
        ta.attn_bwd(x["q"], x["k"], x["v"], o, lse, x["do"], causal)
    return step


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", type=int, default=3)
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--causal", type=int, default=None)
    ap.add_argument("--shape", type=str, default=None, help="B,H,S,D instead of the workload's own (M = N = S)")
    ap.add_argument("--op", type=str, default=None, choices=["merge", "fp8"],
                    help="time attn_merge_fwd/bwd or attn_fwd_fp8 instead of a workload")
    ap.add_argument("--kv-split", type=str, default="auto", choices=["auto", "never", "always"],
                    help="key split of the one-query-tile forward (JVP, D = 128 piecewise)")
    a = ap.parse_args()
    ta.load()
    ta.set_fwd_kv_split(a.kv_split)
    shape = tuple(int(x) for x in a.shape.split(",")) if a.shape else None
    step = make_op_step(a.op, shape) if a.op else make_step(a.workload, a.causal, shape)
    for _ in range(a.warmup):
        step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.steps):
        step()
    e1.record()
    status = ta.sync_status()
    name = f"op {a.op}" if a.op else f"workload {a.workload}"
    print(f"{name}: {e0.elapsed_time(e1) / max(1, a.steps):.3f} ms/step, status {status}")
    return 0 if status == "TA_OK" else 1


if __name__ == "__main__":
    sys.exit(main())
