"""Benchmark: attention forward + backward, bf16, causal, B=1 H=32 M=N=8192 D=128.

One step = one pass of the whole hot path over one batch: attn_fwd (O, L)
then attn_bwd (dQ with delta, then dK/dV) on inputs resident in HBM.  The metric is
throughput in TFLOPS with the FLOP count 4*B*H*M*N*D for the forward, 2.5x
that for the backward, halved for causal (the benchmark harness of "Triton
fused attention tutorial, updated with JVP support", bench_flash_attention).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl {ours,reference}]
For N > 1 launch one process per GPU with torch.distributed.run; every rank
runs the same workload on its own GPU (independent heads: weak scaling, no
collective on the data path; one barrier and a max-reduction of the timing).
--impl reference times the fp64 CPU oracle on a bounded sample instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention fwd+bwd TFLOPS/GPU (bf16, causal) and % of GB300 dense tensor peak"
WORKLOAD = dict(B=1, H=32, M=8192, N=8192, D=128, dtype="bf16", causal=True)
WORKLOAD_NAME = "attention fwd+bwd bf16 causal B1 H32 M=N=8192 D128 (synthetic N(0,1), seeded)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def flops_fwd(B, H, M, N, D, causal):
    f = 4.0 * B * H * M * N * D
    return f * 0.5 if causal else f


def step_flops(w=WORKLOAD):
    f = flops_fwd(w["B"], w["H"], w["M"], w["N"], w["D"], w["causal"])
    return f * (1.0 + 2.5)


def kernel_algorithmic(name, w=WORKLOAD):
    """(bound, per-launch algorithmic FLOPs or bytes) of each library kernel.

    attn_fwd: the forward's two matmuls.  attn_bwd_fused: all five of the
    backward's matmuls (S^T recompute, dP^T, dV, dK, dQ^T).  The two-pass
    backward's attn_bwd_dkdv: four of them (S^T recompute, dP^T, dV, dK);
    attn_bwd_dq: the dQ matmul (its S and dP recomputes are extra work, not
    counted; in the two-pass backward it also forms delta from O and dO).
    bwd_delta: bytes of O and dO read plus delta written (attn_bwd_fused's
    delta pass, which also zeroes its fp32 dQ accumulator).  bwd_dq_convert: the accumulator read, dQ
    written."""
    f = flops_fwd(w["B"], w["H"], w["M"], w["N"], w["D"], w["causal"])
    rows = w["B"] * w["H"] * w["M"]
    table = {
        "attn_fwd": ("tensor", f),
        "attn_bwd_fused": ("tensor", 2.5 * f),
        "attn_bwd_dkdv": ("tensor", 2.0 * f),
        "attn_bwd_dq": ("tensor", 0.5 * f),
        "bwd_delta": ("hbm", rows * w["D"] * 2 * 2 + rows * 4),
        "bwd_dq_convert": ("hbm", rows * w["D"] * (4 + 2)),
    }
    return table.get(name)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def peak_value(peaks, key):
    for k in (key, key.replace("_sustained", "")):
        v = peaks.get(k)
        if isinstance(v, (int, float)):
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "peak", "median"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return FALLBACK_PEAKS.get(key)


def _code_only(text):
    """C++/CUDA source without its comments and blank lines (string literals in
    these sources hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


# The device sources each measured kernel is compiled from: its own .cu file
# and the device headers it includes (launch.h and tattn.h only declare host
# functions; the tensor maps built in api.cu must match the boxes each kernel
# expects, so a change there shows in the kernel's own source too).
_DEVICE_HEADERS = ("common.cuh", "ptx.cuh", "tmem_ldst.cuh")
KERNEL_SOURCES = {
    "attn_fwd": ("fwd.cu", "cluster.cuh"),
    "attn_bwd_dkdv": ("bwd.cu", "bwd_common.cuh"),
    "attn_bwd_dq": ("bwd.cu", "bwd_common.cuh"),
}


def kernel_source_hash(kernel=None):
    """Hash of the code (comments excluded) of the sources `kernel` is compiled
    from (KERNEL_SOURCES), or of every kernel source when `kernel` is None: the
    key under which profiles/traffic.json records the DRAM counters it was
    taken on."""
    csrc = os.path.join(ROOT, "tiled_attention_tcgen05_gb300", "csrc")
    files = sorted(os.listdir(csrc)) if kernel is None else sorted(KERNEL_SOURCES[kernel] + _DEVICE_HEADERS)
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or None
    when the summary was taken on different sources of that kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p) or kernel not in KERNEL_SOURCES:
        return None
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None
    ent = d.get("kernels", {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.idx), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not getattr(self, "out", ""):
            return None
        sm, mx, reasons, pw = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "power_w_median": statistics.median(pw) if pw else None, "samples": len(sm)}


# ------------------------------------------------------------ multi-rank
def max_over_ranks(values, dist=None, device="cpu"):
    """Element-wise maximum of per-rank timings (no-op for one rank)."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def job_tflops(flops_per_rank_step, world, ms):
    """Whole-job throughput: every rank runs the full workload (weak scaling)."""
    return flops_per_rank_step * world / (ms * 1e-3) / 1e12


# --------------------------------------------------------------- CPU oracle
def cpu_oracle_sample(heads: int, threads: int):
    """Runs the oracle's forward + backward on `heads` whole heads of the
    workload in a fresh process with `threads` BLAS threads.  Returns
    (seconds, flops of the sample)."""
    code = f"""
import os, sys, time, json
sys.path.insert(0, {ROOT!r})
import numpy as np
import synth_inputs as si, oracle
w = {WORKLOAD!r}
names = ("q", "k", "v", "do")
x = si.attention_inputs(1, {heads}, w["M"], w["N"], w["D"], w["dtype"], 3, names=names)
t0 = time.perf_counter()
for h in range({heads}):
    oracle.attention_fwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], w["causal"])
    oracle.attention_bwd(x["q"][0, h], x["k"][0, h], x["v"][0, h], x["do"][0, h], w["causal"])
print(json.dumps({{"s": time.perf_counter() - t0}}))
"""
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle sample failed: " + r.stderr[-2000:])
    secs = json.loads(r.stdout.strip().splitlines()[-1])["s"]
    w = WORKLOAD
    f = flops_fwd(1, heads, w["M"], w["N"], w["D"], w["causal"]) * 3.5
    return secs, f


def run_reference(args, rank, world):
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    heads = 1
    times = []
    for _ in range(args.warmup):
        cpu_oracle_sample(heads, threads)
    for _ in range(args.steps):
        s, f = cpu_oracle_sample(heads, threads)
        times.append(s)
    secs = statistics.mean(times)
    tflops = f / secs / 1e12
    sample = f"{heads} of 32 heads (b=0,h=0) of the workload per step, fwd+bwd in fp64 numpy"
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, **WORKLOAD, "sample_heads": heads},
        "cpu_baseline": {"value": tflops, "unit": "TFLOPS", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def merge_measure(ta, torch, dev, stream, o1, l1, o2, do, hbm_peak, iters=20):
    """Times the two-state merge forward and backward (HBM-bound) on states of
    the benchmark's shape, outside the step's timed region; algorithmic bytes
    are every operand read and written once."""
    l2 = l1.flip(-1).contiguous()
    dl = l1.clone()
    rows, D, e = o1.numel() // o1.shape[-1], o1.shape[-1], o1.element_size()
    fwd_bytes = 3 * rows * D * e + 3 * rows * 4
    bwd_bytes = 5 * rows * D * e + 5 * rows * 4
    out = {}
    for name, fn, nbytes in (("fwd", lambda: ta.merge_fwd(o1, l1, o2, l2, stream=stream), fwd_bytes),
                             ("bwd", lambda: ta.merge_bwd(o1, l1, o2, l2, do, dl, stream=stream), bwd_bytes)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = e0.elapsed_time(e1) / iters
        gbs = nbytes / (ms * 1e-3) / 1e9
        out[name] = {"ms": ms, "bytes": nbytes, "achieved": gbs, "frac": gbs / hbm_peak}
    out.update({"bound": "hbm", "unit": "GB/s", "peak": hbm_peak,
                "workload": "merge of two [B,H,M,D] states, B1 H32 M8192 D128 bf16 (inputs larger than L2)"})
    return out


def fp8_measure(ta, torch, si, dev, stream, w, bf16_peak, iters=10):
    """Times the e5m2 forward (attn_fwd_fp8) on the benchmark's shape, outside
    the step's timed region, against the fp8 dense peak taken as the measured
    bf16 peak x the nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)."""
    B, H, M, N, D, causal = w["B"], w["H"], w["M"], w["N"], w["D"], w["causal"]
    q = si.randn((B, H, M, D), "e5m2", si.seed_for(3, 10)).to(dev)
    k = si.randn((B, H, N, D), "e5m2", si.seed_for(3, 11)).to(dev)
    vt = si.randn((B, H, D, N), "e5m2", si.seed_for(3, 12)).to(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # larger than L2
    for _ in range(3):
        ta.attn_fwd_fp8(q, k, vt, causal, stream=stream)
    torch.cuda.synchronize(dev)
    ms = 0.0
    with torch.cuda.stream(stream):
        for _ in range(iters):  # the e5m2 inputs (100 MB) fit in L2: flush it before each timed launch
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            ta.attn_fwd_fp8(q, k, vt, causal, stream=stream)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ms += e0.elapsed_time(e1) / iters
    flops = 4.0 * B * H * M * N * D * (0.5 if causal else 1.0)
    peak = bf16_peak * (4.5 / 2.25)
    tf = flops / (ms * 1e-3) / 1e12
    return {"ms": ms, "flops": flops, "achieved": tf, "unit": "TFLOP/s", "bound": "tensor", "peak": peak,
            "peak_source": "measured bf16 burst x 2 (nominal fp8 / bf16)", "frac": tf / peak,
            "workload": "e5m2 forward, B1 H32 M=N=8192 D128 causal (L2 flushed before each timed launch)"}


def bwd_fused_measure(ta, torch, dev, stream, g, o, lse, w, bf16_peak, iters=10):
    """Times the two backward paths on the benchmark's shape and inputs,
    outside the step's timed region, alternating calls (L2 flushed before
    each): attn_bwd (dQ pass forming delta, dK/dV pass) and attn_bwd_fused (delta,
    one key-stationary pass with the fp32 dQ accumulator, dQ conversion).
    Both against the backward's algorithmic FLOPs (2.5x the forward)."""
    flops = 2.5 * flops_fwd(w["B"], w["H"], w["M"], w["N"], w["D"], w["causal"])
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    bufs = {"two_pass": [torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])],
            "fused": [torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])]}
    calls = {"two_pass": ta.attn_bwd, "fused": ta.attn_bwd_fused}
    for name, fn in calls.items():
        for _ in range(2):
            fn(g["q"], g["k"], g["v"], o, lse, g["do"], w["causal"], None, *bufs[name], stream=stream)
    torch.cuda.synchronize(dev)
    ms = {n: 0.0 for n in calls}
    with torch.cuda.stream(stream):
        for _ in range(iters):
            for name, fn in calls.items():
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn(g["q"], g["k"], g["v"], o, lse, g["do"], w["causal"], None, *bufs[name], stream=stream)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ms[name] += e0.elapsed_time(e1) / iters
    out = {"workload": "backward alone, B1 H32 M=N=8192 D128 bf16 causal (L2 flushed before each call)",
           "flops": flops, "unit": "TFLOP/s", "peak": bf16_peak}
    for name in calls:
        tf = flops / (ms[name] * 1e-3) / 1e12
        out[name] = {"ms": ms[name], "achieved": tf, "frac": tf / bf16_peak}
    return out


def timed_calls(ta, torch, dev, stream, flush, fn, iters):
    """(device ms, call ms) per call of `fn`, L2 flushed before each call.  The
    device time is the sum of the call's kernels, each bracketed by the
    library's own events on the launch stream (ta_profile_*); the call time is
    taken between events recorded before and after the Python call, so it
    also holds any wait of the GPU for the host (marshalling the arguments,
    encoding the tensor maps), which shows when the kernels take only tens of
    microseconds."""
    call = 0.0
    ta.profile_enable(True)
    with torch.cuda.stream(stream):
        for _ in range(iters):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            call += e0.elapsed_time(e1) / iters
    prof = ta.profile_read()
    ta.profile_enable(False)
    return sum(v[1] for v in prof.values()) / iters, call


def jvp_measure(ta, torch, si, dev, stream, bf16_peak, iters=20):
    """Times the JVP forward (attn_fwd_jvp with tL) and its backward
    (attn_bwd_jvp) on the JVP workload's shape, [2, 8, 1024, 64] fp16, causal
    and not, outside the step's timed region, by the library's per-launch
    events; L2 is flushed before each timed call (the inputs, 2 MB a tensor,
    fit in it).  Also on a long key range ([1, 4, 1024 x 8192], where the key
    split pays) and on [1, 32, 4096, 64], which fills the GPU.  Algorithmic FLOPs: the JVP
    forward is 3x the primal forward (6 matmul-equivalents of 2 M N D), the
    backward of the JVP 15 matmul-equivalents (S, T, dtO V^T, dO V^T + dtO tV^T
    and the nine gradient products), i.e. 7.5x the primal forward."""
    B, H, M, D = 2, 8, 1024, 64
    names = ("q", "k", "v", "tq", "tk", "tv", "do", "dto")
    g = {n: t.to(dev) for n, t in si.attention_inputs(B, H, M, M, D, "f16", 4, names=names).items()}
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {"workload": "JVP forward and its backward, B2 H8 M=N=1024 D64 fp16 (L2 flushed before each call)"}
    for causal in (False, True):
        fwd = lambda: ta.attn_fwd_jvp(*(g[n] for n in names[:6]), causal=causal, with_tlse=True, stream=stream)
        o, lse, to, tlse = fwd()
        ws = torch.empty(max(16, ta.load().attn_bwd_jvp_workspace_bytes(B, H, M, M, D, 0)), device=dev,
                         dtype=torch.uint8)
        bwd = lambda: ta.attn_bwd_jvp(*(g[n] for n in names[:6]), o, lse, to, tlse, g["do"], g["dto"],
                                      causal=causal, ws=ws, stream=stream)
        for _ in range(3):
            fwd()
            bwd()
        torch.cuda.synchronize(dev)
        timed = lambda fn: timed_calls(ta, torch, dev, stream, flush, fn, iters)
        res = {"fwd": timed(fwd), "bwd": timed(bwd)}
        # the forward with the key split forced each way (the library's own
        # choice is what "fwd_ms" measured)
        for mode in ("never", "always"):
            ta.set_fwd_kv_split(mode)
            fwd()
            res[mode] = timed(fwd)
        ta.set_fwd_kv_split("auto")
        f = flops_fwd(B, H, M, M, D, causal)
        tf_f = 3 * f / (res["fwd"][0] * 1e-3) / 1e12
        tf_b = 7.5 * f / (res["bwd"][0] * 1e-3) / 1e12
        out["causal" if causal else "noncausal"] = {
            "fwd_ms": res["fwd"][0], "bwd_ms": res["bwd"][0], "fwd_tflops": tf_f, "bwd_tflops": tf_b,
            "fwd_frac": tf_f / bf16_peak, "bwd_frac": tf_b / bf16_peak,
            "fwd_call_ms": res["fwd"][1], "bwd_call_ms": res["bwd"][1],
            "fwd_kv_split": ta.fwd_kv_split("attn_fwd_jvp", B, H, M, M, D, torch.float16, causal),
            "fwd_ms_unsplit": res["never"][0], "fwd_ms_split": res["always"][0]}
    # where the key split pays: few query tiles over a long key range
    Bl, Hl, Ml, Nl = 1, 4, 1024, 8192
    gl = {n: t.to(dev) for n, t in si.attention_inputs(Bl, Hl, Ml, Nl, D, "f16", 4, names=names[:6]).items()}
    fwd = lambda: ta.attn_fwd_jvp(*(gl[n] for n in names[:6]), causal=False, with_tlse=True, stream=stream)
    res = {}
    for mode in ("never", "always", "auto"):
        ta.set_fwd_kv_split(mode)
        fwd()
        res[mode] = timed_calls(ta, torch, dev, stream, flush, fwd, iters)[0]
    ta.set_fwd_kv_split("auto")
    out["long_keys"] = {"shape": "B1 H4 M=1024 N=8192 D64 fp16, non-causal (32 query tiles of 64 key tiles)",
                        "fwd_kv_split": ta.fwd_kv_split("attn_fwd_jvp", Bl, Hl, Ml, Nl, D, torch.float16, False),
                        "fwd_ms": res["auto"], "fwd_ms_unsplit": res["never"], "fwd_ms_split": res["always"]}
    # a shape that fills the GPU several times over: 1024 query tiles
    Bw, Hw, Mw = 1, 32, 4096
    gw = {n: t.to(dev) for n, t in si.attention_inputs(Bw, Hw, Mw, Mw, D, "f16", 4, names=names).items()}
    wide = {"shape": "B1 H32 M=N=4096 D64 fp16"}
    for causal in (False, True):
        fwd = lambda: ta.attn_fwd_jvp(*(gw[n] for n in names[:6]), causal=causal, with_tlse=True, stream=stream)
        o, lse, to, tlse = fwd()
        ws = torch.empty(max(16, ta.load().attn_bwd_jvp_workspace_bytes(Bw, Hw, Mw, Mw, D, 0)), device=dev,
                         dtype=torch.uint8)
        bwd = lambda: ta.attn_bwd_jvp(*(gw[n] for n in names[:6]), o, lse, to, tlse, gw["do"], gw["dto"],
                                      causal=causal, ws=ws, stream=stream)
        fwd()
        bwd()
        f = flops_fwd(Bw, Hw, Mw, Mw, D, causal)
        tf = timed_calls(ta, torch, dev, stream, flush, fwd, iters)[0]
        tb = timed_calls(ta, torch, dev, stream, flush, bwd, iters)[0]
        wide["causal" if causal else "noncausal"] = {
            "fwd_ms": tf, "bwd_ms": tb, "fwd_tflops": 3 * f / (tf * 1e-3) / 1e12,
            "bwd_tflops": 7.5 * f / (tb * 1e-3) / 1e12, "fwd_frac": 3 * f / (tf * 1e-3) / 1e12 / bf16_peak,
            "bwd_frac": 7.5 * f / (tb * 1e-3) / 1e12 / bf16_peak}
    out["wide"] = wide
    return out


def configs_measure(ta, torch, si, dev, stream, bf16_peak, iters=20):
    """Times one fwd+bwd step (forward then backward, inputs resident) on the
    other workloads: 1 (B1 H2 S128 D64 fp16, non-causal), 2 (B4 H16 S2048 D128
    bf16 causal) and 5 (piecewise, B2 H16 S4096 D64 bf16 causal, w = 512),
    and workload 5's shape at D = 128 (piecewise) and at D = 64 and 128 as
    standard attention, for comparison, as the device time of the step's
    kernels (timed_calls).  L2 is flushed
    before each timed step.  FLOPs are the standard count
    (4 M N D per head forward, x 3.5 for forward + backward, x 0.5 causal); the
    piecewise path's second score products on straddling tiles are overhead."""
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    out = {}
    w5 = si.WORKLOADS[5]
    cases = [(str(wid), wid, si.WORKLOADS[wid]) for wid in (1, 2, 5)]
    cases.append(("5_d128", 5, dict(w5, D=128, name="piecewise fwd+bwd bf16 causal B2 H16 S4096 D128 w512")))
    for d in (64, 128):
        cases.append((f"5_std_d{d}", 5, dict(w5, D=d, mode="fwdbwd", w=None,
                                             name=f"fwd+bwd bf16 causal B2 H16 S4096 D{d} (standard)")))
    for key, wid, w in cases:
        B, H, M, N, D, causal = w["B"], w["H"], w["M"], w["N"], w["D"], w["causal"]
        pw = w["mode"] == "piecewise"
        names = ("q1", "k1", "q2", "k2", "v", "do") if pw else ("q", "k", "v", "do")
        g = {n: t.to(dev) for n, t in si.attention_inputs(B, H, M, N, D, w["dtype"], wid, names=names).items()}
        if pw:
            def fn():
                o, lse = ta.piecewise_fwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], w["w"], causal, stream=stream)
                ta.piecewise_bwd(g["q1"], g["k1"], g["q2"], g["k2"], g["v"], o, lse, g["do"], w["w"], causal,
                                 stream=stream)
        else:
            def fn():
                o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], causal, stream=stream)
                ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal, stream=stream)
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        ms, call_ms = timed_calls(ta, torch, dev, stream, flush, fn, iters)
        f = flops_fwd(B, H, M, N, D, causal) * 3.5
        tf = f / (ms * 1e-3) / 1e12
        out[key] = {"workload": w["name"], "ms_per_step": ms, "tflops": tf, "frac": tf / bf16_peak,
                    "call_ms_per_step": call_ms}
    return out


# -------------------------------------------------------------- GPU arm
def run_ours(args, rank, world, local_rank):
    import torch
    import synth_inputs as si
    import tiled_attention_tcgen05_gb300 as ta

    ta.load()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOAD
    B, H, M, N, D, causal = w["B"], w["H"], w["M"], w["N"], w["D"], w["causal"]
    names = ("q", "k", "v", "do")
    cpu = si.attention_inputs(B, H, M, N, D, w["dtype"], 3, names=names)
    host = {n: t.pin_memory() for n, t in cpu.items()}
    g = {n: t.to(dev) for n, t in host.items()}
    o = torch.empty_like(g["q"])
    lse = torch.empty(B, H, M, device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])
    ws = torch.empty(max(16, ta.attn_bwd_workspace_bytes(B, H, M, N, D, torch.bfloat16)), device=dev,
                     dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)

    def step():
        ta.attn_fwd(g["q"], g["k"], g["v"], causal, None, o=o, lse=lse, stream=stream)
        ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], causal, None, dq=dq, dk=dk, dv=dv, ws=ws,
                    stream=stream)

    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(max(3, args.warmup)):
        step()
    if ta.sync_status(stream) != "TA_OK":
        raise RuntimeError("device error word set during warm-up")

    # ---- device-resident timed region (with per-kernel events)
    barrier()
    ta.profile_enable(True)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clk:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
    prof = ta.profile_read()
    ta.profile_enable(False)
    barrier()
    status = ta.sync_status(stream)
    if status != "TA_OK":
        raise RuntimeError(f"device error word: {status}")
    ms = ev0.elapsed_time(ev1) / args.steps

    # ---- the host link's copy rates on this machine (outside every timed region):
    # each direction alone and both at once, one copy of the step's size each
    def link_rates(reps=5):
        n = 268 << 20
        hi = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        ho = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        di = torch.empty(n, dtype=torch.uint8, device=dev)
        do_ = torch.empty(n, dtype=torch.uint8, device=dev)
        s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        rates = {}
        for name, ups, downs in (("h2d_gbs", 1, 0), ("d2h_gbs", 0, 1), ("both_gbs", 1, 1)):
            best = 0.0
            for _ in range(reps):
                torch.cuda.synchronize(dev)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                s1.wait_stream(stream)
                s2.wait_stream(stream)
                if ups:
                    with torch.cuda.stream(s1):
                        di.copy_(hi, non_blocking=True)
                if downs:
                    with torch.cuda.stream(s2):
                        ho.copy_(do_, non_blocking=True)
                stream.wait_stream(s1)
                stream.wait_stream(s2)
                e1.record(stream)
                torch.cuda.synchronize(dev)
                best = max(best, n * (ups + downs) / (e0.elapsed_time(e1) * 1e-3) / 1e9)
            rates[name] = best
        del hi, ho, di, do_
        return rates

    link = link_rates()

    # ---- end-to-end: pinned host inputs -> device -> results back to host.
    # Every step copies its own inputs in and all its results out inside the
    # timed region.  The copies run on their own streams into double-buffered
    # device memory, so step i's kernels overlap step i+1's input copy and
    # step i-1's result copy (a training loop's prefetch).
    # Each direction moves one contiguous buffer per step (one copy each way):
    # the inputs, and the results, are views into it on 256-byte boundaries.
    def packed(like, make):
        offs, total = {}, 0
        for n, t in like.items():
            nbytes = t.numel() * t.element_size()
            offs[n] = (total, nbytes, t.shape, t.dtype)
            total += (nbytes + 255) // 256 * 256
        buf = make(total)
        return buf, {n: buf[a:a + nb].view(dt).view(shape) for n, (a, nb, shape, dt) in offs.items()}

    def pinned(nbytes):
        return torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)

    def on_device(nbytes):
        return torch.empty(nbytes, dtype=torch.uint8, device=dev)

    out_names = ("o", "lse", "dq", "dk", "dv")
    out_like = dict(zip(out_names, (o, lse, dq, dk, dv)))
    nbuf = 2
    host_buf, host_in = packed(host, pinned)
    for n in names:
        host_in[n].copy_(host[n])
    dbuf_in = [packed(host, on_device) for _ in range(nbuf)]
    dbuf_out = [packed(out_like, on_device) for _ in range(nbuf)]
    out_host = [packed(out_like, pinned) for _ in range(nbuf)]
    h2d = host_buf.numel()
    d2h = out_host[0][0].numel()
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_run(nsteps, e_start=None, e_end=None):
        """Enqueues nsteps end-to-end steps; returns the host's wall time
        spent enqueueing them (no synchronisation inside)."""
        t_host = time.perf_counter()
        in_ready = [torch.cuda.Event() for _ in range(nbuf)]
        in_free = [torch.cuda.Event() for _ in range(nbuf)]
        out_ready = [torch.cuda.Event() for _ in range(nbuf)]
        out_free = [torch.cuda.Event() for _ in range(nbuf)]

        def load(i):
            b = i % nbuf
            if i >= nbuf:
                h2d_s.wait_event(in_free[b])
            with torch.cuda.stream(h2d_s):
                dbuf_in[b][0].copy_(host_buf, non_blocking=True)
            in_ready[b].record(h2d_s)

        if e_start is not None:
            e_start.record(h2d_s)
        load(0)
        for i in range(nsteps):
            b = i % nbuf
            if i + 1 < nsteps:
                load(i + 1)
            stream.wait_event(in_ready[b])
            if i >= nbuf:
                stream.wait_event(out_free[b])
            x, y = dbuf_in[b][1], dbuf_out[b][1]
            ta.attn_fwd(x["q"], x["k"], x["v"], causal, None, o=y["o"], lse=y["lse"], stream=stream)
            ta.attn_bwd(x["q"], x["k"], x["v"], y["o"], y["lse"], x["do"], causal, None, dq=y["dq"], dk=y["dk"],
                        dv=y["dv"], ws=ws, stream=stream)
            in_free[b].record(stream)
            out_ready[b].record(stream)
            d2h_s.wait_event(out_ready[b])
            with torch.cuda.stream(d2h_s):
                out_host[b][0].copy_(dbuf_out[b][0], non_blocking=True)
            out_free[b].record(d2h_s)
        if e_end is not None:
            e_end.record(d2h_s)
        return time.perf_counter() - t_host

    e2e_run(2)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_host_ms = e2e_run(args.steps, e0, e1) * 1e3 / args.steps
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / args.steps
    if ta.sync_status(stream) != "TA_OK":
        raise RuntimeError("device error word set in the end-to-end run")
    # the results that came back are the step's: spot-check one output against the device copy
    last = (args.steps - 1) % nbuf
    if not torch.equal(out_host[last][1]["lse"], dbuf_out[last][1]["lse"].cpu()):
        raise RuntimeError("end-to-end result copy differs from the device result")

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], dist, dev)

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    f_step = step_flops()
    value = job_tflops(f_step, world, ms)
    e2e_value = job_tflops(f_step, world, e2e_ms)
    peaks, src = load_peaks()
    bf16_peak = peak_value(peaks, "bf16_tflops")
    hbm_peak = peak_value(peaks, "hbm_gbs")

    kernels = {}
    for name, (n, tot) in prof.items():
        kernels[name] = {"launches": n, "total_ms": tot, "avg_ms": tot / max(1, n)}
    dom = max(kernels, key=lambda k: kernels[k]["total_ms"])
    bound, algo = kernel_algorithmic(dom)
    avg_s = kernels[dom]["avg_ms"] * 1e-3
    if bound == "tensor":
        achieved = algo / avg_s / 1e12
        peak, unit = bf16_peak, "TFLOP/s"
    else:
        achieved = algo / avg_s / 1e9
        peak, unit = hbm_peak, "GB/s"
    for name, k in kernels.items():
        ka = kernel_algorithmic(name)
        if ka:
            b, a = ka
            rate = a / (k["avg_ms"] * 1e-3)
            k["achieved"] = rate / 1e12 if b == "tensor" else rate / 1e9
            k["unit"] = "TFLOP/s" if b == "tensor" else "GB/s"
            k["frac_of_" + src] = k["achieved"] / (bf16_peak if b == "tensor" else hbm_peak)

    merge = merge_measure(ta, torch, dev, stream, o, lse, dq, g["do"], hbm_peak)
    fp8 = fp8_measure(ta, torch, si, dev, stream, w, bf16_peak)
    bwd_paths = bwd_fused_measure(ta, torch, dev, stream, g, o, lse, w, bf16_peak)
    jvp = jvp_measure(ta, torch, si, dev, stream, bf16_peak)
    other = configs_measure(ta, torch, si, dev, stream, bf16_peak)
    if ta.sync_status(stream) != "TA_OK":
        raise RuntimeError("device error word set in the merge measurement")

    cpu_heads = 6
    cpu_secs, cpu_f = cpu_oracle_sample(cpu_heads, os.cpu_count() or 1)
    launches = sum(k["launches"] for k in kernels.values())
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, **w, "l2": "inputs (q,k,v,dO 268 MB) larger than L2 (129 MB)",
                   "flops_per_step": f_step},
        "pct_of_peak": value / world / bf16_peak,
        "peak_source": src,
        "e2e": {"value": e2e_value, "unit": "TFLOPS", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms,
                "host_enqueue_ms_per_step": e2e_host_ms,
                "link": {**link, "copy_floor_ms": (h2d + d2h) / (link["both_gbs"] * 1e9) * 1e3,
                         "how": "pinned copies of 268 MB, best of 5, each direction alone and both at once"},
                "method": "pinned host inputs copied in and all results copied out every step (one contiguous "
                          "buffer each way), on copy streams overlapping the neighbouring steps' kernels "
                          "(double-buffered device memory); "
                          "host_enqueue_ms_per_step is the host's wall time to issue a step's copies, "
                          "launches and stream waits (near ms_per_step: the host, not the GPU, sets the pace)"},
        "gpu_launches": launches,
        "roofline": {"bound": bound, "kernel": dom, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "peak_source": src + (" (burst)" if bound == "tensor" else ""),
                     "traffic": ncu_traffic(dom), "algorithmic_per_launch": algo},
        "kernels": kernels,
        "merge": merge,
        "fp8_fwd": fp8,
        "bwd_paths": bwd_paths,
        "jvp": jvp,
        "other_workloads": other,
        "cpu_baseline": {"value": cpu_f / cpu_secs / 1e12, "unit": "TFLOPS", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": "%d of 32 heads (b=0, h<%d), fwd+bwd, fp64 numpy, %.1f s"
                                   % (cpu_heads, cpu_heads, cpu_secs)},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if "RANK" not in os.environ:
        world = 1  # a single process drives one GPU; N > 1 needs one process per GPU
    if args.impl == "reference":
        return run_reference(args, rank, world)
    return run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    sys.exit(main())
