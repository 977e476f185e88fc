"""The library's calls inside a CUDA graph: attn_fwd + attn_bwd (and the
backward of the JVP) captured once on a side stream and replayed give
bit-identical results to the eager calls (every kernel is deterministic: no
atomics, fixed reduction orders), and a replay after new inputs are copied
into the captured buffers computes on the new inputs."""
import pytest
import torch

import oracle
from _parity import TOL, compare, inputs, o_tol

pytestmark = pytest.mark.gpu


def test_fwd_bwd_graph_replay_matches_eager(gpu_lib):
    ta = gpu_lib
    B, H, M, N, D = 1, 4, 640, 640, 128
    cpu, g = inputs(B, H, M, N, D, "bf16", 71, ("q", "k", "v", "do"))
    o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True)
    dq, dk, dv = ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], True)
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]

    go, glse = torch.empty_like(o), torch.empty_like(lse)
    gdq, gdk, gdv = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    ws = torch.empty(max(16, ta.attn_bwd_workspace_bytes(B, H, M, N, D, torch.bfloat16)), device="cuda",
                     dtype=torch.uint8)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        # one eager pass on the side stream first (first-call attribute setup happens outside capture)
        ta.attn_fwd(g["q"], g["k"], g["v"], True, o=go, lse=glse, stream=side)
        ta.attn_bwd(g["q"], g["k"], g["v"], go, glse, g["do"], True, dq=gdq, dk=gdk, dv=gdv, ws=ws, stream=side)
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            ta.attn_fwd(g["q"], g["k"], g["v"], True, o=go, lse=glse, stream=side)
            ta.attn_bwd(g["q"], g["k"], g["v"], go, glse, g["do"], True, dq=gdq, dk=gdk, dv=gdv, ws=ws,
                        stream=side)
    for t in (go, glse, gdq, gdk, gdv):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert ta.sync_status() == "TA_OK"
    for name, got, r in zip(("O", "L", "dQ", "dK", "dV"), (go, glse, gdq, gdk, gdv), ref):
        assert torch.equal(got, r), f"{name} differs between graph replay and eager"

    # new inputs in the captured buffers: the replay computes on them
    cpu2, g2 = inputs(B, H, M, N, D, "bf16", 72, ("q", "k", "v", "do"))
    for n in ("q", "k", "v", "do"):
        g[n].copy_(g2[n])
    graph.replay()
    torch.cuda.synchronize()
    assert ta.sync_status() == "TA_OK"
    O, L = oracle.attention_fwd_bhsd(cpu2["q"], cpu2["k"], cpu2["v"], True)
    dQ, dK, dV = oracle.attention_bwd_bhsd(cpu2["q"], cpu2["k"], cpu2["v"], cpu2["do"], True)
    compare("O", go, O, o_tol("bf16"))
    compare("L", glse, L, TOL["L"])
    for name, got, r in zip(("dQ", "dK", "dV"), (gdq, gdk, gdv), (dQ, dK, dV)):
        compare(name, got, r, TOL["grad"])


def test_jvp_backward_graph_replay_matches_eager(gpu_lib):
    ta = gpu_lib
    names = ("q", "k", "v", "tq", "tk", "tv", "do", "dto")
    cpu, g = inputs(2, 2, 256, 256, 64, "f16", 73, names)
    o, lse, to, tlse = ta.attn_fwd_jvp(*(g[n] for n in names[:6]), causal=True, with_tlse=True)
    ref = ta.attn_bwd_jvp(*(g[n] for n in names[:6]), o, lse, to, tlse, g["do"], g["dto"], causal=True)
    ref = [t.clone() for t in ref]
    ws = torch.empty(max(16, ta.load().attn_bwd_jvp_workspace_bytes(2, 2, 256, 256, 64, 0)), device="cuda",
                     dtype=torch.uint8)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        ta.attn_bwd_jvp(*(g[n] for n in names[:6]), o, lse, to, tlse, g["do"], g["dto"], causal=True, ws=ws,
                        stream=side)
        side.synchronize()
        with torch.cuda.graph(graph, stream=side):
            out = ta.attn_bwd_jvp(*(g[n] for n in names[:6]), o, lse, to, tlse, g["do"], g["dto"], causal=True,
                                  ws=ws, stream=side)
    graph.replay()
    torch.cuda.synchronize()
    assert ta.sync_status() == "TA_OK"
    for got, r in zip(out, ref):
        assert torch.equal(got, r)
