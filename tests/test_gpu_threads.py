"""Entry points called from several host threads at once, each thread on its
own stream with its own buffers: the results are bit-identical to the same
calls made one at a time (no kernel uses atomics, so a call's result does
not depend on what else runs), and the device error word stays clear."""
import threading

import pytest
import torch

from _parity import inputs

pytestmark = pytest.mark.gpu


def _job(kind, ta, g, stream):
    if kind == "std_bf16":
        o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], True, stream=stream)
        return (o, lse) + tuple(ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], True, stream=stream))
    if kind == "std_f16":
        o, lse = ta.attn_fwd(g["q"], g["k"], g["v"], False, stream=stream)
        return (o, lse) + tuple(ta.attn_bwd(g["q"], g["k"], g["v"], o, lse, g["do"], False, stream=stream))
    if kind == "jvp":
        o, lse, to, tl = ta.attn_fwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], causal=True,
                                         with_tlse=True, stream=stream)
        gr = ta.attn_bwd_jvp(g["q"], g["k"], g["v"], g["tq"], g["tk"], g["tv"], o, lse, to, tl, g["do"],
                             g["dto"], causal=True, stream=stream)
        return (o, lse, to, tl) + tuple(gr)
    o, lse = ta.piecewise_fwd(g["q"], g["k"], g["tq"], g["tk"], g["v"], 100, True, stream=stream)
    return (o, lse) + tuple(ta.piecewise_bwd(g["q"], g["k"], g["tq"], g["tk"], g["v"], o, lse, g["do"], 100, True,
                                             stream=stream))


JOBS = [("std_bf16", (1, 4, 640, 640, 128, "bf16")), ("std_f16", (2, 2, 300, 200, 64, "f16")),
        ("jvp", (1, 3, 384, 384, 64, "bf16")), ("piecewise", (1, 2, 512, 512, 128, "bf16"))]


def test_concurrent_host_threads_match_one_at_a_time(gpu_lib):
    ta = gpu_lib
    names = ("q", "k", "v", "do", "tq", "tk", "tv", "dto")
    data = [inputs(*shape, 71 + i, names)[1] for i, (_, shape) in enumerate(JOBS)]
    streams = [torch.cuda.Stream() for _ in JOBS]
    ref = []
    for (kind, _), g, s in zip(JOBS, data, streams):
        ref.append(_job(kind, ta, g, s))
    torch.cuda.synchronize()
    assert ta.sync_status() == "TA_OK"

    for _ in range(3):
        out = [None] * len(JOBS)
        errors = []
        start = threading.Barrier(len(JOBS))

        def run(i):
            try:
                with torch.cuda.stream(streams[i]):
                    start.wait()
                    out[i] = _job(JOBS[i][0], ta, data[i], streams[i])
            except Exception as e:  # reported below, on the main thread
                errors.append(e)

        threads = [threading.Thread(target=run, args=(i,)) for i in range(len(JOBS))]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors, errors
        torch.cuda.synchronize()
        assert ta.sync_status() == "TA_OK"
        for (kind, _), r, o in zip(JOBS, ref, out):
            for j, (a, b) in enumerate(zip(r, o)):
                assert torch.equal(a, b), f"{kind}: output {j} differs from the one-at-a-time result"
