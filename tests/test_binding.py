"""The Python binding without a GPU: every entry point refuses host (CPU)
tensors with an error instead of computing anything (the package has no CPU
path), refuses tensors that are not [B, H, S, D], and the package imports
nothing of the oracle."""
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ta():
    from tiled_attention_tcgen05_gb300 import build
    path = build.build()
    import tiled_attention_tcgen05_gb300 as pkg
    pkg.load(path)
    return pkg


def _t(*shape, dtype=torch.bfloat16):
    return torch.zeros(*shape, dtype=dtype)


def test_every_entry_point_refuses_host_tensors(ta):
    q = k = v = do = _t(1, 2, 128, 64)
    lse = torch.zeros(1, 2, 128)
    calls = {
        "attn_fwd": lambda: ta.attn_fwd(q, k, v, True),
        "attn_bwd": lambda: ta.attn_bwd(q, k, v, q, lse, do, True),
        "attn_fwd_jvp": lambda: ta.attn_fwd_jvp(q, k, v, q, k, v, causal=True, with_tlse=True),
        "attn_bwd_jvp": lambda: ta.attn_bwd_jvp(q, k, v, q, k, v, q, lse, q, lse, do, do, causal=True),
        "piecewise_fwd": lambda: ta.piecewise_fwd(q, k, q, k, v, 64, True),
        "piecewise_bwd": lambda: ta.piecewise_bwd(q, k, q, k, v, q, lse, do, 64, True),
        "merge_fwd": lambda: ta.merge_fwd(q, lse, q, lse),
        "merge_bwd": lambda: ta.merge_bwd(q, lse, q, lse, do),
        "attn_fwd_fp8": lambda: ta.attn_fwd_fp8(_t(1, 2, 128, 64, dtype=torch.float8_e5m2),
                                                _t(1, 2, 128, 64, dtype=torch.float8_e5m2),
                                                _t(1, 2, 64, 128, dtype=torch.float8_e5m2), True),
    }
    for name, call in calls.items():
        with pytest.raises(ValueError, match="CUDA"):
            call()


def test_tensors_must_be_four_dimensional(ta):
    with pytest.raises(ValueError, match=r"\[B, H, S, D\]"):
        ta.attn_fwd(_t(2, 128, 64), _t(2, 128, 64), _t(2, 128, 64))


def test_package_holds_no_path_to_the_oracle():
    pkg = os.path.join(ROOT, "tiled_attention_tcgen05_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert not re.search(r"\bimport\s+oracle\b|\bfrom\s+oracle\b", text), f"{f} imports the oracle"
