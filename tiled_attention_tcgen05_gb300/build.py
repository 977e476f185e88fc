"""Builds libtattn.so in-tree from csrc/*.cu for sm_103a (GB300).

Each translation unit is compiled by its own nvcc process (in parallel), then
the objects are linked into ``tiled_attention_tcgen05_gb300/libtattn.so``.
Re-running is incremental: a unit is rebuilt only when a source or header
under csrc/ or include/ is newer than its object.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtattn.so")
# The guard build (device-side checks compiled in with TA_GUARD, see
# csrc/guard.cuh): a test library, built beside the product one.
BUILD_GUARD = os.path.join(PKG, "_build_guard")
LIB_GUARD = os.path.join(PKG, "libtattn_guard.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtattn.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(ROOT, "include", "tattn.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths if os.path.exists(p))


def build(verbose: bool = False, ptxas_info: bool = False, guard: bool = False) -> str:
    """Compile and link; returns the path of libtattn.so (guard=True:
    libtattn_guard.so, the same sources with the device-side checks)."""
    nvcc = _nvcc()
    bdir, lib = (BUILD_GUARD, LIB_GUARD) if guard else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    newest = _deps_mtime()
    srcs = _sources()
    objs = [os.path.join(bdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DTA_GUARD"] if guard else [])

    def compile_one(pair):
        src, obj = pair
        if not ptxas_info and os.path.exists(obj) and os.path.getmtime(obj) >= newest:
            return None
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return r.stderr if (verbose or ptxas_info) else None

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        logs = list(ex.map(compile_one, zip(srcs, objs)))
    for log in logs:
        if log:
            sys.stderr.write(log)
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv))
