"""Builds libdgq.so in-tree with nvcc for sm_103a (one -gencode; the eight translation units
of csrc/ compiled in parallel).  Used by ``__graft_entry__.build()`` and by the binding when the
library is missing or older than its sources."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdgq.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
# The quantiser's fp32 steps are bit-exact IEEE operations: no FMA contraction there.
UNITS = {
    "dgq_compress.cu": ["-fmad=false", "-prec-div=true", "-prec-sqrt=true"],
    "dgq_compress_cluster.cu": ["-fmad=false", "-prec-div=true", "-prec-sqrt=true"],
    "dgq_append.cu": ["-fmad=false", "-prec-div=true", "-prec-sqrt=true"],
    "dgq_formats.cu": ["-fmad=false", "-prec-div=true", "-prec-sqrt=true"],
    "dgq_prefill.cu": ["-fmad=false", "-prec-div=true", "-prec-sqrt=true"],
    "dgq_attn.cu": [],
    "dgq_host.cu": [],
    "dgq_noalloc.cu": [],
}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
            if f.endswith((".cu", ".cuh", ".h"))] + [os.path.join(INCLUDE, "dgq.h")]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)

    def compile_unit(name: str) -> str:
        obj = os.path.join(OUT_DIR, name.replace(".cu", ".o"))
        cmd = [nvcc, *COMMON, *ARCH, *UNITS[name], "-c", os.path.join(CSRC, name), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {name}:\n{res.stderr}")
        if verbose and res.stderr:
            print(res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        objs = list(ex.map(compile_unit, UNITS))
    tmp = LIB + f".{os.getpid()}.tmp"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
