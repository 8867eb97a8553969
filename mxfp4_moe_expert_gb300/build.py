"""Builds libmoe_mxfp4.so in-tree with nvcc for sm_103a (one -gencode).

Each .cu file is compiled to an object in parallel, then linked into a shared
library under mxfp4_moe_expert_gb300/lib/.  Run as a module or call build().
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "lib")
LIB_NAME = "libmoe_mxfp4.so"
GENCODE = "arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags() -> list[str]:
    return ["-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def build(verbose: bool = False) -> str:
    """Compiles the library; returns the path of the shared object."""
    obj_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    nvcc = _nvcc()
    sources = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "moe_mxfp4.h"))
    newest_header = max(os.path.getmtime(p) for p in headers)

    def compile_one(src: str) -> str:
        s = os.path.join(CSRC, src)
        o = os.path.join(obj_dir, src[:-3] + ".o")
        if (not verbose and os.path.exists(o)
                and os.path.getmtime(o) >= max(os.path.getmtime(s), newest_header)):
            return o
        cmd = [nvcc, *_flags(), "-c", s, "-o", o]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return o

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, len(sources)))) as ex:
        objs = list(ex.map(compile_one, sources))
    lib = os.path.join(OUT_DIR, LIB_NAME)
    tmp = lib + ".tmp"
    r = subprocess.run([nvcc, "-gencode", GENCODE, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
