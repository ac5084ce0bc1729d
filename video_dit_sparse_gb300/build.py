"""Builds ``libsparse_attn.so`` in-tree from ``csrc/*.cu`` for sm_103a.

Each translation unit is compiled in parallel with nvcc, then linked into a
shared library with the CUDA runtime linked statically.  No CMake.
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
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsparse_attn.so")
SOURCES = ["sa_api.cu", "sa_forward.cu", "sa_builder.cu", "sa_colstat.cu", "sa_layout.cu", "sa_format.cu", "sa_pipeline.cu", "sa_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsparse_attn.so")


def _flags(verbose: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I" + INCLUDE, "-I" + CSRC]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "sparse_attn.h"))
    objs, todo = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or verbose or _stale(o, [s] + headers):
            todo.append((s, o))
    exe = nvcc()

    def compile_one(item):
        s, o = item
        cmd = [exe] + _flags(verbose) + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(s)}:\n{r.stdout}\n{r.stderr}")
        return r.stderr

    logs = []
    with cf.ThreadPoolExecutor(max_workers=jobs or len(todo) or 1) as ex:
        logs = list(ex.map(compile_one, todo))
    if verbose:
        for log in logs:
            sys.stderr.write(log)
    if force or todo or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [exe] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static", "-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
