"""Builds the CUDA library libtopk_paged.so in-tree for sm_103a with nvcc.

Ten translation units are compiled in parallel and linked into one shared library
that exports the C ABI of include/topk_paged.h, include/indexer_prologue.h,
include/indexer_logits.h and include/hisparse_resolver.h (no torch types cross it).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtopk_paged.so")
SOURCES = ["select.cu", "short.cu", "medium.cu", "rowcluster.cu", "plan.cu", "abi.cu", "noalloc.cu",
           "prologue.cu", "resolver.cu", "logits.cu"]
HEADERS = ["common.cuh", "keys.cuh", "plan_logic.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def _flags(extra=()):
    return (ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", os.path.join(ROOT, "include")] + list(extra))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          trace: bool = False) -> str:
    """trace=True builds libtopk_paged_trace.so with the phase timer stamps compiled in
    (exports topk_trace_select / topk_trace_plan); the default build has none."""
    bdir = os.path.join(BUILD, "trace") if trace else BUILD
    lib = LIB.replace(".so", "_trace.so") if trace else LIB
    defs = ["-DTOPK_TRACE"] if trace else []
    os.makedirs(bdir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", h)
                                                        for h in ("topk_paged.h", "indexer_prologue.h",
                                                                  "indexer_logits.h",
                                                                  "hisparse_resolver.h")]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or ptxas_info or _stale(o, [s] + hdrs):
            extra = ["-Xptxas", "-v"] if ptxas_info else []
            jobs.append([nvcc()] + _flags(extra + defs) + ["-c", s, "-o", o])
    if jobs:
        with concurrent.futures.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            futs = [ex.submit(subprocess.run, j, capture_output=True, text=True) for j in jobs]
            for j, f in zip(jobs, futs):
                r = f.result()
                if verbose or ptxas_info:
                    sys.stderr.write(r.stdout + r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed:\n{' '.join(j)}\n{r.stdout}\n{r.stderr}")
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                trace="--trace" in sys.argv))
