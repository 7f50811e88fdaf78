"""Builds libcsa.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m long_context_compressed_16_b300.build [--verbose] [--force]
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libcsa.so")
SOURCES = ["api.cu", "compress.cu", "index_score.cu", "topk.cu", "attend.cu", "attend_tc.cu", "noalloc.cu", "selftest.cu", "proj.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _run(cmd):
    return subprocess.run(cmd, capture_output=True, text=True)


def build(verbose: bool = False, force: bool = False) -> str:
    """Compiles every source to an object file (in parallel, one nvcc per file) and links the
    shared library.  Skips the work when the library is newer than every source and header."""
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, "common.cuh"), os.path.join(CSRC, "tc.cuh"), os.path.join(ROOT, "include", "csa.h")]
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(p) <= t for p in deps):
            return LIB
    objdir = os.path.join(PKG, "_build")
    os.makedirs(objdir, exist_ok=True)
    common = [nvcc(), "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", *ARCH, "-I", os.path.join(ROOT, "include")]
    if verbose:
        common.insert(1, "-Xptxas=-v")
    objs = [os.path.join(objdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    headers = deps[len(srcs):]
    stale = [(s, o) for s, o in zip(srcs, objs)
             if force or not os.path.exists(o) or any(os.path.getmtime(p) > os.path.getmtime(o) for p in [s, *headers])]
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=max(1, min(len(stale), os.cpu_count() or 4))) as ex:
        results = list(ex.map(_run, [common + ["-c", s, "-o", o] for s, o in stale]))
    for (s, _), r in zip(stale, results):
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n" + r.stdout + r.stderr)
        if verbose:
            sys.stderr.write(f"== {os.path.basename(s)}\n" + r.stdout + r.stderr)
    r = _run([nvcc(), "-shared", *ARCH, "-o", LIB + ".tmp", *objs, "-lcudart"])
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n" + r.stdout + r.stderr)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, force="--force" in sys.argv))
