"""Builds the C-ABI shared library for sm_103a in-tree.

    python dropout_lowbias32_hash32_gb300/build.py [--verbose]

compiles every csrc/*.cu with nvcc (one process per translation unit, in
parallel) and links them into _lib/librng_lowbias32.so, with the CUDA
runtime linked statically.  Sources are never compiled with fast-math: the
dropout quotient and the ziggurat's slow path rely on IEEE operations.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIBNAME = "librng_lowbias32.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _flags(verbose: bool) -> list[str]:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _compile(src: str, verbose: bool) -> tuple[str, str]:
    obj = os.path.join(OBJ, os.path.basename(src)[:-3] + ".o")
    deps = [src] + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(CSRC, "*.inc")) + glob.glob(os.path.join(ROOT, "include", "*"))
    if not verbose and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(d) for d in deps):
        return obj, ""
    proc = subprocess.run([nvcc(), *_flags(verbose), "-c", src, "-o", obj], capture_output=True, text=True)
    if proc.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{proc.stdout}{proc.stderr}")
    return obj, proc.stdout + proc.stderr


def build(verbose: bool = False) -> str:
    """Compile and link; returns the path of the shared library."""
    os.makedirs(OBJ, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(len(sources), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), sources))
    if verbose:
        for _, log in results:
            if log:
                sys.stdout.write(log)
    lib = os.path.join(LIBDIR, LIBNAME)
    objs = [o for o, _ in results]
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + ".tmp"
        subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs], check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv))
