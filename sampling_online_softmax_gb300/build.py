"""Compile libspecverify.so (the CUDA kernels and their C ABI) in-tree for sm_103a.

The kernel's modes live in separate translation units (csrc/kern_*.cu), which
are compiled in parallel and linked with the host side (csrc/spec_verify.cu,
csrc/tree_build.cpp).
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libspecverify.so")
SOURCES = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
DEPENDS = SOURCES + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + \
    [os.path.join(INCLUDE, "spec_verify.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMPILE_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libspecverify.so")


def up_to_date(out: str = LIB_PATH) -> bool:
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(d) <= t for d in DEPENDS)


def build(force: bool = False, out: str = LIB_PATH, extra_flags=(), verbose: bool = False) -> str:
    """Build the shared library (skipped when newer than its sources)."""
    if not force and up_to_date(out):
        return out
    objdir = out + ".objs.%d" % os.getpid()
    os.makedirs(objdir, exist_ok=True)
    try:
        def compile_one(src):
            obj = os.path.join(objdir, os.path.basename(src) + ".o")
            cmd = [nvcc(), *COMPILE_FLAGS, *extra_flags, "-I", INCLUDE, "-c", "-o", obj, src]
            res = subprocess.run(cmd, capture_output=True, text=True)
            return src, obj, res

        workers = max(1, min(len(SOURCES), os.cpu_count() or 1))
        with concurrent.futures.ThreadPoolExecutor(workers) as ex:
            results = list(ex.map(compile_one, SOURCES))
        log = []
        for src, obj, res in results:
            log.append(res.stdout + res.stderr)
            if res.returncode != 0:
                raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, res.stdout, res.stderr))
        tmp = out + ".tmp.%d" % os.getpid()
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[obj for _, obj, _ in results]]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + res.stdout + res.stderr)
        if verbose:
            print("".join(log))
        os.replace(tmp, out)
    finally:
        shutil.rmtree(objdir, ignore_errors=True)
    return out


if __name__ == "__main__":
    build(force=True, verbose=True)
    print(LIB_PATH)
