"""Compile libspecverify.so (the CUDA kernels and their C ABI) in-tree for sm_103a."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libspecverify.so")
SOURCES = [os.path.join(CSRC, "spec_verify.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, f) for f in ("verify_kernels.cuh", "tree_mask.cuh", "ptx.cuh")] + \
    [os.path.join(INCLUDE, "spec_verify.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-shared", "-Xptxas", "-v"]


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
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-o", tmp, *SOURCES]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
    if verbose:
        print(res.stdout + res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    build(force=True, verbose=True)
    print(LIB_PATH)
