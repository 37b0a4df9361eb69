"""Build libspecverify.so in-tree with nvcc for sm_103a (GB300).

One translation unit, one -gencode, no cmake: a single nvcc invocation that
takes well under a minute.  The library links the CUDA runtime statically so
it only needs the driver at run time; PyTorch's own runtime is not involved.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "spec_verify.cu")
HDR = os.path.join(ROOT, "include", "spec_verify.h")
LIB = os.path.join(PKG, "libspecverify.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found: set CUDA_HOME")
    return found


def nvcc_command(out: str = LIB, extra=()) -> list:
    return [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "--shared",
            "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
            "-I", os.path.join(ROOT, "include"), "-cudart", "static",
            *extra, "-o", out, SRC]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile the CUDA library if it is missing or older than its sources."""
    if not force and not stale() and not extra:
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp, extra)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        print(" ".join(cmd))
        print(res.stdout)
        print(res.stderr)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed building libspecverify.so")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True, extra=("-Xptxas", "-v"))
