"""Build libspecverify.so in-tree with nvcc for sm_103a (GB300).

Five translation units (verification, sampling, the LM-head-fused
verification, tree verification, the benchmark's read probe), one -gencode, no cmake: each
is compiled by its own nvcc process in parallel, then one nvcc call links the
shared library.  The library links the CUDA runtime statically so it only
needs the driver at run time; PyTorch's own runtime is not involved.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SRCS = [os.path.join(CSRC, "spec_verify.cu"), os.path.join(CSRC, "spec_sample.cu"),
        os.path.join(CSRC, "spec_lmhead.cu"), os.path.join(CSRC, "spec_tree.cu"),
        os.path.join(CSRC, "bench_read.cu")]
DEPS = [os.path.join(CSRC, "device_common.cuh"), os.path.join(CSRC, "internal.h"),
        os.path.join(CSRC, "resolve.cuh"), os.path.join(CSRC, "exp2_table.h"),
        os.path.join(ROOT, "include", "spec_lmhead.h"),
        os.path.join(ROOT, "include", "spec_verify.h"),
        os.path.join(ROOT, "include", "spec_sample.h"),
        os.path.join(ROOT, "include", "spec_bench.h"),
        os.path.join(ROOT, "include", "spec_tree.h")]
SRC = SRCS[0]
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


def compile_command(src: str, obj: str, extra=()) -> list:
    return [nvcc_path(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-c",
            "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
            "-I", os.path.join(ROOT, "include"), *extra, "-o", obj, src]


def link_command(objs, out: str) -> list:
    return [nvcc_path(), *ARCH, "--shared", "-cudart", "static", "-o", out, *objs]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (*SRCS, *DEPS, __file__))


def _run(cmd, verbose):
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        print(" ".join(cmd))
        print(res.stdout)
        print(res.stderr)
    return res.returncode


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile the CUDA library if it is missing or older than its sources."""
    if not force and not stale() and not extra:
        return LIB
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(CSRC, os.path.basename(s) + tag + ".o") for s in SRCS]
    try:
        with ThreadPoolExecutor(len(SRCS)) as ex:
            rcs = list(ex.map(lambda so: _run(compile_command(so[0], so[1], extra), verbose),
                              zip(SRCS, objs)))
        if any(rcs):
            raise RuntimeError("nvcc failed compiling the CUDA sources")
        tmp = LIB + tag
        if _run(link_command(objs, tmp), verbose):
            raise RuntimeError("nvcc failed linking libspecverify.so")
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True, extra=("-Xptxas", "-v"))
