"""Builds liblora_sgmv.so (the CUDA kernels and the C ABI) in-tree with nvcc
for sm_103a.  Usage: python -m adapter_gemm_02_b300.build [--verbose]."""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "liblora_sgmv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--shared", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                  + [os.path.join(ROOT, "include", "lora_sgmv.h")])


def stale(path: str = LIB) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in sources() + headers())


def build(verbose: bool = False, extra=(), out: str = LIB) -> str:
    """Compiles every .cu file to an object (in parallel, under _build/) and
    links them into `out`."""
    objdir = os.path.join(ROOT, "_build", "obj" + ("" if out == LIB else "_" + os.path.basename(out)))
    os.makedirs(objdir, exist_ok=True)
    flags = [f for f in NVCC_FLAGS if f != "--shared"]
    jobs, objs = [], []
    for src in sources():
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = [_nvcc(), *ARCH, *flags, *extra, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd))
        jobs.append((cmd, subprocess.Popen(cmd)))
    failed = [cmd for cmd, p in jobs if p.wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(1, failed[0])
    subprocess.run([_nvcc(), *ARCH, "--shared", "-Xcompiler", "-fPIC", *objs, "-o", out + ".tmp"], check=True)
    os.replace(out + ".tmp", out)
    return out


TEST_HOOKS_LIB = os.path.join(PKG, "liblora_sgmv_testhooks.so")


def build_test_hooks(verbose: bool = False) -> str:
    """The library as tests build it to exercise bounded waits that run out:
    20 ms per wait, and hooks (lora_test_withhold) that make a kernel
    withhold one signal.  Never loaded by the product path."""
    return build(verbose, extra=("-DLSG_WAIT_LIMIT_NS=20000000ull", "-DLSG_TEST_HOOKS=1"), out=TEST_HOOKS_LIB)


if __name__ == "__main__":
    build(verbose="--verbose" in sys.argv)
    print(LIB)
