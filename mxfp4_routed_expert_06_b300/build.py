"""Build libk3moe.so (the CUDA path and its C ABI) in-tree for sm_103a.

Usage: ``python mxfp4_routed_expert_06_b300/build.py [--force]`` (run it by path: importing
the package itself needs the built library).  nvcc cross-compiles
without a GPU, so this also runs on a CPU-only machine.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libk3moe.so")
SOURCES = ["capi.cu", "pack.cu", "router.cu", "decode_ffn.cu", "noalloc.cu", "glue.cu", "gemm_tc.cu", "cachesim.cu",
           "misscopy.cu"]
HEADERS = ["k3moe_internal.cuh"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-Xptxas", "-warn-spills"]


def _deps():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "k3moe.h")]
            + [os.path.abspath(__file__)])


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


SAN_LIB = os.path.join(HERE, "libk3moe_san.so")
# (nvcc splits -Xcompiler values at commas: one flag per sanitizer)
SAN_FLAGS = ["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined", "-Xcompiler",
             "-fno-omit-frame-pointer", "-Xcompiler", "-fno-sanitize-recover=all", "-g"]


def build(force: bool = False, verbose: bool = False, checks: bool = False, sanitize: bool = False) -> str:
    """checks=True builds the self-checking variant (K3MOE_DEVICE_CHECKS): device-side copy
    addresses are checked and a failure is recorded and skipped instead of faulting.
    sanitize=True builds libk3moe_san.so instead: the same library with its host code (argument
    checks, workspace, cache bookkeeping, the cache simulator) under AddressSanitizer and
    UndefinedBehaviorSanitizer, for the plain C driver in tests/c/."""
    out = SAN_LIB if sanitize else LIB
    if not force and not checks and os.path.exists(out) and not any(
            os.path.getmtime(p) > os.path.getmtime(out) for p in _deps()):
        return out
    objdir = os.path.join(HERE, "_build_san" if sanitize else "_build")
    os.makedirs(objdir, exist_ok=True)
    extra = (["-DK3MOE_DEVICE_CHECKS"] if checks else []) + (SAN_FLAGS if sanitize else [])
    objs = []
    for src in SOURCES:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = ["nvcc", *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.check_call(cmd)
        objs.append(obj)
    tmp = out + ".tmp"
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-shared", *objs, "-o", tmp,
                           "-lcudart", *(["-Xcompiler", "-fsanitize=address", "-Xcompiler", "-fsanitize=undefined"]
                                       if sanitize else [])])
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv or "--checks" in sys.argv, verbose="-v" in sys.argv,
                checks="--checks" in sys.argv, sanitize="--sanitize" in sys.argv))
