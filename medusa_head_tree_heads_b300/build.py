"""Builds libmedusa.so in-tree with nvcc for sm_103a (B300).

    python -m medusa_head_tree_heads_b300.build [--verbose-ptxas]
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libmedusa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def build(verbose_ptxas: bool = False, out: str = LIB, extra=()) -> str:
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-O2",
           "-cudart", "shared", "--expt-relaxed-constexpr", "-o", out, *extra, *sources()]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(PKG, "..", "include", "medusa.h")]
    return all(os.path.getmtime(d) <= t for d in deps if os.path.exists(d))


if __name__ == "__main__":
    build(verbose_ptxas="--verbose-ptxas" in sys.argv)
    print(LIB)
