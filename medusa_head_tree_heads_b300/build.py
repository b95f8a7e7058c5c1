"""Builds libmedusa.so in-tree with nvcc for sm_103a (B300).

    python -m medusa_head_tree_heads_b300.build [--verbose-ptxas]

Each CUDA source compiles to its own object under _build/ (in parallel, one
nvcc per file), then one nvcc call links the shared library.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libmedusa.so")
OBJ = os.path.join(PKG, "..", "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def build(verbose_ptxas: bool = False, out: str = LIB, extra=()) -> str:
    os.makedirs(OBJ, exist_ok=True)
    srcs = sources()
    objs = [os.path.join(OBJ, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(so):
        src, obj = so
        cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", "-o", obj, src]
        if verbose_ptxas:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)

    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        list(ex.map(compile_one, zip(srcs, objs)))
    subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", out, *objs], check=True)
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
