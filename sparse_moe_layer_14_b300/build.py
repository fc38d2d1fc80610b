"""Build libbeammoe.so (the C-ABI library of the Beam MoE block) in-tree for sm_103a.

    python -m sparse_moe_layer_14_b300.build [--force]

nvcc cross-compiles without a GPU; the library links the CUDA runtime
statically and resolves the tensor-map encoder through the driver at run time,
so it needs no libcuda at link time.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libbeammoe.so")
SOURCES = ["router.cu", "permute.cu", "expert_gemm.cu", "combine.cu", "norm.cu", "api.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "kernels.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] +
            [os.path.join(ROOT, "include", "beammoe.h"), os.path.abspath(__file__)])


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    if not force and not stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "--shared", "-Xcompiler", "-fPIC,-O3",
           "-Xlinker", "--no-undefined",
           "-I", os.path.join(ROOT, "include"), "-o", tmp, *[os.path.join(CSRC, s) for s in SOURCES]]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    if extra:
        cmd[1:1] = extra
    subprocess.check_call(cmd)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
