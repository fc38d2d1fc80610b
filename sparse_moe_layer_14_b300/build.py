"""Build libbeammoe.so (the C-ABI library of the Beam MoE block) in-tree for sm_103a.

    python -m sparse_moe_layer_14_b300.build [--force] [--debug]

--debug builds libbeammoe_debug.so instead: the same kernels with bounds checks
on every data-dependent index (BEAMMOE_DEBUG_CHECKS; a failed check latches
MOE_DEV_CHECK and skips the access). The binding loads it when the environment
variable BEAMMOE_LIBRARY is "debug".

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
LIB_DEBUG = os.path.join(HERE, "libbeammoe_debug.so")
SOURCES = ["router.cu", "permute.cu", "expert_gemm.cu", "combine.cu", "norm.cu", "api.cu", "noalloc.cu"]
HEADERS = ["common.cuh", "kernels.h", "schedule.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] +
            [os.path.join(ROOT, "include", "beammoe.h"), os.path.abspath(__file__)])


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and not stale(lib):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "--shared", "-Xcompiler", "-fPIC,-O3",
           "-Xlinker", "--no-undefined",
           "-I", os.path.join(ROOT, "include"), "-o", tmp, *[os.path.join(CSRC, s) for s in SOURCES]]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    if debug:
        cmd.insert(1, "-DBEAMMOE_DEBUG_CHECKS")
    if extra:
        cmd[1:1] = extra
    subprocess.check_call(cmd)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
