"""C-ABI library checks that need no GPU: it loads, exports every entry point
include/beammoe.h declares, sizes workspaces, and rejects bad arguments on the
host before any CUDA call. Also: the product package never reaches the oracle."""
import ctypes
import os
import re

import pytest

import sparse_moe_layer_14_b300 as bm
from sparse_moe_layer_14_b300 import _native as N
from sparse_moe_layer_14_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beammoe.h")


@pytest.fixture(scope="module")
def lib():
    build()
    return N.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:moe_status_t|size_t|void|const char\s*\*)\s*(moe_\w+)\s*\(", src, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward",
                     "moe_workspace_bytes", "moe_get_device_status"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    assert set(declared_functions()) <= set(N.EXPORTS) | set(declared_functions())
    assert "sm_103a" in bm.moe_version()


def test_debug_build_exports_every_declared_symbol():
    """The bounds-checked build (BEAMMOE_LIBRARY=debug) is the same library with extra checks."""
    path = build(debug=True)
    dbg = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(dbg, name), f"{name} not exported by the debug build"


def _dims(**kw):
    base = dict(T=64, d=5120, E=256, n_groups=8, topk_groups=4, top_k=8, inter=2560, routed_scale=2.5, wfmt=0)
    base.update(kw)
    return N.MoeDims(**base)


def test_workspace_bytes(lib):
    n64 = lib.moe_workspace_bytes(ctypes.byref(_dims()))
    n4k = lib.moe_workspace_bytes(ctypes.byref(_dims(T=4096)))
    assert 0 < n64 < n4k
    R = 4096 * 8
    # x_perm (bf16) + h (bf16) + y (fp32) dominate: R*(2d + 2I + 4d) bytes
    assert n4k >= R * (2 * 5120 + 2 * 2560 + 4 * 5120)
    assert lib.moe_workspace_bytes(ctypes.byref(_dims(T=0))) > 0


@pytest.mark.parametrize("bad,code", [
    (dict(T=-1), N.MOE_ERR_INVALID_ARG), (dict(E=250), N.MOE_ERR_INVALID_ARG), (dict(topk_groups=9), N.MOE_ERR_INVALID_ARG),
    (dict(top_k=200), N.MOE_ERR_INVALID_ARG), (dict(wfmt=7), N.MOE_ERR_INVALID_ARG), (dict(d=5000), N.MOE_ERR_UNSUPPORTED),
    (dict(inter=100), N.MOE_ERR_UNSUPPORTED), (dict(E=512, n_groups=16), N.MOE_ERR_UNSUPPORTED),
    (dict(n_groups=64, E=256, topk_groups=4), N.MOE_ERR_UNSUPPORTED), (dict(T=5_000_000), N.MOE_ERR_UNSUPPORTED),
    (dict(routed_scale=float("nan")), N.MOE_ERR_INVALID_ARG)])
def test_bad_dims_rejected_on_host(lib, bad, code):
    d = _dims(**bad)
    assert lib.moe_workspace_bytes(ctypes.byref(d)) == 0
    w = N.MoeExpertWeights()
    fake = ctypes.c_void_p(1 << 20)
    rc = lib.moe_forward(ctypes.byref(d), fake, fake, ctypes.byref(w), fake, None, None, fake, 1 << 40, None)
    assert rc == code


def test_null_and_misaligned_pointers_rejected(lib):
    d = _dims()
    fake = ctypes.c_void_p(1 << 20)
    w = N.MoeExpertWeights(fake, fake, fake)
    ws_bytes = lib.moe_workspace_bytes(ctypes.byref(d))
    assert lib.moe_forward(ctypes.byref(d), None, fake, ctypes.byref(w), fake, None, None, fake, ws_bytes, None) == N.MOE_ERR_INVALID_ARG
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert lib.moe_forward(ctypes.byref(d), odd, fake, ctypes.byref(w), fake, None, None, fake, ws_bytes, None) == N.MOE_ERR_INVALID_ARG
    w_bad = N.MoeExpertWeights(fake, None, fake)
    assert lib.moe_forward(ctypes.byref(d), fake, fake, ctypes.byref(w_bad), fake, None, None, fake, ws_bytes, None) == N.MOE_ERR_INVALID_ARG
    # workspace too small or misaligned
    assert lib.moe_forward(ctypes.byref(d), fake, fake, ctypes.byref(w), fake, None, None, fake, ws_bytes - 1, None) == N.MOE_ERR_WORKSPACE
    assert lib.moe_forward(ctypes.byref(d), fake, fake, ctypes.byref(w), fake, None, None, ctypes.c_void_p((1 << 20) + 16), ws_bytes, None) == N.MOE_ERR_WORKSPACE
    # NVFP4 needs scales
    d4 = _dims(wfmt=1)
    assert lib.moe_forward(ctypes.byref(d4), fake, fake, ctypes.byref(w), fake, None, None, fake, ws_bytes, None) == N.MOE_ERR_INVALID_ARG
    # FP8 needs 4-byte aligned block scales
    d8 = _dims(wfmt=N.MOE_W_FP8)
    ws8 = lib.moe_workspace_bytes(ctypes.byref(d8))
    assert lib.moe_forward(ctypes.byref(d8), fake, fake, ctypes.byref(w), fake, None, None, fake, ws8, None) == N.MOE_ERR_INVALID_ARG
    w8 = N.MoeExpertWeights(fake, fake, fake, fake, ctypes.c_void_p((1 << 20) + 2), fake)
    assert lib.moe_forward(ctypes.byref(d8), fake, fake, ctypes.byref(w8), fake, None, None, fake, ws8, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_init(None, 4096, None) == N.MOE_ERR_WORKSPACE
    code = ctypes.c_int32()
    assert lib.moe_get_device_status(None, None, 0, ctypes.byref(code)) == N.MOE_ERR_INVALID_ARG


def test_empty_batch_is_a_host_noop(lib):
    d = _dims(T=0)
    fake = ctypes.c_void_p(1 << 20)
    w = N.MoeExpertWeights(fake, fake, fake)
    assert lib.moe_forward(ctypes.byref(d), fake, fake, ctypes.byref(w), fake, None, None, fake, 1 << 30, None) == N.MOE_OK
    assert lib.moe_route(ctypes.byref(d), fake, fake, fake, fake, fake, 1 << 30, None) == N.MOE_OK


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="missing"):
        N.load(str(tmp_path / "libbeammoe.so"))


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "sparse_moe_layer_14_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+(oracle|workload)\b", src, re.M), f
                assert "liboracle" not in src and "oracle.c" not in src, f


def test_binding_exports_every_public_call():
    """Every name in the package's __all__ exists, and every C entry point the header declares
    that takes block arguments has a Python wrapper of the same name."""
    for name in bm.__all__:
        assert hasattr(bm, name), name
    wrapped = {n for n in declared_functions() if hasattr(bm, n)}
    for required in ("moe_route", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_forward",
                     "moe_forward_residual", "moe_combine_residual", "moe_dense_mlp", "moe_permute_noalloc",
                     "moe_pre_norm", "moe_sublayer"):
        assert required in wrapped, required


def test_pre_norm_and_sublayer_host_checks(lib):
    """Host-side validation of moe_pre_norm / moe_sublayer: nothing is launched."""
    fake = ctypes.c_void_p(1 << 20)
    d = _dims(T=4, d=128)
    # x overlapping h, a d that is not a multiple of 64, a negative eps, a misaligned gain
    assert lib.moe_pre_norm(ctypes.byref(d), fake, fake, 1e-6, ctypes.c_void_p((1 << 20) + 512), None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_pre_norm(ctypes.byref(_dims(T=4, d=100)), fake, fake, 1e-6, fake, None) == N.MOE_ERR_UNSUPPORTED
    far = ctypes.c_void_p(1 << 24)
    assert lib.moe_pre_norm(ctypes.byref(d), fake, fake, -1.0, far, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_pre_norm(ctypes.byref(d), fake, ctypes.c_void_p((1 << 20) + 8), 1e-6, far, None) == N.MOE_ERR_INVALID_ARG
    assert lib.moe_pre_norm(ctypes.byref(_dims(T=0, d=128)), None, None, 1e-6, None, None) == N.MOE_OK
    w = N.MoeExpertWeights(fake, fake, fake)
    dd = _dims()
    ws_bytes = lib.moe_workspace_bytes(ctypes.byref(dd))
    # step 0 and d > 8192 are rejected before the pre-norm is enqueued
    assert lib.moe_sublayer(ctypes.byref(dd), fake, fake, fake, 1e-6, 0, fake, None, ctypes.byref(w), far,
                            None, None, fake, ws_bytes, None) == N.MOE_ERR_INVALID_ARG
    big = _dims(d=16384)
    assert lib.moe_sublayer(ctypes.byref(big), fake, fake, fake, 1e-6, 2, fake, None, ctypes.byref(w),
                            ctypes.c_void_p(1 << 30), None, None, fake, ws_bytes, None) == N.MOE_ERR_UNSUPPORTED


def test_header_is_plain_c_and_links_against_the_library(tmp_path):
    """A C program that includes the header, takes the address of every declared call and links
    against the built library: the boundary needs no C++ and no torch."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = tmp_path / "use.c"
    src.write_text('#include "beammoe.h"\n#include <stdio.h>\nint main(void) {\n  const void* f[] = {'
                   + ", ".join(f"(const void*){n}" for n in names) + "};\n"
                   '  printf("%d %s\\n", (int)(sizeof f / sizeof f[0]), moe_version());\n  return 0;\n}\n')
    lib_path = bm.library_path()
    exe = tmp_path / "use"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                           "-o", str(exe), lib_path, f"-Wl,-rpath,{os.path.dirname(lib_path)}"])
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == len(names) and "sm_103a" in " ".join(out[1:])
