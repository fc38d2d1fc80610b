"""ctypes declarations of libbeammoe.so (include/beammoe.h)."""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# BEAMMOE_LIBRARY=debug selects the build with bounds checks (python -m sparse_moe_layer_14_b300.build --debug)
LIB_PATH = os.path.join(HERE, "libbeammoe_debug.so" if os.environ.get("BEAMMOE_LIBRARY") == "debug" else "libbeammoe.so")

# moe_status_t
MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_WORKSPACE, MOE_ERR_CUDA = 0, 1, 2, 3, 4
MOE_ERR_DEVICE_STATUS, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_SCRATCH_LIMIT = 5, 6, 7
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
                4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_STATUS", 6: "MOE_ERR_DEVICE_TIMEOUT",
                7: "MOE_ERR_SCRATCH_LIMIT"}
# moe_device_code_t
MOE_DEV_OK, MOE_DEV_BAD_EXPERT, MOE_DEV_BAD_ROW, MOE_DEV_DUP_EXPERT, MOE_DEV_TIMEOUT, MOE_DEV_ZERO_SUM = 0, 1, 2, 3, 6, 7
MOE_DEV_CHECK = 8  # debug build only
# moe_wfmt_t
MOE_W_BF16, MOE_W_NVFP4, MOE_W_FP8 = 0, 1, 2

EXPORTS = ["moe_workspace_bytes", "moe_workspace_init", "moe_route", "moe_permute", "moe_expert_ffn",
           "moe_combine", "moe_forward", "moe_get_device_status", "moe_set_wait_bound", "moe_set_stage_events",
           "moe_version", "moe_permute_noalloc", "moe_dense_workspace_bytes", "moe_dense_mlp", "moe_route_ex",
           "moe_forward_ex", "moe_combine_residual", "moe_forward_residual", "moe_pre_norm", "moe_sublayer"]


class MoeDims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("d", ctypes.c_int32), ("E", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("inter", ctypes.c_int32), ("routed_scale", ctypes.c_float), ("wfmt", ctypes.c_int32)]


class MoeExpertWeights(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p),
                ("gate_sf", ctypes.c_void_p), ("up_sf", ctypes.c_void_p), ("down_sf", ctypes.c_void_p),
                ("gate_ts", ctypes.c_void_p), ("up_ts", ctypes.c_void_p), ("down_ts", ctypes.c_void_p)]


_lib = None


def load(path: str = LIB_PATH):
    """Load the library and declare every entry point. Raises if it is not built."""
    global _lib
    if _lib is not None and path == LIB_PATH:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m sparse_moe_layer_14_b300.build`"
                           + (" --debug" if path.endswith("_debug.so") else ""))
    L = ctypes.CDLL(path)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    pd, pw = ctypes.POINTER(MoeDims), ctypes.POINTER(MoeExpertWeights)
    L.moe_workspace_bytes.argtypes = [pd]
    L.moe_workspace_bytes.restype = sz
    L.moe_workspace_init.argtypes = [vp, sz, vp]
    L.moe_workspace_init.restype = st
    L.moe_route.argtypes = [pd, vp, vp, vp, vp, vp, sz, vp]
    L.moe_route.restype = st
    L.moe_permute.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_permute.restype = st
    L.moe_expert_ffn.argtypes = [pd, vp, vp, pw, vp, vp, sz, vp]
    L.moe_expert_ffn.restype = st
    L.moe_combine.argtypes = [pd, vp, vp, vp, vp, vp, sz, vp]
    L.moe_combine.restype = st
    L.moe_forward.argtypes = [pd, vp, vp, pw, vp, vp, vp, vp, sz, vp]
    L.moe_route_ex.argtypes = [pd, vp, vp, vp, vp, vp, vp, sz, vp]
    L.moe_route_ex.restype = st
    L.moe_forward_ex.argtypes = [pd, vp, vp, vp, pw, vp, vp, vp, vp, sz, vp]
    L.moe_forward_ex.restype = st
    L.moe_combine_residual.argtypes = [pd, vp, vp, vp, vp, ctypes.c_float, ctypes.c_int32, vp, vp, sz, vp]
    L.moe_combine_residual.restype = st
    L.moe_forward_residual.argtypes = [pd, vp, vp, vp, pw, vp, ctypes.c_float, ctypes.c_int32, vp, vp, vp, vp, sz,
                                       vp]
    L.moe_forward_residual.restype = st
    L.moe_pre_norm.argtypes = [pd, vp, vp, ctypes.c_float, vp, vp]
    L.moe_pre_norm.restype = st
    L.moe_sublayer.argtypes = [pd, vp, vp, vp, ctypes.c_float, ctypes.c_int32, vp, vp, pw, vp, vp, vp, vp, sz, vp]
    L.moe_sublayer.restype = st
    L.moe_forward.restype = st
    L.moe_get_device_status.argtypes = [vp, vp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    L.moe_get_device_status.restype = st
    L.moe_set_wait_bound.argtypes = [ctypes.c_int64]
    L.moe_set_wait_bound.restype = None
    L.moe_permute_noalloc.argtypes = [pd, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.moe_permute_noalloc.restype = st
    L.moe_set_stage_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32]
    L.moe_set_stage_events.restype = st
    L.moe_dense_workspace_bytes.argtypes = [pd]
    L.moe_dense_workspace_bytes.restype = sz
    L.moe_dense_mlp.argtypes = [pd, vp, pw, vp, vp, sz, vp]
    L.moe_dense_mlp.restype = st
    L.moe_version.argtypes = []
    L.moe_version.restype = ctypes.c_char_p
    if path == LIB_PATH:
        _lib = L
    return L
