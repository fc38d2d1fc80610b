"""Beam MoE block forward on one NVIDIA B300: Python binding of libbeammoe.so.

The functions here carry the C entry points' names (include/beammoe.h) and do
argument marshalling only: they check dtypes, shapes and devices of torch
tensors, pass raw device pointers and the current CUDA stream, and raise
MoEError on a non-zero status. Every step of the block runs in the library's
CUDA kernels; there is no CPU path, and a missing library is an error.

Block (Reflection "Beam 1.0" release article, section "Mixture of Experts"):
sigmoid router over E experts in n_groups groups, groups ranked by the sum of
their two best scores, topk_groups kept, top_k experts chosen inside them,
weights normalised to sum 1 then scaled by routed_scale; SwiGLU experts; no
shared expert. FP32 router and SwiGLU product (section "Residual stream").
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _native as N
from ._native import (MOE_DEV_BAD_EXPERT, MOE_DEV_BAD_ROW, MOE_DEV_CHECK, MOE_DEV_DUP_EXPERT, MOE_DEV_OK,  # noqa: F401
                      MOE_DEV_TIMEOUT, MOE_DEV_ZERO_SUM, MOE_W_BF16, MOE_W_FP8, MOE_W_NVFP4, MoeDims, MoeExpertWeights)

__all__ = ["MoEError", "Dims", "ExpertWeights", "moe_workspace_bytes", "moe_workspace_init", "moe_route",
           "moe_permute", "moe_permute_noalloc", "moe_expert_ffn", "moe_combine", "moe_combine_residual",
           "moe_forward", "moe_forward_residual", "moe_pre_norm", "moe_sublayer", "moe_dense_workspace_bytes",
           "moe_dense_mlp",
           "moe_get_device_status", "moe_set_wait_bound", "moe_set_stage_events", "moe_version",
           "allocate_workspace", "allocate_dense_workspace", "library_path",
           "MOE_DEV_OK", "MOE_DEV_BAD_EXPERT", "MOE_DEV_BAD_ROW", "MOE_DEV_DUP_EXPERT", "MOE_DEV_CHECK", "MOE_DEV_TIMEOUT", "MOE_DEV_ZERO_SUM",
           "MOE_W_BF16", "MOE_W_NVFP4", "MOE_W_FP8"]


class MoEError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} returned {N.STATUS_NAMES.get(status, status)}")
        self.status = status


@dataclass(frozen=True)
class Dims:
    """Shape of one MoE block (moe_dims_t)."""

    T: int
    d: int
    E: int
    n_groups: int
    topk_groups: int
    top_k: int
    inter: int
    routed_scale: float = 2.5
    wfmt: int = MOE_W_BF16

    @staticmethod
    def from_config(cfg, T: int | None = None) -> "Dims":
        return Dims(cfg.T if T is None else T, cfg.d, cfg.E, cfg.n_groups, cfg.topk_groups, cfg.top_k, cfg.inter,
                    cfg.routed_scale, _WFMT[cfg.wfmt])

    def c(self) -> MoeDims:
        return MoeDims(self.T, self.d, self.E, self.n_groups, self.topk_groups, self.top_k, self.inter,
                       self.routed_scale, self.wfmt)


@dataclass
class ExpertWeights:
    """Expert weights on the device. bf16: gate/up [E, inter, d], down [E, d, inter] (bf16 or int16 bits).
    NVFP4: gate/up/down packed uint8 [E, N, K/2], *_sf uint8 [E, N, K/16], *_ts float32 [E].
    FP8: gate/up/down e4m3 codes uint8 [E, N, K], *_sf float32 [E, N/128, K/128] (block scales)."""

    gate: torch.Tensor
    up: torch.Tensor
    down: torch.Tensor
    gate_sf: torch.Tensor | None = None
    up_sf: torch.Tensor | None = None
    down_sf: torch.Tensor | None = None
    gate_ts: torch.Tensor | None = None
    up_ts: torch.Tensor | None = None
    down_ts: torch.Tensor | None = None

    def c(self) -> MoeExpertWeights:
        def p(t):
            return None if t is None else _ptr(t)
        return MoeExpertWeights(p(self.gate), p(self.up), p(self.down), p(self.gate_sf), p(self.up_sf),
                                p(self.down_sf), p(self.gate_ts), p(self.up_ts), p(self.down_ts))


def _lib():
    return N.load()


def library_path() -> str:
    return N.LIB_PATH


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(call: str, status: int):
    if status != 0:
        raise MoEError(call, status)


def _expect(t, dtypes, shape, name):
    if t is None:
        return
    if t.dtype not in dtypes:
        raise ValueError(f"{name}: dtype {t.dtype} not in {dtypes}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")


_BF16 = (torch.bfloat16, torch.int16)
_WFMT = {"bf16": MOE_W_BF16, "nvfp4": MOE_W_NVFP4, "fp8": MOE_W_FP8}


def moe_workspace_bytes(dims: Dims) -> int:
    n = _lib().moe_workspace_bytes(ctypes.byref(dims.c()))
    if n == 0:
        raise MoEError("moe_workspace_bytes", N.MOE_ERR_INVALID_ARG)
    return int(n)


def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check("moe_workspace_init", _lib().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def allocate_workspace(dims: Dims, device="cuda") -> torch.Tensor:
    """A zero-headed workspace of moe_workspace_bytes(dims) bytes (torch allocation, 256-B aligned)."""
    ws = torch.empty(moe_workspace_bytes(dims), dtype=torch.uint8, device=device)
    if ws.data_ptr() % 256:
        raise RuntimeError("workspace is not 256-byte aligned")
    moe_workspace_init(ws)
    return ws


def moe_route(dims: Dims, x, w_r, topk_idx, topk_w, ws, stream=None, sel_bias=None):
    """sel_bias: optional [E] fp32 per-expert selection bias (choice only; weights unbiased)."""
    _expect(x, _BF16, (dims.T, dims.d), "x")
    _expect(w_r, (torch.float32,), (dims.d, dims.E), "w_r")
    _expect(topk_idx, (torch.int32,), (dims.T, dims.top_k), "topk_idx")
    _expect(topk_w, (torch.float32,), (dims.T, dims.top_k), "topk_w")
    _expect(sel_bias, (torch.float32,), (dims.E,), "sel_bias")
    _check("moe_route", _lib().moe_route_ex(ctypes.byref(dims.c()), _ptr(x), _ptr(w_r), _ptr(sel_bias), _ptr(topk_idx),
                                            _ptr(topk_w), _ptr(ws), ws.numel(), _stream(stream)))


def moe_permute(dims: Dims, x, topk_idx, counts, offsets, row_token, inv_row, x_perm, ws, stream=None):
    R = dims.T * dims.top_k
    _expect(x, _BF16, (dims.T, dims.d), "x")
    _expect(topk_idx, (torch.int32,), (dims.T, dims.top_k), "topk_idx")
    _expect(counts, (torch.int32,), (dims.E,), "counts")
    _expect(offsets, (torch.int32,), (dims.E + 1,), "offsets")
    _expect(row_token, (torch.int32,), (R,), "row_token")
    _expect(inv_row, (torch.int32,), (R,), "inv_row")
    _expect(x_perm, _BF16, (R, dims.d), "x_perm")
    _check("moe_permute", _lib().moe_permute(ctypes.byref(dims.c()), _ptr(x), _ptr(topk_idx), _ptr(counts),
                                             _ptr(offsets), _ptr(row_token), _ptr(inv_row), _ptr(x_perm), _ptr(ws),
                                             ws.numel(), _stream(stream)))


def moe_permute_noalloc(dims: Dims, x, topk_idx, counts, offsets, row_token, inv_row, x_perm, device_status=None,
                        stream=None):
    """moe_permute without a workspace, for callers that cannot allocate device memory:
    the library's fixed ~1 MiB device scratch is used instead (T <= 16384, E <= 256).
    The first call on a device does a one-time set-up; make it before any stream
    capture. Calls share the scratch, so do not overlap them on the GPU."""
    R = dims.T * dims.top_k
    _expect(x, _BF16, (dims.T, dims.d), "x")
    _expect(topk_idx, (torch.int32,), (dims.T, dims.top_k), "topk_idx")
    _expect(counts, (torch.int32,), (dims.E,), "counts")
    _expect(offsets, (torch.int32,), (dims.E + 1,), "offsets")
    _expect(row_token, (torch.int32,), (R,), "row_token")
    _expect(inv_row, (torch.int32,), (R,), "inv_row")
    _expect(x_perm, _BF16, (R, dims.d), "x_perm")
    _expect(device_status, (torch.int32,), (1,), "device_status")
    _check("moe_permute_noalloc", _lib().moe_permute_noalloc(
        ctypes.byref(dims.c()), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(offsets), _ptr(row_token),
        _ptr(inv_row), _ptr(x_perm), _ptr(device_status), _stream(stream)))


def _check_weights(dims: Dims, w: ExpertWeights):
    if dims.wfmt == MOE_W_BF16:
        _expect(w.gate, _BF16, (dims.E, dims.inter, dims.d), "gate")
        _expect(w.up, _BF16, (dims.E, dims.inter, dims.d), "up")
        _expect(w.down, _BF16, (dims.E, dims.d, dims.inter), "down")
    elif dims.wfmt == MOE_W_FP8:
        for name, n, k in (("gate", dims.inter, dims.d), ("up", dims.inter, dims.d), ("down", dims.d, dims.inter)):
            _expect(getattr(w, name), (torch.uint8,), (dims.E, n, k), name)
            _expect(getattr(w, name + "_sf"), (torch.float32,), (dims.E, n // 128, k // 128), name + "_sf")
            if getattr(w, name + "_sf") is None:
                raise ValueError(f"FP8 weights need {name}_sf")
    else:
        for name, n, k in (("gate", dims.inter, dims.d), ("up", dims.inter, dims.d), ("down", dims.d, dims.inter)):
            _expect(getattr(w, name), (torch.uint8,), (dims.E, n, k // 2), name)
            _expect(getattr(w, name + "_sf"), (torch.uint8,), (dims.E, n, k // 16), name + "_sf")
            _expect(getattr(w, name + "_ts"), (torch.float32,), (dims.E,), name + "_ts")
            if getattr(w, name + "_sf") is None or getattr(w, name + "_ts") is None:
                raise ValueError(f"NVFP4 weights need {name}_sf and {name}_ts")


def moe_expert_ffn(dims: Dims, x_perm, offsets, weights: ExpertWeights, y_perm, ws, stream=None):
    R = dims.T * dims.top_k
    _expect(x_perm, _BF16, (R, dims.d), "x_perm")
    _expect(offsets, (torch.int32,), (dims.E + 1,), "offsets")
    _expect(y_perm, (torch.float32,), (R, dims.d), "y_perm")
    _check_weights(dims, weights)
    _check("moe_expert_ffn", _lib().moe_expert_ffn(ctypes.byref(dims.c()), _ptr(x_perm), _ptr(offsets),
                                                   ctypes.byref(weights.c()), _ptr(y_perm), _ptr(ws), ws.numel(),
                                                   _stream(stream)))


def moe_combine(dims: Dims, y_perm, inv_row, topk_w, out, ws=None, stream=None):
    R = dims.T * dims.top_k
    _expect(y_perm, (torch.float32,), (R, dims.d), "y_perm")
    _expect(inv_row, (torch.int32,), (R,), "inv_row")
    _expect(topk_w, (torch.float32,), (dims.T, dims.top_k), "topk_w")
    _expect(out, _BF16, (dims.T, dims.d), "out")
    _check("moe_combine", _lib().moe_combine(ctypes.byref(dims.c()), _ptr(y_perm), _ptr(inv_row), _ptr(topk_w),
                                             _ptr(out), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def moe_combine_residual(dims: Dims, y_perm, inv_row, topk_w, norm_gain, eps: float, step: int, resid, ws=None,
                         stream=None):
    """Combine + post-norm (RMSNorm with gain norm_gain [d]) + depth-scaled residual update of
    resid [T, d] in place: resid = sqrt((step-1)/step) resid + (1/sqrt(step)) RMSNorm(out)."""
    R = dims.T * dims.top_k
    _expect(y_perm, (torch.float32,), (R, dims.d), "y_perm")
    _expect(inv_row, (torch.int32,), (R,), "inv_row")
    _expect(topk_w, (torch.float32,), (dims.T, dims.top_k), "topk_w")
    _expect(norm_gain, _BF16, (dims.d,), "norm_gain")
    _expect(resid, _BF16, (dims.T, dims.d), "resid")
    _check("moe_combine_residual", _lib().moe_combine_residual(
        ctypes.byref(dims.c()), _ptr(y_perm), _ptr(inv_row), _ptr(topk_w), _ptr(norm_gain), float(eps), int(step),
        _ptr(resid), _ptr(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def moe_forward_residual(dims: Dims, x, w_r, weights: ExpertWeights, norm_gain, eps: float, step: int, resid, ws,
                         topk_idx=None, counts=None, stream=None, sel_bias=None):
    """moe_forward whose last stage is the post-norm and residual update of resid (in place)."""
    _expect(x, _BF16, (dims.T, dims.d), "x")
    _expect(w_r, (torch.float32,), (dims.d, dims.E), "w_r")
    _expect(norm_gain, _BF16, (dims.d,), "norm_gain")
    _expect(resid, _BF16, (dims.T, dims.d), "resid")
    _expect(topk_idx, (torch.int32,), (dims.T, dims.top_k), "topk_idx")
    _expect(counts, (torch.int32,), (dims.E,), "counts")
    _expect(sel_bias, (torch.float32,), (dims.E,), "sel_bias")
    _check_weights(dims, weights)
    _check("moe_forward_residual", _lib().moe_forward_residual(
        ctypes.byref(dims.c()), _ptr(x), _ptr(w_r), _ptr(sel_bias), ctypes.byref(weights.c()), _ptr(norm_gain),
        float(eps), int(step), _ptr(resid), _ptr(topk_idx), _ptr(counts), _ptr(ws), ws.numel(), _stream(stream)))


def moe_pre_norm(dims: Dims, h, gain, eps: float, x, stream=None):
    """x = bf16(RMSNorm(h) * gain) per token row, FP32 (x must not overlap h)."""
    _expect(h, _BF16, (dims.T, dims.d), "h")
    _expect(gain, _BF16, (dims.d,), "gain")
    _expect(x, _BF16, (dims.T, dims.d), "x")
    _check("moe_pre_norm", _lib().moe_pre_norm(ctypes.byref(dims.c()), _ptr(h), _ptr(gain), float(eps), _ptr(x),
                                               _stream(stream)))


def moe_sublayer(dims: Dims, resid, pre_gain, post_gain, eps: float, step: int, w_r, weights: ExpertWeights, x, ws,
                 topk_idx=None, counts=None, stream=None, sel_bias=None):
    """The MoE sublayer: x = pre-norm(resid) (into x), the block forward on x, then the post-norm and
    depth-scaled update of resid in place."""
    _expect(resid, _BF16, (dims.T, dims.d), "resid")
    _expect(pre_gain, _BF16, (dims.d,), "pre_gain")
    _expect(post_gain, _BF16, (dims.d,), "post_gain")
    _expect(w_r, (torch.float32,), (dims.d, dims.E), "w_r")
    _expect(x, _BF16, (dims.T, dims.d), "x")
    _expect(topk_idx, (torch.int32,), (dims.T, dims.top_k), "topk_idx")
    _expect(counts, (torch.int32,), (dims.E,), "counts")
    _expect(sel_bias, (torch.float32,), (dims.E,), "sel_bias")
    _check_weights(dims, weights)
    _check("moe_sublayer", _lib().moe_sublayer(
        ctypes.byref(dims.c()), _ptr(resid), _ptr(pre_gain), _ptr(post_gain), float(eps), int(step), _ptr(w_r),
        _ptr(sel_bias), ctypes.byref(weights.c()), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(ws), ws.numel(),
        _stream(stream)))


def _dense(dims: Dims) -> Dims:
    return Dims(dims.T, dims.d, 1, 1, 1, 1, dims.inter, 1.0, dims.wfmt)


def moe_dense_workspace_bytes(dims: Dims) -> int:
    n = _lib().moe_dense_workspace_bytes(ctypes.byref(dims.c()))
    if n == 0:
        raise MoEError("moe_dense_workspace_bytes", N.MOE_ERR_INVALID_ARG)
    return int(n)


def allocate_dense_workspace(dims: Dims, device="cuda") -> torch.Tensor:
    """A zero-headed workspace of moe_dense_workspace_bytes(dims) bytes."""
    ws = torch.empty(moe_dense_workspace_bytes(dims), dtype=torch.uint8, device=device)
    if ws.data_ptr() % 256:
        raise RuntimeError("workspace is not 256-byte aligned")
    moe_workspace_init(ws)
    return ws


def moe_dense_mlp(dims: Dims, x, weights: ExpertWeights, out, ws, stream=None):
    """Dense SwiGLU MLP (one expert's layout, E = 1): out = bf16(bf16(silu(x Wg) * (x Wu)) Wd)."""
    _expect(x, _BF16, (dims.T, dims.d), "x")
    _expect(out, _BF16, (dims.T, dims.d), "out")
    _check_weights(_dense(dims), weights)
    _check("moe_dense_mlp", _lib().moe_dense_mlp(ctypes.byref(dims.c()), _ptr(x), ctypes.byref(weights.c()), _ptr(out),
                                                 _ptr(ws), ws.numel(), _stream(stream)))


def moe_forward(dims: Dims, x, w_r, weights: ExpertWeights, out, ws, topk_idx=None, counts=None, stream=None,
                sel_bias=None):
    """sel_bias: optional [E] fp32 per-expert selection bias (choice only; weights unbiased)."""
    _expect(x, _BF16, (dims.T, dims.d), "x")
    _expect(w_r, (torch.float32,), (dims.d, dims.E), "w_r")
    _expect(out, _BF16, (dims.T, dims.d), "out")
    _expect(topk_idx, (torch.int32,), (dims.T, dims.top_k), "topk_idx")
    _expect(counts, (torch.int32,), (dims.E,), "counts")
    _expect(sel_bias, (torch.float32,), (dims.E,), "sel_bias")
    _check_weights(dims, weights)
    if sel_bias is None:
        rc = _lib().moe_forward(ctypes.byref(dims.c()), _ptr(x), _ptr(w_r), ctypes.byref(weights.c()), _ptr(out),
                                _ptr(topk_idx), _ptr(counts), _ptr(ws), ws.numel(), _stream(stream))
    else:
        rc = _lib().moe_forward_ex(ctypes.byref(dims.c()), _ptr(x), _ptr(w_r), _ptr(sel_bias),
                                   ctypes.byref(weights.c()), _ptr(out), _ptr(topk_idx), _ptr(counts), _ptr(ws),
                                   ws.numel(), _stream(stream))
    _check("moe_forward", rc)


def moe_get_device_status(ws, clear: bool = False, stream=None) -> int:
    code = ctypes.c_int32(0)
    _check("moe_get_device_status", _lib().moe_get_device_status(_ptr(ws), _stream(stream), 1 if clear else 0,
                                                                 ctypes.byref(code)))
    return code.value


def moe_set_wait_bound(spins: int):
    _lib().moe_set_wait_bound(int(spins))


def moe_set_stage_events(events):
    """Record device events between the stages of later moe_forward calls (None: off).
    `events` is a list of 6 torch.cuda.Event(enable_timing=True); each is recorded
    once here so that its CUDA handle exists."""
    if events is None:
        _check("moe_set_stage_events", _lib().moe_set_stage_events(None, 0))
        return
    if len(events) < 6:
        raise ValueError("need 6 events")
    for ev in events:
        if ev.cuda_event == 0:
            ev.record()
    arr = (ctypes.c_void_p * len(events))(*[ev.cuda_event for ev in events])
    _check("moe_set_stage_events", _lib().moe_set_stage_events(arr, len(events)))


def moe_version() -> str:
    return _lib().moe_version().decode()
