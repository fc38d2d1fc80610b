"""Seeded synthetic workloads for one Beam MoE block.

The shapes follow the Beam release article (section "Architecture": hidden size
5,120; section "Mixture of Experts": 256 experts in 8 groups of 32, 4 groups
kept, 8 routed per token, SwiGLU intermediate 2,560, combine scale 2.5).

This module draws inputs only. It holds none of the block's arithmetic; the
CUDA path (tests, bench) and the CPU oracle both consume what it produces.
All draws come from the counter-based generator in ``gen.c``, so any slice of
any tensor (one expert's weights, a range of tokens) can be regenerated on its
own and is identical wherever it is generated.

Input recipe (per seed):
  x      [T, d]      bf16  ~ N(0, 1)                       (skewed: + m, m ~ N(0, 0.25 I))
  w_r    [d, E]      fp32  ~ N(0, 1/d)                     (skewed: hot columns + beta * m/|m|)
  gate   [E, I, d]   bf16  ~ N(0, 1/d)    (K-contiguous rows: row i = column i of W_gate)
  up     [E, I, d]   bf16  ~ N(0, 1/d)
  down   [E, d, I]   bf16  ~ N(0, 1/I)    (row n = column n of W_down)
NVFP4 weights are quantised from the same bf16 draws (``quantize_nvfp4``).
"""
from __future__ import annotations

import ctypes
import json
import math
import os
import subprocess
from dataclasses import dataclass, field, replace

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "libgen.so")

# tensor ids of the counter-based streams
TID_X, TID_WR, TID_GATE, TID_UP, TID_DOWN, TID_SKEW_MEAN, TID_TOPK, TID_AUX = 1, 2, 3, 4, 5, 6, 7, 8


@dataclass(frozen=True)
class MoEConfig:
    """Shape of one MoE block and its workload."""

    name: str
    T: int
    d: int
    E: int
    n_groups: int
    topk_groups: int
    top_k: int
    inter: int
    routed_scale: float = 2.5
    wfmt: str = "bf16"  # "bf16" | "nvfp4" | "fp8"
    skew: bool = False
    hot_experts: tuple = field(default_factory=tuple)

    def with_tokens(self, T: int) -> "MoEConfig":
        return replace(self, T=T)


def _hot_set(groups=(1, 5), per_group=8, stride=4, group_size=32):
    return tuple(g * group_size + stride * j for g in groups for j in range(per_group))


CONFIGS = {
    # tiny block for full oracle parity
    "tiny": MoEConfig("tiny", T=64, d=128, E=16, n_groups=4, topk_groups=2, top_k=4, inter=64),
    # Beam shape, decode batch
    "decode": MoEConfig("decode", T=64, d=5120, E=256, n_groups=8, topk_groups=4, top_k=8, inter=2560),
    # Beam shape, prefill with near-uniform routing
    "prefill": MoEConfig("prefill", T=4096, d=5120, E=256, n_groups=8, topk_groups=4, top_k=8, inter=2560),
    # Beam shape, long prefill with 16 hot experts (about 4x mean load) in 2 groups
    "skewed": MoEConfig("skewed", T=32768, d=5120, E=256, n_groups=8, topk_groups=4, top_k=8, inter=2560,
                        skew=True, hot_experts=_hot_set()),
    # Beam shape prefill with NVFP4 expert weights
    "nvfp4": MoEConfig("nvfp4", T=4096, d=5120, E=256, n_groups=8, topk_groups=4, top_k=8, inter=2560,
                       wfmt="nvfp4"),
    # Beam shape prefill with FP8 expert weights (128 x 128 block scales)
    "fp8": MoEConfig("fp8", T=4096, d=5120, E=256, n_groups=8, topk_groups=4, top_k=8, inter=2560,
                     wfmt="fp8"),
}


# --------------------------------------------------------------------------------------
# native generator
# --------------------------------------------------------------------------------------

def build(force: bool = False) -> str:
    """Compile gen.c into libgen.so (in-tree)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        u64, i64, vp, dbl = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
        L.gen_normal_bf16.argtypes = [u64, u64, i64, i64, dbl, vp, i64, vp]
        L.gen_normal_f32.argtypes = [u64, u64, i64, i64, dbl, vp]
        L.gen_normal_f64.argtypes = [u64, u64, i64, i64, dbl, vp]
        L.gen_uniform_f64.argtypes = [u64, u64, i64, i64, vp]
        L.gen_random_topk.argtypes = [u64, u64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      dbl, vp]
        L.gen_quantize_nvfp4.argtypes = [vp, i64, i64, vp, vp]
        L.gen_quantize_fp8.argtypes = [vp, i64, i64, vp, vp]
        L.gen_quantize_fp8.restype = None
        L.gen_quantize_nvfp4.restype = ctypes.c_float
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def normal_bf16(seed, tid, start, count, std, mean=None, out=None) -> np.ndarray:
    """bf16 bit patterns (uint16) of std*N(0,1) (+ mean[column]) for draws [start, start+count)."""
    out = np.empty(count, np.uint16) if out is None else out
    mp, nc = (None, 1) if mean is None else (_ptr(mean), mean.size)
    lib().gen_normal_bf16(seed, tid, start, count, std, mp, nc, _ptr(out))
    return out


def normal_f32(seed, tid, start, count, std) -> np.ndarray:
    out = np.empty(count, np.float32)
    lib().gen_normal_f32(seed, tid, start, count, std, _ptr(out))
    return out


def normal_f64(seed, tid, start, count, std=1.0) -> np.ndarray:
    out = np.empty(count, np.float64)
    lib().gen_normal_f64(seed, tid, start, count, std, _ptr(out))
    return out


def uniform_f64(seed, tid, start, count) -> np.ndarray:
    out = np.empty(count, np.float64)
    lib().gen_uniform_f64(seed, tid, start, count, _ptr(out))
    return out


def random_topk(seed, T, E, K, hot_count=0, hot_prob=0.0, tid=TID_TOPK) -> np.ndarray:
    """[T, K] int32: K distinct experts per token (optionally skewed to experts < hot_count)."""
    out = np.empty((T, K), np.int32)
    lib().gen_random_topk(seed, tid, T, E, K, hot_count, hot_prob, _ptr(out))
    return out


def bf16_to_f32(a: np.ndarray) -> np.ndarray:
    return (a.astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------------------
# workload tensors
# --------------------------------------------------------------------------------------

_SKEW_FILE = os.path.join(_HERE, "skew_beta.json")


def skew_beta() -> float:
    """Router bias strength of the skewed workload, calibrated with the oracle by
    ``calibrate_skew.py`` so the hot experts carry about 4x the mean load."""
    with open(_SKEW_FILE) as f:
        return float(json.load(f)["beta"])


def skew_mean(cfg: MoEConfig, seed: int) -> np.ndarray:
    """Token-mean vector m ~ N(0, 0.25 I) of the skewed workload (double)."""
    return normal_f64(seed, TID_SKEW_MEAN, 0, cfg.d, 0.5)


def gen_x(cfg: MoEConfig, seed: int, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """Activations rows [t0, t1) as bf16 bits, shape [t1-t0, d]."""
    t1 = cfg.T if t1 is None else t1
    mean = skew_mean(cfg, seed) if cfg.skew else None
    out = normal_bf16(seed, TID_X, t0 * cfg.d, (t1 - t0) * cfg.d, 1.0, mean)
    return out.reshape(t1 - t0, cfg.d)


def gen_wr(cfg: MoEConfig, seed: int, beta: float | None = None) -> np.ndarray:
    """Router weight [d, E] fp32 ~ N(0, 1/d); the skewed workload adds
    beta * m/|m| to the hot experts' columns."""
    std = 1.0 / math.sqrt(cfg.d)
    if not cfg.skew:
        return normal_f32(seed, TID_WR, 0, cfg.d * cfg.E, std).reshape(cfg.d, cfg.E)
    base = normal_f64(seed, TID_WR, 0, cfg.d * cfg.E, std).reshape(cfg.d, cfg.E)
    m = skew_mean(cfg, seed)
    b = skew_beta() if beta is None else beta
    hot = list(cfg.hot_experts)
    base[:, hot] += (b / np.linalg.norm(m)) * m[:, None]
    return base.astype(np.float32)


_WSHAPE = {"gate": (TID_GATE, "I", "d"), "up": (TID_UP, "I", "d"), "down": (TID_DOWN, "d", "I")}


def weight_shape(cfg: MoEConfig, which: str):
    _, n, k = _WSHAPE[which]
    dims = {"I": cfg.inter, "d": cfg.d}
    return dims[n], dims[k]


def gen_expert_bf16(cfg: MoEConfig, seed: int, which: str, e0: int, e1: int, out=None) -> np.ndarray:
    """bf16 bits of experts [e0, e1) of matrix `which` ("gate", "up", "down"),
    shape [e1-e0, N, K]; std = 1/sqrt(fan_in) with fan_in = K."""
    tid = _WSHAPE[which][0]
    N, K = weight_shape(cfg, which)
    n = N * K
    flat = None if out is None else out.reshape(-1)
    flat = normal_bf16(seed, tid, e0 * n, (e1 - e0) * n, 1.0 / math.sqrt(K), out=flat)
    return flat.reshape(e1 - e0, N, K)


def quantize_nvfp4(w: np.ndarray):
    """NVFP4 encoding of one bf16 matrix w [N, K] (uint16 bits).

    Returns (packed [N, K/2] uint8, scales [N, K/16] uint8 e4m3, tensor_scale float).
    s_t = amax/(6*448); s_b = e4m3(amax_block/(6*s_t)); q = e2m1(w/(s_b*s_t)).
    """
    N, K = w.shape
    assert K % 16 == 0
    w = np.ascontiguousarray(w)
    packed = np.empty((N, K // 2), np.uint8)
    scales = np.empty((N, K // 16), np.uint8)
    st = lib().gen_quantize_nvfp4(_ptr(w), N, K, _ptr(packed), _ptr(scales))
    return packed, scales, float(st)


def gen_expert_nvfp4(cfg: MoEConfig, seed: int, which: str, e0: int, e1: int):
    """NVFP4 encodings of experts [e0, e1): (packed [n,N,K/2], scales [n,N,K/16], ts [n])."""
    N, K = weight_shape(cfg, which)
    n = e1 - e0
    packed = np.empty((n, N, K // 2), np.uint8)
    scales = np.empty((n, N, K // 16), np.uint8)
    ts = np.empty(n, np.float32)
    for i in range(n):
        w = gen_expert_bf16(cfg, seed, which, e0 + i, e0 + i + 1)[0]
        packed[i], scales[i], ts[i] = quantize_nvfp4(w)
    return packed, scales, ts


def quantize_fp8(w: np.ndarray):
    """FP8 encoding of one bf16 matrix w [N, K] (uint16 bits), 128 x 128 block scales.

    Returns (codes [N, K] uint8 e4m3, scales [N/128, K/128] float32).
    s = amax_block / 448; q = e4m3(w / s), round to nearest even, saturating.
    """
    N, K = w.shape
    assert N % 128 == 0 and K % 128 == 0
    w = np.ascontiguousarray(w)
    codes = np.empty((N, K), np.uint8)
    scales = np.empty((N // 128, K // 128), np.float32)
    lib().gen_quantize_fp8(_ptr(w), N, K, _ptr(codes), _ptr(scales))
    return codes, scales


def gen_expert_fp8(cfg: MoEConfig, seed: int, which: str, e0: int, e1: int):
    """FP8 encodings of experts [e0, e1): (codes [n,N,K], scales [n,N/128,K/128] f32)."""
    N, K = weight_shape(cfg, which)
    n = e1 - e0
    codes = np.empty((n, N, K), np.uint8)
    scales = np.empty((n, N // 128, K // 128), np.float32)
    for i in range(n):
        w = gen_expert_bf16(cfg, seed, which, e0 + i, e0 + i + 1)[0]
        codes[i], scales[i] = quantize_fp8(w)
    return codes, scales


def make_host_inputs(cfg: MoEConfig, seed: int = 0):
    """All inputs of a (small) configuration as host numpy arrays."""
    out = {"x": gen_x(cfg, seed), "w_r": gen_wr(cfg, seed)}
    for which in ("gate", "up", "down"):
        if cfg.wfmt == "bf16":
            out[which] = gen_expert_bf16(cfg, seed, which, 0, cfg.E)
        elif cfg.wfmt == "fp8":
            out[which], out[which + "_sf"] = gen_expert_fp8(cfg, seed, which, 0, cfg.E)
        else:
            p, s, t = gen_expert_nvfp4(cfg, seed, which, 0, cfg.E)
            out[which], out[which + "_sf"], out[which + "_ts"] = p, s, t
    return out
