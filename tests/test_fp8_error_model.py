"""Where the FP8 typical-error bar comes from (CPU only).

The expert GEMMs take bf16 operands, so FP8 weights are dequantised on chip as
bf16(fp32(e4m3 * block scale)); the oracle keeps the exact product. This test
repeats exactly those roundings in numpy (bf16 weights, FP32 SwiGLU, bf16 h,
FP32 y) and measures their error against the oracle: it must sit below the
bar the GPU tests use, and removing the weight rounding must bring it back
below the bf16 bar. A bar that merely hid a kernel bug would not be explained
by this model.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from support import RMS_BAR, TOL_FP8



def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).float().numpy()


def _model(x, row_e, host, d, inter, round_weights):
    vals = np.array([O.e4m3_value(c) for c in range(256)])
    deq = {}
    for which in ("gate", "up", "down"):
        q = vals[host[which]]
        s = host[which + "_sf"]
        sc = np.repeat(np.repeat(s, 128, axis=1), 128, axis=2)
        deq[which] = (_bf16(q.astype(np.float32) * sc) if round_weights else q * sc.astype(np.float64))
    xf = W.bf16_to_f32(x).astype(np.float64)
    y = np.empty((len(row_e), d))
    for i, e in enumerate(row_e):
        g = (deq["gate"][e] @ xf[i]).astype(np.float32)
        u = (deq["up"][e] @ xf[i]).astype(np.float32)
        h = _bf16(g / (1 + np.exp(-g)) * u).astype(np.float64)
        y[i] = (deq["down"][e] @ h).astype(np.float32)
    return y


def _case(n=160, d=256, inter=384, E=2, seed=3):
    cfg = W.MoEConfig("fp8m", T=n, d=d, E=E, n_groups=1, topk_groups=1, top_k=1, inter=inter, wfmt="fp8")
    host = {}
    for which in ("gate", "up", "down"):
        host[which], host[which + "_sf"] = W.gen_expert_fp8(cfg, seed, which, 0, E)
    x = W.normal_bf16(seed, W.TID_X, 0, n * d, 1.0).reshape(n, d)
    row_e = np.arange(n, dtype=np.int32) % E
    ref = O.ffn_rows(row_e, x, host, d, inter, "fp8")
    return x, row_e, host, d, inter, ref


def test_fp8_bar_is_the_weight_rounding():
    x, row_e, host, d, inter, ref = _case()
    rms = np.sqrt(np.mean(ref ** 2))
    rel = {rw: np.sqrt(np.mean((_model(x, row_e, host, d, inter, rw) - ref) ** 2)) / rms for rw in (True, False)}
    assert 2.5e-3 < rel[True] < RMS_BAR["fp8"], rel
    assert rel[False] < RMS_BAR["bf16"], rel


def _model_batched(x, row_e, host, E, round_weights=True):
    """_model with each expert's rows in one matrix product (the Beam shape is large)."""
    vals = np.array([O.e4m3_value(c) for c in range(256)], np.float32)
    xf = W.bf16_to_f32(x).astype(np.float64)
    y = np.empty((len(row_e), host["down"].shape[1]))
    for e in range(E):
        deq = {}
        for which in ("gate", "up", "down"):
            sc = np.repeat(np.repeat(host[which + "_sf"][e], 128, axis=0), 128, axis=1)
            w = vals[host[which][e]] * sc
            deq[which] = (_bf16(w) if round_weights else w).astype(np.float64)
        r = np.nonzero(row_e == e)[0]
        g = (xf[r] @ deq["gate"].T).astype(np.float32)
        u = (xf[r] @ deq["up"].T).astype(np.float32)
        h = _bf16(g / (1 + np.exp(-g)) * u).astype(np.float64)
        y[r] = (h @ deq["down"].T).astype(np.float32)
    return y


def test_fp8_max_bar_follows_from_the_model():
    """The max-error bar of the FP8 tests, from the model: over n compared elements its max error
    behaves like c * RMS * sqrt(2 ln n), with c from 1.0 (Beam shape, d = 5120) to ~1.45 (small
    reduction lengths, d = 256: fewer terms, heavier tails). Over the largest GPU comparison
    (~4e6 elements) the worst shape's max is expected at c * RMS * sqrt(2 ln 4e6) ~ 2.8e-2 of the
    output RMS; TOL_FP8 sits 1.15-2x above that (not at the NVFP4 bar)."""
    worst = 0.0
    for n, d, inter in ((384, 256, 384), (96, 5120, 2560)):
        x, row_e, host, _, _, ref = _case(n=n, d=d, inter=inter, E=2, seed=5)
        rms = np.sqrt(np.mean(ref ** 2))
        err = np.abs(_model_batched(x, row_e, host, 2) - ref) / rms
        rel_rms, rel_max = float(np.sqrt(np.mean(err ** 2))), float(err.max())
        c = rel_max / (rel_rms * np.sqrt(2 * np.log(err.size)))
        assert 2.5e-3 < rel_rms < RMS_BAR["fp8"] and c <= 1.6, (d, rel_rms, rel_max, c)
        worst = max(worst, c * rel_rms * np.sqrt(2 * np.log(4e6)))
    assert 1.15 * worst <= TOL_FP8 <= 2.0 * worst, (worst, TOL_FP8)
