"""Where the FP8 typical-error bar comes from (CPU only).

The expert GEMMs take bf16 operands, so FP8 weights are dequantised on chip as
bf16(fp32(e4m3 * block scale)); the oracle keeps the exact product. This test
repeats exactly those roundings in numpy (bf16 weights, FP32 SwiGLU, bf16 h,
bf16 y) and measures their error against the oracle: it must sit below the
bar the GPU tests use, and removing the weight rounding must bring it back
below the bf16 bar. A bar that merely hid a kernel bug would not be explained
by this model.
"""
import numpy as np
import pytest
import torch

import oracle as O
import workload as W
from support import RMS_BAR



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
        y[i] = _bf16((deq["down"][e] @ h).astype(np.float32))
    return y


def test_fp8_bar_is_the_weight_rounding():
    d, inter, E, n = 256, 384, 2, 160
    cfg = W.MoEConfig("fp8m", T=n, d=d, E=E, n_groups=1, topk_groups=1, top_k=1, inter=inter, wfmt="fp8")
    host = {}
    for which in ("gate", "up", "down"):
        host[which], host[which + "_sf"] = W.gen_expert_fp8(cfg, 3, which, 0, E)
    x = W.normal_bf16(3, W.TID_X, 0, n * d, 1.0).reshape(n, d)
    row_e = np.arange(n, dtype=np.int32) % E
    ref = O.ffn_rows(row_e, x, host, d, inter, "fp8")
    rms = np.sqrt(np.mean(ref ** 2))
    rel = {rw: np.sqrt(np.mean((_model(x, row_e, host, d, inter, rw) - ref) ** 2)) / rms for rw in (True, False)}
    assert 2.5e-3 < rel[True] < RMS_BAR["fp8"], rel
    assert rel[False] < RMS_BAR["bf16"], rel
