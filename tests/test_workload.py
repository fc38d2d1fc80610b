"""Seeded input generators: determinism, slicing, distributions, skew calibration."""
import json
import os

import numpy as np
import pytest

import workload as W


def test_slices_are_consistent(wl):
    full = W.normal_bf16(1, W.TID_GATE, 0, 10_000, 0.1)
    part = W.normal_bf16(1, W.TID_GATE, 3_001, 5_000, 0.1)
    assert np.array_equal(full[3_001:8_001], part)
    cfg = W.CONFIGS["tiny"]
    allx = W.gen_x(cfg, 3)
    assert np.array_equal(allx[10:20], W.gen_x(cfg, 3, 10, 20))
    e_all = W.gen_expert_bf16(cfg, 3, "down", 0, cfg.E)
    assert np.array_equal(e_all[5:7], W.gen_expert_bf16(cfg, 3, "down", 5, 7))


def test_seeds_and_streams_differ(wl):
    a = W.normal_bf16(1, W.TID_X, 0, 1000, 1.0)
    assert not np.array_equal(a, W.normal_bf16(2, W.TID_X, 0, 1000, 1.0))
    assert not np.array_equal(a, W.normal_bf16(1, W.TID_WR, 0, 1000, 1.0))


def test_distributions(wl):
    cfg = W.CONFIGS["decode"]
    x = W.bf16_to_f32(W.gen_x(cfg.with_tokens(64), 0)).astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    wr = W.gen_wr(cfg, 0).astype(np.float64)
    assert abs(wr.std() * np.sqrt(cfg.d) - 1.0) < 0.01
    g = W.bf16_to_f32(W.gen_expert_bf16(cfg, 0, "gate", 7, 8)).astype(np.float64)
    assert abs(g.std() * np.sqrt(cfg.d) - 1.0) < 0.01
    dn = W.bf16_to_f32(W.gen_expert_bf16(cfg, 0, "down", 7, 8)).astype(np.float64)
    assert abs(dn.std() * np.sqrt(cfg.inter) - 1.0) < 0.01
    # kurtosis of a normal is 3
    z = W.normal_f64(5, W.TID_AUX, 0, 200_000)
    assert abs(((z - z.mean()) ** 4).mean() / z.var() ** 2 - 3.0) < 0.05


def test_random_topk_distinct(wl):
    idx = W.random_topk(1, 1000, 256, 8, hot_count=16, hot_prob=0.3)
    assert idx.min() >= 0 and idx.max() < 256
    for row in idx:
        assert len(set(row.tolist())) == 8
    counts = np.bincount(idx.ravel(), minlength=256)
    assert counts[:16].mean() > 3 * counts[16:].mean()


def test_skew_beta_reproduces_target(wl, olib):
    """The stored beta gives hot experts about 4x the mean load (checked with the oracle
    on the calibration tokens and on a second, unseen token range)."""
    import oracle as O

    info = json.load(open(os.path.join(os.path.dirname(W.__file__), "skew_beta.json")))
    cfg = W.CONFIGS["skewed"]
    assert list(cfg.hot_experts) == info["hot_experts"]
    wr = W.gen_wr(cfg, 0)
    for t0 in (0, 20_000):
        x = W.gen_x(cfg, 0, t0, t0 + 1024)
        r = O.route(cfg.with_tokens(1024), x, wr)
        counts = np.bincount(r["idx"].ravel(), minlength=cfg.E)
        ratio = counts[list(cfg.hot_experts)].mean() / (1024 * cfg.top_k / cfg.E)
        assert 3.6 < ratio < 4.4, ratio


def test_fp8_quantiser_round_trip():
    """FP8 with 128 x 128 block scales: every block scale is amax/448 (fp32), and every weight,
    decoded with torch's float8 e4m3 type, is within half an e4m3 step of the bf16 original
    (3 mantissa bits: 2^-4 relative for normal codes, 2^-10 * scale below)."""
    import torch
    cfg = W.MoEConfig("q8", T=4, d=256, E=1, n_groups=1, topk_groups=1, top_k=1, inter=384, wfmt="fp8")
    w = W.gen_expert_bf16(cfg, 3, "gate", 0, 1)[0]
    codes, scales = W.quantize_fp8(w)
    wf = W.bf16_to_f32(w).astype(np.float64)
    amax = np.abs(wf).reshape(3, 128, 2, 128).max(axis=(1, 3))
    assert np.array_equal(scales, (amax / 448.0).astype(np.float32))
    s = np.repeat(np.repeat(scales.astype(np.float64), 128, 0), 128, 1)
    deq = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * s
    assert np.all(np.abs(deq - wf) <= np.maximum(np.abs(wf) * 2.0 ** -4, 2.0 ** -10 * s) * (1 + 1e-12))
    assert np.all(np.abs(deq) <= np.abs(wf).max() * (1 + 2.0 ** -4))
