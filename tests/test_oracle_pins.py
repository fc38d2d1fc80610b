"""Pins of the CPU oracle against facts fixed outside it.

Each check pins the oracle to something other than itself: the block facts the
Beam release article prints (tests/golden/beam_block.json), closed forms
(uniform scores), brute-force enumeration on tiny inputs, library routines
(numpy matmul, scipy's logistic, numpy's stable sort, torch's float8/bfloat16
conversions) on special cases. ``test_oracle_mutants`` plants plausible
mistakes in copies of the oracle and checks that these pins catch each one.
"""
import itertools
import json
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch
from scipy.special import expit

import oracle as O
import workload as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "beam_block.json")

TINY = W.CONFIGS["tiny"]


def _bf16_bits(a_f32: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits with torch's round-to-nearest-even."""
    return torch.from_numpy(np.ascontiguousarray(a_f32, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return W.bf16_to_f32(bits).astype(np.float64)


# ----------------------------------------------------------------------------------------
# checks (each takes an oracle library handle so mutants can be run through them)
# ----------------------------------------------------------------------------------------

def check_uniform_scores(L):
    """W_r = 0 gives every score sigmoid(0) = 0.5; all group scores tie at 1.0, so the
    lowest-index groups and experts win and every weight is routed_scale / top_k."""
    for (E, G, Gk, K) in [(256, 8, 4, 8), (16, 4, 2, 4), (12, 3, 2, 5)]:
        d = 64
        x = W.normal_bf16(3, W.TID_AUX, 0, 5 * d, 1.0).reshape(5, d)
        wr = np.zeros((d, E), np.float32)
        logits, scores = O.router_scores(x, wr, L)
        assert np.all(logits == 0.0) and np.all(scores == 0.5)
        r = O.select(scores, G, Gk, K, 2.5, L)
        assert np.all(r["gscores"] == 1.0)
        assert np.array_equal(r["idx"], np.tile(np.arange(K, dtype=np.int32), (5, 1)))
        assert np.all(r["w"] == 2.5 / K)
        if (E, K) == (256, 8):
            assert np.all(r["w"] == 0.3125)


def check_router_logits(L):
    """Logits equal the float32 rounding of the float64 matmul (numpy); scores equal
    scipy's logistic of those logits rounded to float32 (1-ulp slack for the
    libraries' own rounding); one-hot rows return rows of W_r exactly."""
    T, d, E = 33, 96, 16
    x = W.normal_bf16(5, W.TID_AUX, 0, T * d, 1.0).reshape(T, d)
    wr = W.normal_f32(5, W.TID_AUX + 1, 0, d * E, 1 / np.sqrt(d)).reshape(d, E)
    logits, scores = O.router_scores(x, wr, L)
    ref = (_f(x) @ wr.astype(np.float64)).astype(np.float32)
    assert np.all(np.abs(logits - ref) <= np.spacing(np.abs(ref)))
    sref = expit(logits.astype(np.float64)).astype(np.float32)
    assert np.all(np.abs(scores - sref) <= np.spacing(sref))
    onehot = np.zeros((d, d), np.float32)
    onehot[np.arange(d), np.arange(d)] = 1.0
    lo, _ = O.router_scores(_bf16_bits(onehot), wr, L)
    assert np.array_equal(lo, wr)


def _brute_select(s, G, Gk, K):
    E = s.size
    gsz = E // G
    gs = []
    for g in range(G):
        grp = s[g * gsz:(g + 1) * gsz]
        if gsz == 1:
            gs.append(np.float32(grp[0]))
        else:
            gs.append(max(np.float32(grp[i]) + np.float32(grp[j]) for i, j in itertools.combinations(range(gsz), 2)))
    best_groups = max(itertools.combinations(range(G), Gk), key=lambda c: sum(float(gs[g]) for g in c))
    cand = [e for e in range(E) if e // gsz in best_groups]
    best = max(itertools.combinations(cand, K), key=lambda c: sum(float(s[e]) for e in c))
    return set(best), np.array(gs, np.float32)


def check_select_bruteforce(L):
    """Group scores, kept groups and chosen experts equal the argmax over all pairs and
    all subsets (random scores, so no ties); weights are 2.5 * s / sum(s)."""
    for (E, G, Gk, K, seed) in [(16, 4, 2, 4, 1), (12, 3, 2, 3, 2), (16, 8, 3, 4, 3), (10, 5, 4, 6, 4), (16, 4, 2, 4, 5)]:
        T = 40
        s = W.uniform_f64(seed, W.TID_AUX, 0, T * E).astype(np.float32).reshape(T, E)
        r = O.select(s, G, Gk, K, 2.5, L)
        for t in range(T):
            chosen, gs = _brute_select(s[t], G, Gk, K)
            assert set(r["idx"][t].tolist()) == chosen, (E, G, Gk, K, t)
            assert np.array_equal(r["gscores"][t], gs)
            # slots are in descending score order
            sv = s[t][r["idx"][t]]
            assert np.all(np.diff(sv.astype(np.float64)) <= 0)
            ws = 2.5 * sv.astype(np.float64) / sv.astype(np.float64).sum()
            assert np.allclose(r["w"][t], ws, rtol=1e-15, atol=0)


def check_select_bias(L):
    """Selection bias (the balancing bias of DeepSeek-V3's router, which the article's router
    follows): the choice is the brute-force group-limited top-k of s + b (float32 add), slots in
    descending s + b; the weights are 2.5 * s / sum(s) with the unbiased scores; a zero bias
    changes nothing; a bias far above the score range puts that expert in every choice."""
    for (E, G, Gk, K, seed) in [(16, 4, 2, 4, 11), (12, 3, 2, 3, 12), (16, 8, 3, 4, 13)]:
        T = 40
        s = W.uniform_f64(seed, W.TID_AUX, 0, T * E).astype(np.float32).reshape(T, E)
        b = (0.3 * (W.uniform_f64(seed, W.TID_AUX + 1, 0, E) - 0.5)).astype(np.float32)
        r = O.select(s, G, Gk, K, 2.5, L, bias=b)
        for t in range(T):
            sel = (s[t] + b).astype(np.float32)
            chosen, gs = _brute_select(sel, G, Gk, K)
            assert set(r["idx"][t].tolist()) == chosen, (E, G, Gk, K, t)
            assert np.array_equal(r["gscores"][t], gs)
            assert np.all(np.diff(sel[r["idx"][t]].astype(np.float64)) <= 0)
            sv = s[t][r["idx"][t]].astype(np.float64)
            assert np.allclose(r["w"][t], 2.5 * sv / sv.sum(), rtol=1e-15, atol=0)
        r0 = O.select(s, G, Gk, K, 2.5, L, bias=np.zeros(E, np.float32))
        rn = O.select(s, G, Gk, K, 2.5, L)
        assert np.array_equal(r0["idx"], rn["idx"]) and np.array_equal(r0["w"], rn["w"])
    E, G, Gk, K = 16, 4, 2, 4
    s = W.uniform_f64(14, W.TID_AUX, 0, 30 * E).astype(np.float32).reshape(30, E)
    b = np.zeros(E, np.float32)
    b[5] = 4.0
    r = O.select(s, G, Gk, K, 2.5, L, bias=b)
    assert np.all(r["idx"][:, 0] == 5)
    s64 = s.astype(np.float64)
    assert np.allclose(r["w"][:, 0], 2.5 * s64[:, 5] / np.take_along_axis(s64, r["idx"].astype(np.int64), 1).sum(1),
                       rtol=1e-12, atol=0)


def check_select_invariants(L):
    """Chosen experts are distinct, lie in kept groups; weights are >= 0 and sum to 2.5;
    margins are non-negative."""
    E, G, Gk, K = 256, 8, 4, 8
    T = 300
    logits = W.normal_f32(9, W.TID_AUX, 0, T * E, 1.0).reshape(T, E)
    s = expit(logits.astype(np.float64)).astype(np.float32)
    r = O.select(s, G, Gk, K, 2.5, L)
    idx = r["idx"]
    for t in range(T):
        assert len(set(idx[t].tolist())) == K
        kept = np.argsort(-r["gscores"][t].astype(np.float64), kind="stable")[:Gk]
        assert set((idx[t] // (E // G)).tolist()) <= set(kept.tolist())
    assert np.all(r["w"] >= 0)
    assert np.all(np.abs(r["w"].sum(1) - 2.5) <= 1e-6)
    assert np.all(r["margin_group"] >= 0) and np.all(r["margin_expert"] >= 0)


def _dense_swiglu_ref(xb, gate, up, down):
    """Dense SwiGLU MLP with library matmuls: h = silu(x Wg) * (x Wu) formed in float32 and
    rounded to bf16 (torch), y = h Wd in float64."""
    x = _f(xb)
    g = (x @ _f(gate).T).astype(np.float32)
    u = (x @ _f(up).T).astype(np.float32)
    silu = (g.astype(np.float64) * expit(g.astype(np.float64))).astype(np.float32)
    h = _bf16_bits(silu * u)
    return _f(h) @ _f(down).T, h


def check_single_expert_dense(L):
    """E=1, one group, top-1: the block is 2.5 * SwiGLU(x), the dense MLP the Beam
    article uses in its first three layers."""
    d, I, T = 128, 64, 24
    x = W.normal_bf16(11, W.TID_AUX, 0, T * d, 1.0).reshape(T, d)
    gate = W.normal_bf16(11, W.TID_AUX + 1, 0, I * d, 1 / np.sqrt(d)).reshape(1, I, d)
    up = W.normal_bf16(11, W.TID_AUX + 2, 0, I * d, 1 / np.sqrt(d)).reshape(1, I, d)
    down = W.normal_bf16(11, W.TID_AUX + 3, 0, d * I, 1 / np.sqrt(I)).reshape(1, d, I)
    wr = W.normal_f32(11, W.TID_AUX + 4, 0, d, 1 / np.sqrt(d)).reshape(d, 1)
    cfg = W.MoEConfig("one", T=T, d=d, E=1, n_groups=1, topk_groups=1, top_k=1, inter=I)
    r = O.route(cfg, x, wr, L)
    assert np.all(r["idx"] == 0) and np.all(r["w"] == 2.5)
    weights = {"gate": gate, "up": up, "down": down}
    out = O.forward_tokens(cfg, x, r["idx"], r["w"], np.arange(T), weights, L)
    yref, href = _dense_swiglu_ref(x, gate[0], up[0], down[0])
    ref = 2.5 * yref
    rms = np.sqrt((ref ** 2).mean())
    assert np.max(np.abs(out - ref)) <= 1e-3 * rms
    y, h = O.ffn_rows(np.zeros(T, np.int32), x, weights, d, I, want_h=True, L=L)
    assert np.mean(h != href) < 2e-3  # rare 1-ulp flips from summation order only
    assert np.max(np.abs(_f(h) - _f(href))) <= np.max(np.abs(_f(href))) * 2 ** -7


def check_identical_experts(L):
    """All experts equal: for any routing the weights sum to 2.5, so the block is
    2.5 * SwiGLU(x) whatever the router picks."""
    cfg = TINY
    T, d, I = cfg.T, cfg.d, cfg.inter
    x = W.gen_x(cfg, 4)
    wr = W.gen_wr(cfg, 4)
    g1 = W.gen_expert_bf16(cfg, 4, "gate", 0, 1)
    u1 = W.gen_expert_bf16(cfg, 4, "up", 0, 1)
    d1 = W.gen_expert_bf16(cfg, 4, "down", 0, 1)
    weights = {k: np.ascontiguousarray(np.repeat(v, cfg.E, axis=0)) for k, v in (("gate", g1), ("up", u1), ("down", d1))}
    r = O.route(cfg, x, wr, L)
    assert len(np.unique(r["idx"])) > 4
    out = O.forward_tokens(cfg, x, r["idx"], r["w"], np.arange(T), weights, L)
    yref, _ = _dense_swiglu_ref(x, g1[0], u1[0], d1[0])
    ref = 2.5 * yref
    assert np.max(np.abs(out - ref)) <= 1e-3 * np.sqrt((ref ** 2).mean())


def check_permute(L):
    """Rows grouped by expert, tokens ascending inside an expert: numpy's stable sort of
    the flattened (token, slot) list by expert id gives the same row order."""
    for (T, E, K, hot) in [(64, 16, 4, 0), (257, 256, 8, 0), (500, 32, 8, 4), (1, 8, 2, 0)]:
        idx = W.random_topk(7, T, E, K, hot_count=hot, hot_prob=0.5 if hot else 0.0)
        counts, offsets, row_token, inv_row = O.permute(idx, E, L)
        flat = idx.reshape(-1)
        order = np.argsort(flat, kind="stable")
        assert np.array_equal(counts, np.bincount(flat, minlength=E))
        assert np.array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        assert np.array_equal(row_token, order // K)
        inv = np.empty_like(order)
        inv[order] = np.arange(order.size)
        assert np.array_equal(inv_row, inv)


def check_combine(L):
    """out[t] = sum_k w[t,k] * y[inv_row[t,k]] against numpy's einsum."""
    T, K, d, E = 50, 4, 48, 16
    idx = W.random_topk(8, T, E, K)
    _, _, _, inv_row = O.permute(idx, E, L)
    y = W.normal_f32(8, W.TID_AUX, 0, T * K * d, 1.0).reshape(T * K, d)
    w = W.uniform_f64(8, W.TID_AUX + 1, 0, T * K).reshape(T, K)
    out = O.combine(y, inv_row, w, L)
    ref = np.einsum("tk,tkd->td", w, y.astype(np.float64)[inv_row.reshape(T, K)])
    assert np.allclose(out, ref, rtol=1e-13, atol=1e-13)


def check_forward_matches_stages(L):
    """The block forward equals permute -> per-row expert MLP -> combine."""
    cfg = TINY
    inp = W.make_host_inputs(cfg, 2)
    r = O.route(cfg, inp["x"], inp["w_r"], L)
    out = O.forward_tokens(cfg, inp["x"], r["idx"], r["w"], np.arange(cfg.T), inp, L)
    counts, offsets, row_token, inv_row = O.permute(r["idx"], cfg.E, L)
    row_expert = np.repeat(np.arange(cfg.E, dtype=np.int32), counts)
    y = O.ffn_rows(row_expert, inp["x"][row_token], inp, cfg.d, cfg.inter, L=L)
    ref = np.einsum("tk,tkd->td", r["w"], y[inv_row.reshape(cfg.T, cfg.top_k)])
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


E2M1_POINTS = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def check_nvfp4_decode(L):
    """e2m1 codes decode to the format's code points (sign in bit 3); e4m3 codes decode
    exactly as torch.float8_e4m3fn does, NaN included."""
    for c in range(16):
        v = O.e2m1_value(c, L)
        mag = E2M1_POINTS[c & 7]
        assert v == (-mag if c & 8 else mag), c
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([O.e4m3_value(c, L) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def _dequant_ref(packed, scales, ts):
    """Dequantised weights via torch's float8_e4m3fn and the e2m1 code-point list."""
    lo = packed & 15
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(packed.shape[0], -1)
    pts = np.array(E2M1_POINTS, np.float64)
    q = np.where(codes & 8, -1.0, 1.0) * pts[codes & 7]
    sb = torch.from_numpy(np.ascontiguousarray(scales)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return q * np.repeat(sb, 16, axis=1) * float(ts)


def check_nvfp4_ffn(L):
    """The NVFP4 expert MLP equals a dense float64 MLP on the dequantised weights."""
    cfg = W.MoEConfig("q", T=16, d=128, E=2, n_groups=1, topk_groups=1, top_k=1, inter=64, wfmt="nvfp4")
    x = W.gen_x(cfg, 6)
    q = {}
    deq = {}
    for which in ("gate", "up", "down"):
        p, s, t = W.gen_expert_nvfp4(cfg, 6, which, 0, 2)
        q[which], q[which + "_sf"], q[which + "_ts"] = p, s, t
        deq[which] = np.stack([_dequant_ref(p[e], s[e], t[e]) for e in range(2)])
    rows = np.array([0, 1] * 8, np.int32)
    y, h = O.ffn_rows(rows, x, q, cfg.d, cfg.inter, "nvfp4", want_h=True, L=L)
    xf = _f(x)
    for r in range(16):
        e = rows[r]
        g = (xf[r] @ deq["gate"][e].T).astype(np.float32)
        u = (xf[r] @ deq["up"][e].T).astype(np.float32)
        silu = (g.astype(np.float64) * expit(g.astype(np.float64))).astype(np.float32)
        hr = _f(_bf16_bits(silu * u))
        yr = hr @ deq["down"][e].T
        assert np.max(np.abs(y[r] - yr)) <= 1e-3 * np.sqrt((yr ** 2).mean())


def check_fp8_ffn(L):
    """The FP8 expert MLP equals a dense float64 MLP on weights dequantised with torch's own
    float8 e4m3 decoding times each 128 x 128 block's scale. Each block of the seeded weights is
    scaled by its own factor first, so every block scale differs and a wrong block index shows."""
    cfg = W.MoEConfig("q8", T=12, d=256, E=2, n_groups=1, topk_groups=1, top_k=1, inter=256, wfmt="fp8")
    x = W.gen_x(cfg, 7)
    q, deq = {}, {}
    factor = np.array([[1.0, 2.0], [3.0, 5.0]], np.float32)
    for which in ("gate", "up", "down"):
        N, K = W.weight_shape(cfg, which)
        codes = np.empty((2, N, K), np.uint8)
        scales = np.empty((2, N // 128, K // 128), np.float32)
        for e in range(2):
            w = _f(W.gen_expert_bf16(cfg, 7, which, e, e + 1)[0]).astype(np.float32)
            w *= np.repeat(np.repeat(factor * (e + 1), 128, 0), 128, 1)
            codes[e], scales[e] = W.quantize_fp8(_bf16_bits(w))
        assert np.unique(scales).size == scales.size
        q[which], q[which + "_sf"] = codes, scales
        vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        deq[which] = vals * np.repeat(np.repeat(scales.astype(np.float64), 128, 1), 128, 2)
    rows = np.array([0, 1] * 6, np.int32)
    y, h = O.ffn_rows(rows, x, q, cfg.d, cfg.inter, "fp8", want_h=True, L=L)
    xf = _f(x)
    for r in range(12):
        e = rows[r]
        g = (xf[r] @ deq["gate"][e].T).astype(np.float32)
        u = (xf[r] @ deq["up"][e].T).astype(np.float32)
        silu = (g.astype(np.float64) * expit(g.astype(np.float64))).astype(np.float32)
        hr = _f(_bf16_bits(silu * u))
        yr = hr @ deq["down"][e].T
        assert np.max(np.abs(y[r] - yr)) <= 1e-3 * np.sqrt((yr ** 2).mean())


def _bf16_const(v, n):
    return _bf16_bits(np.full(n, v, np.float32))


def check_residual_step1_normalises(L):
    """At step k = 1 nothing of the old stream is kept and the sublayer output is RMS-normalised:
    each row's mean square is gamma^2 * ms / (ms + eps), which is gamma^2 for eps = 0, whatever
    the output's own scale."""
    T, d = 12, 96
    out = W.normal_f32(31, W.TID_AUX, 0, T * d, 3.0).reshape(T, d).astype(np.float64)
    h_old = W.normal_bf16(31, W.TID_AUX + 1, 0, T * d, 1.0).reshape(T, d)
    for g, eps in ((1.0, 0.0), (2.0, 0.0), (1.0, 1e-2)):
        hn = O.residual_update(out, h_old, _bf16_const(g, d), eps, 1, L)
        ms = (out ** 2).mean(1)
        assert np.allclose((hn ** 2).mean(1), g * g * ms / (ms + eps), rtol=1e-12, atol=0)
    hn1 = O.residual_update(out, h_old, _bf16_const(1.0, d), 0.0, 1, L)
    hn7 = O.residual_update(7.0 * out, h_old, _bf16_const(1.0, d), 0.0, 1, L)
    assert np.allclose(hn1, hn7, rtol=1e-12, atol=1e-15)


def check_residual_equal_weights(L):
    """The article's claim: counting the input embedding as step 1 and adding 104 sublayer
    outputs, every output and the embedding carry the same weight in the final stream. With
    orthogonal unit-RMS vectors v_1..v_105 (scaled one-hot rows), the final stream's component
    along each is 1/sqrt(105) (the stream is kept in bf16 between steps: rounding drifts the
    coefficients by up to ~3 %; a wrong weight rule is off by tens of percent)."""
    N, d = 105, 128
    v = np.sqrt(d) * np.eye(d)[:N]               # v_j: unit RMS, mutually orthogonal
    h = _bf16_bits(v[0].astype(np.float32))[None]  # step 1: the embedding
    for k in range(2, N + 1):
        hn = O.residual_update(v[k - 1][None], h, _bf16_const(1.0, d), 0.0, k, L)
        h = _bf16_bits(hn.astype(np.float32))
    coef = _f(h[0])[:N] / np.sqrt(d)
    assert np.allclose(coef, 1 / np.sqrt(N), rtol=4e-2, atol=0), (coef.min(), coef.max())
    assert np.all(_f(h[0])[N:] == 0)


def check_residual_constant_scale(L):
    """The weights' squares sum to one, so a unit-RMS stream plus an independent unit-RMS
    output stays at unit RMS on average, at every step."""
    T, d = 400, 256
    for k in (2, 5, 52):
        h_old = W.normal_bf16(40 + k, W.TID_AUX, 0, T * d, 1.0).reshape(T, d)
        out = W.normal_f32(40 + k, W.TID_AUX + 1, 0, T * d, 0.3).reshape(T, d).astype(np.float64)
        hn = O.residual_update(out, h_old, _bf16_const(1.0, d), 0.0, k, L)
        assert abs((hn ** 2).mean() - 1.0) < 0.02, (k, (hn ** 2).mean())


def check_pre_norm_closed_forms(L):
    """RMSNorm before the sublayer, in closed forms that hold exactly for bf16 inputs with
    eps = 0: a constant row maps to sign * gain; a one-hot row a * e_j maps to
    sign(a) * sqrt(d) * gain_j at j and 0 elsewhere (sqrt(64) = 8); scaling a row by a power
    of two changes nothing; a positive eps shrinks the mean square to ms / (ms + eps)."""
    d = 64
    gain = _bf16_bits(np.linspace(0.5, 1.5, d).astype(np.float32))
    g = _f(gain)
    for c in (3.0, -0.375, 1e-3):
        x = O.pre_norm(_bf16_const(c, d)[None], gain, 0.0, L)
        assert np.array_equal(_f(x[0]), np.sign(c) * g)
    for j, a in ((0, 2.5), (17, -0.75), (63, 40.0)):
        h = np.zeros(d, np.float32)
        h[j] = a
        x = _f(O.pre_norm(_bf16_bits(h)[None], gain, 0.0, L)[0])
        want = np.zeros(d)
        want[j] = _f(_bf16_bits(np.array([np.sign(a) * 8.0 * g[j]], np.float32)))[0]
        assert np.array_equal(x, want), (j, x[j], want[j])
    h = W.normal_bf16(51, W.TID_AUX, 0, 16 * d, 1.0).reshape(16, d)
    x1 = O.pre_norm(h, gain, 0.0, L)
    x8 = O.pre_norm(_bf16_bits(_f(h) * 8.0), gain, 0.0, L)
    assert np.array_equal(x1, x8)
    ones = _bf16_const(1.0, d)
    ms = (_f(h).astype(np.float64) ** 2).mean(1)
    for eps in (0.0, 0.5):
        xr = _f(O.pre_norm(h, ones, eps, L)).astype(np.float64)
        assert np.allclose((xr ** 2).mean(1), ms / (ms + eps), rtol=5e-3, atol=0)


CHECKS = [check_uniform_scores, check_router_logits, check_select_bruteforce, check_select_bias,
          check_select_invariants,
          check_single_expert_dense, check_identical_experts, check_permute, check_combine,
          check_forward_matches_stages, check_nvfp4_decode, check_nvfp4_ffn, check_fp8_ffn,
          check_residual_step1_normalises,
          check_residual_equal_weights, check_residual_constant_scale, check_pre_norm_closed_forms]


@pytest.mark.parametrize("check", CHECKS, ids=lambda c: c.__name__)
def test_oracle_pin(check, olib):
    check(olib)


def test_printed_block_facts():
    """The workload shapes are the ones the article prints, and its parameter
    arithmetic closes: 3*5120*2560 ~ 39M per expert, 49*256 experts ~ 98.4% of 501B,
    and the routed parameters plus the replicated rest fit the 23B active figure."""
    g = json.load(open(GOLDEN))
    for name in ("decode", "prefill", "skewed", "nvfp4", "fp8"):
        c = W.CONFIGS[name]
        assert (c.d, c.E, c.n_groups, c.E // c.n_groups, c.topk_groups, c.top_k, c.inter, c.routed_scale) == (
            g["hidden"], g["experts"], g["groups"], g["group_size"], g["groups_kept"], g["routed_per_token"],
            g["intermediate"], g["routed_scale"])
    per_expert = 3 * g["hidden"] * g["intermediate"]
    assert abs(per_expert - g["expert_params_approx"]) / g["expert_params_approx"] < 0.01
    expert_total = g["moe_layers"] * g["experts"] * per_expert
    assert abs(expert_total / g["total_params"] - g["expert_share_of_params"]) < 0.001
    active = g["moe_layers"] * g["routed_per_token"] * per_expert + (g["total_params"] - expert_total)
    assert abs(active - g["active_params"]) / g["active_params"] < 0.03
    assert g["layers"] == g["dense_layers"] + g["moe_layers"]


# ----------------------------------------------------------------------------------------
# planted mistakes: every mutant of the oracle must fail at least one pin
# ----------------------------------------------------------------------------------------

MUTANTS = {
    "sigmoid_sign": ("1.0 / (1.0 + exp(-(double)l))", "1.0 / (1.0 + exp((double)l))"),
    "group_top1_only": ("(sel[b1] + sel[b2])", "(sel[b1] + sel[b1])"),
    "group_max_not_sum": ("(sel[b1] + sel[b2])", "(sel[b1])"),
    "silu_is_sigmoid": ("(double)gf / (1.0 + exp(-(double)gf))", "1.0 / (1.0 + exp(-(double)gf))"),
    "gate_up_swapped": ("g += xbuf[j] * wmat_at(gate", "g += xbuf[j] * wmat_at(up"),
    "no_normalisation": ("w[k] = scale * (double)s[idx[k]] / sum;", "w[k] = scale * (double)s[idx[k]];"),
    "no_scale": ("w[k] = scale * (double)s[idx[k]] / sum;", "w[k] = (double)s[idx[k]] / sum;"),
    "tie_to_higher_index": ("if (kept[e / gsz] && !taken[e] && (best < 0 || sel[e] > sel[best])) best = e;",
                            "if (kept[e / gsz] && !taken[e] && (best < 0 || sel[e] >= sel[best])) best = e;"),
    "bias_ignored": ("sel[e] = bias ? s[e] + bias[e] : s[e];", "sel[e] = s[e];"),
    "bias_in_weights": ("w[k] = scale * (double)s[idx[k]] / sum;", "w[k] = scale * (double)sel[idx[k]] / sum;"),
    "bias_in_weight_sum": ("sum += (double)s[best];", "sum += (double)sel[best];"),
    "residual_keep_linear": ("sqrt((double)(k - 1) / (double)k)", "((double)(k - 1) / (double)k)"),
    "residual_keep_on_output": ("keep * bf16_value(h_old", "add * bf16_value(h_old"),
    "rms_sum_not_mean": ("sqrt(ss / d + eps)", "sqrt(ss + eps)"),
    "post_norm_no_gain": (" * bf16_value(gamma[c]))", ")"),
    "fp8_block_transposed": ("bs[((int64_t)e * nbn + n / 128) * nbk + k / 128]",
                             "bs[((int64_t)e * nbn + k / 128) * nbk + n / 128]"),
    "pre_norm_no_gain": ("bf16_round((float)(bf16_value(row[c]) / r * bf16_value(gamma[c])))",
                         "bf16_round((float)(bf16_value(row[c]) / r))"),
    "pre_norm_abs_not_square": ("ss += bf16_value(row[c]) * bf16_value(row[c]);",
                                "ss += fabs(bf16_value(row[c]));"),
    "pre_norm_eps_outside_sqrt": ("const double r = sqrt(ss / d + eps);\n    for (int c = 0; c < d; ++c)\n      x[",
                                  "const double r = sqrt(ss / d) + eps;\n    for (int c = 0; c < d; ++c)\n      x["),
    "pre_norm_sum_not_mean": ("const double r = sqrt(ss / d + eps);\n    for (int c = 0; c < d; ++c)\n      x[",
                              "const double r = sqrt(ss + eps);\n    for (int c = 0; c < d; ++c)\n      x["),
    "fp8_scale_dropped": ("(double)bs[((int64_t)e * nbn + n / 128) * nbk + k / 128]", "1.0"),
    "fp8_scales_of_expert_0": ("bs[((int64_t)e * nbn + n / 128)", "bs[((int64_t)0 * nbn + n / 128)"),
    "no_group_limit": ("if (kept[e / gsz] && !taken[e] && (best < 0", "if (!taken[e] && (best < 0"),
    "h_not_rounded": ("hbuf[i] = bf16_value(hb);", "hbuf[i] = (double)(silu * uf);"),
    "down_transposed": ("acc += hbuf[i] * wmat_at(down, e, n, i);", "acc += hbuf[i] * wmat_at(down, e, i % d, n % I);"),
    "e4m3_bias": ("ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    "nibble_order": ("(k & 1) ? (byte >> 4) : (byte & 15)", "(k & 1) ? (byte & 15) : (byte >> 4)"),
    "permute_token_desc": ("for (int t = 0; t < T; ++t)\n      for (int k = 0; k < K; ++k)\n        if (idx",
                           "for (int t = T - 1; t >= 0; --t)\n      for (int k = 0; k < K; ++k)\n        if (idx"),
    "combine_slot_weight": ("acc += w[(int64_t)t * K + k] * (double)y", "acc += w[(int64_t)t * K] * (double)y"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_oracle_mutants(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(O._SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    msrc = tmp_path / "oracle_mut.c"
    msrc.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    O.build(force=True, src=str(msrc), out=str(so))
    L = O.load(str(so))
    failed = []
    for check in CHECKS:
        try:
            check(L)
        except (AssertionError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
