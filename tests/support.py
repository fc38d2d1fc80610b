"""Shared helpers of the GPU tests: device upload of seeded inputs and the
routing comparison with the near-tie rule.

Routing must match the oracle exactly (expert sets, slot order, per-expert
counts) except for tokens whose decision margin is within 1e-6 (the 4th vs 5th
group score, or the 8th vs 9th candidate score): those are excluded from the
exact check, the GPU's choice is checked to be one of the tied optima, and
their reference output is recomputed with the GPU's choice.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
import workload as W
import sparse_moe_layer_14_b300 as bm

TIE_EPS = 1e-6
TOL_BF16 = 2e-2   # max |err| <= TOL * RMS(oracle output), bf16 weights
TOL_NVFP4 = 5e-2  # ... NVFP4 weights
# FP8 weights: the max bar follows from the error of the on-chip weight rounding bf16(e4m3 x
# scale), which a CPU model of exactly these roundings reproduces (test_fp8_error_model.py, which
# derives this bar): a relative RMS of ~3.5e-3 with tails up to ~1.45 x Gaussian at small
# reduction lengths, so over the largest comparison a test makes (~4e6 elements) the max is
# expected near 2.8e-2; the bar keeps a fifth above that.
TOL_FP8 = 3.5e-2
TOL = {"bf16": TOL_BF16, "nvfp4": TOL_NVFP4, "fp8": TOL_FP8}
# Typical (RMS) error bar of the expert FFN relative to the RMS output. bf16 and
# NVFP4 weights reach the tensor cores exactly, leaving fp32 summation order and
# 1-ulp flips of the bf16 h and output (~1.1e-3 to 1.7e-3). FP8 weights are
# dequantised on chip to bf16 (e4m3 x block scale rounded to fp32, then to bf16, ulp 2^-7; the
# oracle keeps the exact product): a relative error of RMS ~2^-8 / sqrt(3) /
# sqrt(2) ~ 1.6e-3 per weight, reaching y through gate, up and down. A CPU model
# of exactly these roundings gives 3.9e-3 on the ragged-tile case, as the kernel
# does; the bar leaves room for seeds.
RMS_BAR = {"bf16": 2e-3, "nvfp4": 2e-3, "fp8": 5e-3}


# One line per parity check (routing exclusions, error ratios), printed at the end of the test
# session by conftest.py so that a quiet run still shows them.
REPORT: list[str] = []


def report(label: str, text: str):
    REPORT.append(f"{label}: {text}")


def plan_n_max(T: int, E: int, top_k: int, decoded: bool) -> int:
    """Token-tile size the library's expert GEMM uses for a batch (the rule of its work-item
    plan): a quarter above the mean rows per expert, rounded up to 16, clamped to [64, 256]
    (192 with NVFP4 or FP8 weights) and to the batch rounded up to 16."""
    R = T * top_k
    mean = -(-R // max(E, 1))
    n = (mean + mean // 4 + 15) // 16 * 16
    n = max(64, min(192 if decoded else 256, n))
    return min(n, (max(T, 1) + 15) // 16 * 16)


def work_item_rows(counts, n_max: int, rng):
    """Permuted rows that put at least one checked row in every work item of the expert GEMMs.
    A work item is (expert, weight tile, token tile); comparing a whole output row covers every
    weight tile of its token tile, so it is enough to pick rows per token tile. Tiles are cut as
    the library's schedule cuts them: ceil(n / n_max) tiles of near-equal size (a multiple of
    16). Per tile: a row of its first 16-token chunk and, when the tile has more, one of its
    second chunk (the epilogue's two warpgroups take alternate 16-token chunks). Returns
    (rows, number of token tiles)."""
    rows = []
    tiles = 0
    off = 0
    for n in (int(c) for c in counts):
        if n > 0:
            ntiles = -(-n // n_max)
            tsz = min(n_max, (-(-n // ntiles) + 15) // 16 * 16)
            for j in range(-(-n // tsz)):
                tiles += 1
                a, b = off + j * tsz, off + min(n, (j + 1) * tsz)
                rows.append(a + int(rng.integers(0, min(16, b - a))))
                if b - a > 16:
                    rows.append(a + 16 + int(rng.integers(0, min(16, b - a - 16))))
        off += n
    return np.array(sorted(set(rows)), np.int64), tiles


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    """Host numpy -> device tensor; uint16 bf16 bit patterns become torch.bfloat16."""
    t = torch.from_numpy(np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """Device bf16 tensor -> uint16 bit patterns on the host."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return W.bf16_to_f32(bits).astype(np.float64)


class DeviceWeights:
    """Seeded expert weights generated one expert at a time straight into device
    tensors; optional host copies for the oracle."""

    def __init__(self, cfg, seed=0, keep_host=True, device="cuda"):
        self.cfg = cfg
        self.host = {}
        E = cfg.E
        if cfg.wfmt == "bf16":
            tens = {}
            for which in ("gate", "up", "down"):
                N, K = W.weight_shape(cfg, which)
                t = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
                h = np.empty((E, N, K), np.uint16) if keep_host else None
                step = max(1, min(E, (1 << 28) // (N * K)))
                for e0 in range(0, E, step):
                    e1 = min(E, e0 + step)
                    chunk = W.gen_expert_bf16(cfg, seed, which, e0, e1)
                    t[e0:e1].copy_(torch.from_numpy(chunk).view(torch.int16).view(torch.bfloat16))
                    if keep_host:
                        h[e0:e1] = chunk
                tens[which] = t
                if keep_host:
                    self.host[which] = h
            self.dev = bm.ExpertWeights(tens["gate"], tens["up"], tens["down"])
        elif cfg.wfmt == "fp8":
            tens = {}
            for which in ("gate", "up", "down"):
                codes, scales = W.gen_expert_fp8(cfg, seed, which, 0, E)
                tens[which], tens[which + "_sf"] = dev(codes), dev(scales)
                if keep_host:
                    self.host[which], self.host[which + "_sf"] = codes, scales
            self.dev = bm.ExpertWeights(**tens)
        else:
            tens = {}
            for which in ("gate", "up", "down"):
                p, s, ts = W.gen_expert_nvfp4(cfg, seed, which, 0, E)
                tens[which], tens[which + "_sf"], tens[which + "_ts"] = dev(p), dev(s), dev(ts)
                if keep_host:
                    self.host[which], self.host[which + "_sf"], self.host[which + "_ts"] = p, s, ts
            self.dev = bm.ExpertWeights(**tens)


def compare_routing(cfg, gpu_idx: np.ndarray, gpu_w: np.ndarray, orc: dict, all_tokens=True, bias=None,
                    label=None):
    """Check GPU routing against the oracle; returns (excluded token list, ref_idx, ref_w)
    where ref_* is the routing to use for the reference output. With a selection bias
    [E], slot order and tie validity are judged on s + bias (float32), weights on s.
    The excluded near-ties are logged (count, first tokens and their margins)."""
    T, K = gpu_idx.shape
    G, Gk = cfg.n_groups, cfg.topk_groups
    gsz = cfg.E // G
    s = orc["scores"].astype(np.float64)
    sel = s if bias is None else (orc["scores"] + np.asarray(bias, np.float32)).astype(np.float32).astype(np.float64)
    near = (orc["margin_group"] < TIE_EPS) | (orc["margin_expert"] < TIE_EPS)
    excluded = np.nonzero(near)[0]
    shown = ", ".join(f"t{t} (group {orc['margin_group'][t]:.2e}, expert {orc['margin_expert'][t]:.2e})"
                      for t in excluded[:4])
    report(label or cfg.name, f"routing T={T}: {excluded.size} near-tie tokens excluded"
           + (f" [{shown}{', ...' if excluded.size > 4 else ''}]" if excluded.size else "")
           + f"; {T - excluded.size} decided tokens compared")
    ok = ~near
    # exact sets and slot order on decided tokens
    gs_sorted = np.sort(gpu_idx[ok], axis=1)
    os_sorted = np.sort(orc["idx"][ok], axis=1)
    bad = np.nonzero(np.any(gs_sorted != os_sorted, axis=1))[0]
    assert bad.size == 0, f"routing differs on {bad.size} decided tokens, e.g. {np.nonzero(ok)[0][bad[:5]]}"
    sv = np.take_along_axis(sel, gpu_idx.astype(np.int64), axis=1)
    assert np.all(np.diff(sv[ok], axis=1) <= TIE_EPS), "slots not in descending score order"
    # per-expert counts over decided tokens (bit-exact)
    cg = np.bincount(gpu_idx[ok].ravel(), minlength=cfg.E)
    co = np.bincount(orc["idx"][ok].ravel(), minlength=cfg.E)
    assert np.array_equal(cg, co)
    # weights: same expert -> same weight up to fp32 rounding
    order_g = np.argsort(gpu_idx[ok], axis=1)
    order_o = np.argsort(orc["idx"][ok], axis=1)
    wg = np.take_along_axis(gpu_w[ok].astype(np.float64), order_g, axis=1)
    wo = np.take_along_axis(orc["w"][ok], order_o, axis=1)
    assert np.max(np.abs(wg - wo), initial=0.0) <= 2e-6 * cfg.routed_scale
    assert np.all(np.abs(gpu_w.astype(np.float64).sum(1) - cfg.routed_scale) <= 1e-5 * cfg.routed_scale)
    ref_idx = orc["idx"].copy()
    ref_w = orc["w"].copy()
    for t in excluded:
        chosen = gpu_idx[t]
        assert len(set(chosen.tolist())) == K
        assert any(_valid_under_ties(sel[t], orc["gscores"][t].astype(np.float64), chosen, gsz, Gk, K, kept)
                   for kept in _tied_kept_sets(orc["gscores"][t].astype(np.float64), Gk)), \
            f"token {t}: GPU choice is not one of the tied optima"
        ref_idx[t] = chosen
        ref_w[t] = cfg.routed_scale * s[t, chosen] / s[t, chosen].sum()
    return excluded, ref_idx, ref_w


def _tied_kept_sets(gs, Gk):
    """Every kept-group set consistent with the group scores up to TIE_EPS: groups clearly
    above the cut are kept, groups clearly below are dropped, the rest fill the remainder."""
    import itertools
    cut = np.sort(gs)[::-1][Gk - 1]
    must = [g for g in range(gs.size) if gs[g] > cut + TIE_EPS]
    amb = [g for g in range(gs.size) if abs(gs[g] - cut) <= TIE_EPS]
    for extra in itertools.combinations(amb, Gk - len(must)):
        yield set(must) | set(extra)


def _valid_under_ties(s, gs, chosen, gsz, Gk, K, kept):
    """The chosen experts lie in `kept` and are a top-K of its candidates up to TIE_EPS."""
    if not all(int(e) // gsz in kept for e in chosen):
        return False
    cand = [e for e in range(s.size) if e // gsz in kept]
    rest = [e for e in cand if e not in set(chosen.tolist())]
    return not rest or s[chosen].min() >= max(s[e] for e in rest) - TIE_EPS


def check_output(gpu_out_bits: np.ndarray, ref: np.ndarray, tol: float, label: str | None = None,
                 rms_bar: float | None = None):
    """max |gpu - ref| <= tol * RMS(ref) (and, given rms_bar, RMS(gpu - ref) <= rms_bar * RMS(ref));
    logs both ratios under `label`; returns (max_err, rms). gpu_out_bits: bf16 bit patterns
    (uint16) or float32 values."""
    g = bf16_to_f64(gpu_out_bits) if gpu_out_bits.dtype == np.uint16 else gpu_out_bits.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    e = np.abs(g - ref)
    err = float(np.max(e))
    rerr = float(np.sqrt(np.mean(e ** 2)))
    if label:
        report(label, f"{e.size} elements: max|err|/RMS = {err / rms:.3e} (bar {tol:g}), "
                      f"RMS(err)/RMS = {rerr / rms:.3e}" + (f" (bar {rms_bar:g})" if rms_bar else ""))
    assert np.all(np.isfinite(g)), "non-finite output"
    assert err <= tol * rms, f"max|err| {err:.4g} > {tol} * RMS {rms:.4g}"
    if rms_bar is not None:
        assert rerr <= rms_bar * rms, f"RMS(err) {rerr:.4g} > {rms_bar} * RMS {rms:.4g}"
    return err, rms


def oracle_weights(dw: DeviceWeights):
    return dw.host
