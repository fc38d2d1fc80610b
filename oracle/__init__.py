"""CPU oracle of the Beam MoE block (ctypes binding of ``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the package smoke check
and the benchmark's CPU-baseline leg, never by the product path. It restates
the block as the Beam release article defines it (section "Mixture of
Experts": sigmoid router over 256 experts, 8 groups of 32, top-2-sum group
score, 4 groups kept, top-8 experts, weights normalised to 1 then x2.5, SwiGLU
experts; section "Residual stream": router and SwiGLU product in FP32), with
double accumulation. See ``oracle.c`` for each function's definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

WFMT = {"bf16": 0, "nvfp4": 1, "fp8": 2}


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle into a shared library (plain gcc, OpenMP, no fp contraction)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, src, "-lm"])
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (and declare) an oracle library; ``path`` selects a variant build."""
    L = ctypes.CDLL(path or build())
    i32, vp, dbl = ctypes.c_int, ctypes.c_void_p, ctypes.c_double
    L.oracle_e2m1_value.argtypes = [i32]
    L.oracle_e2m1_value.restype = dbl
    L.oracle_e4m3_value.argtypes = [i32]
    L.oracle_e4m3_value.restype = dbl
    L.oracle_router_scores.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    L.oracle_select.argtypes = [i32, i32, i32, i32, i32, dbl, vp, vp, vp, vp, vp, vp]
    L.oracle_select.restype = i32
    L.oracle_select_biased.argtypes = [i32, i32, i32, i32, i32, dbl, vp, vp, vp, vp, vp, vp, vp]
    L.oracle_select_biased.restype = i32
    L.oracle_permute.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp]
    L.oracle_ffn_rows.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.oracle_combine.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    L.oracle_forward_tokens.argtypes = [i32, i32, i32, i32, vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp,
                                        vp, vp, vp, vp]
    L.oracle_num_threads.restype = i32
    L.oracle_residual_update.argtypes = [i32, i32, vp, vp, vp, dbl, i32, vp]
    L.oracle_pre_norm.argtypes = [i32, i32, vp, vp, dbl, vp]
    return L


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return lib().oracle_num_threads()


def router_scores(x, w_r, L=None):
    """FP32 logits and sigmoid scores [T, E] from bf16 x [T, d] and fp32 w_r [d, E]."""
    L = L or lib()
    T, d = x.shape
    E = w_r.shape[1]
    logits = np.empty((T, E), np.float32)
    scores = np.empty((T, E), np.float32)
    L.oracle_router_scores(T, d, E, _p(x), _p(w_r), _p(logits), _p(scores))
    return logits, scores


def select(scores, n_groups, topk_groups, top_k, routed_scale=2.5, L=None, bias=None):
    """Group-limited top-k: returns dict(idx [T,K] i32, w [T,K] f64, gscores [T,G] f32,
    margin_group [T], margin_expert [T]). `bias` [E] f32: per-expert selection bias (it
    steers the choice; the weights use the unbiased scores)."""
    L = L or lib()
    scores = np.ascontiguousarray(scores, np.float32)
    T, E = scores.shape
    idx = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float64)
    gs = np.empty((T, n_groups), np.float32)
    mg = np.empty(T, np.float64)
    me = np.empty(T, np.float64)
    if bias is None:
        rc = L.oracle_select(T, E, n_groups, topk_groups, top_k, routed_scale, _p(scores), _p(idx), _p(w),
                             _p(gs), _p(mg), _p(me))
    else:
        bias = np.ascontiguousarray(bias, np.float32)
        assert bias.shape == (E,)
        rc = L.oracle_select_biased(T, E, n_groups, topk_groups, top_k, routed_scale, _p(scores), _p(bias),
                                    _p(idx), _p(w), _p(gs), _p(mg), _p(me))
    if rc < 0:
        raise ValueError("invalid selection dims")
    return {"idx": idx, "w": w, "gscores": gs, "margin_group": mg, "margin_expert": me,
            "zero_sum_tokens": rc}


def route(cfg, x, w_r, L=None, bias=None):
    """Router of the block: scores then group-limited selection (optional selection bias [E])."""
    logits, scores = router_scores(x, w_r, L)
    out = select(scores, cfg.n_groups, cfg.topk_groups, cfg.top_k, cfg.routed_scale, L, bias=bias)
    out["logits"], out["scores"] = logits, scores
    return out


def permute(idx, E, L=None):
    """(counts [E], offsets [E+1], row_token [T*K], inv_row [T*K]) for routing idx [T, K]."""
    L = L or lib()
    idx = np.ascontiguousarray(idx, np.int32)
    T, K = idx.shape
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    row_token = np.empty(T * K, np.int32)
    inv_row = np.empty(T * K, np.int32)
    L.oracle_permute(T, E, K, _p(idx), _p(counts), _p(offsets), _p(row_token), _p(inv_row))
    return counts, offsets, row_token, inv_row


def _wargs(weights, wfmt):
    if wfmt == "bf16":
        return [_p(weights["gate"]), _p(weights["up"]), _p(weights["down"]), None, None, None, None, None, None]
    if wfmt == "fp8":  # e4m3 codes and fp32 128 x 128 block scales
        return [_p(weights["gate"]), _p(weights["up"]), _p(weights["down"]),
                _p(weights["gate_sf"]), _p(weights["up_sf"]), _p(weights["down_sf"]), None, None, None]
    return [_p(weights["gate"]), _p(weights["up"]), _p(weights["down"]),
            _p(weights["gate_sf"]), _p(weights["up_sf"]), _p(weights["down_sf"]),
            _p(weights["gate_ts"]), _p(weights["up_ts"]), _p(weights["down_ts"])]


def ffn_rows(row_expert, xrows, weights, d, inter, wfmt="bf16", want_h=False, L=None):
    """Expert SwiGLU MLP on independent rows: returns y [n, d] f64 (and h [n, I] bf16 bits)."""
    L = L or lib()
    row_expert = np.ascontiguousarray(row_expert, np.int32)
    xrows = np.ascontiguousarray(xrows, np.uint16)
    n = row_expert.size
    y = np.empty((n, d), np.float64)
    h = np.empty((n, inter), np.uint16) if want_h else None
    L.oracle_ffn_rows(n, d, inter, WFMT[wfmt], _p(row_expert), _p(xrows), *_wargs(weights, wfmt), _p(h), _p(y))
    return (y, h) if want_h else y


def combine(y_rows, inv_row, w, L=None):
    """out [T, d] f64 = sum_k w[t,k] * y_rows[inv_row[t*K+k]]."""
    L = L or lib()
    y_rows = np.ascontiguousarray(y_rows, np.float32)
    w = np.ascontiguousarray(w, np.float64)
    T, K = w.shape
    d = y_rows.shape[1]
    out = np.empty((T, d), np.float64)
    L.oracle_combine(T, K, d, _p(y_rows), _p(np.ascontiguousarray(inv_row, np.int32)), _p(w), _p(out))
    return out


def residual_update(out, h_old, gamma, eps, step, L=None):
    """Post-norm and depth-scaled residual addition: h_new [T, d] f64 from the sublayer output
    out [T, d] f64, the stream h_old [T, d] bf16 bits, the norm gain gamma [d] bf16 bits."""
    L = L or lib()
    out = np.ascontiguousarray(out, np.float64)
    T, d = out.shape
    h_new = np.empty((T, d), np.float64)
    L.oracle_residual_update(T, d, _p(out), _p(np.ascontiguousarray(h_old, np.uint16)),
                             _p(np.ascontiguousarray(gamma, np.uint16)), float(eps), int(step), _p(h_new))
    return h_new


def pre_norm(h, gamma, eps, L=None):
    """Pre-norm of the sublayer input: x [T, d] bf16 bits = bf16(RMSNorm(h) * gamma) from the
    stream h [T, d] bf16 bits and the gain gamma [d] bf16 bits."""
    L = L or lib()
    h = np.ascontiguousarray(h, np.uint16)
    T, d = h.shape
    x = np.empty((T, d), np.uint16)
    L.oracle_pre_norm(T, d, _p(h), _p(np.ascontiguousarray(gamma, np.uint16)), float(eps), _p(x))
    return x


def forward_tokens(cfg, x, idx, w, tokens, weights, L=None):
    """Block output [len(tokens), d] f64 for the given tokens under routing (idx, w)."""
    L = L or lib()
    tokens = np.ascontiguousarray(tokens, np.int32)
    out = np.empty((tokens.size, cfg.d), np.float64)
    L.oracle_forward_tokens(cfg.d, cfg.inter, cfg.top_k, WFMT[cfg.wfmt], _p(np.ascontiguousarray(x)),
                            _p(np.ascontiguousarray(idx, np.int32)), _p(np.ascontiguousarray(w, np.float64)),
                            tokens.size, _p(tokens), *_wargs(weights, cfg.wfmt), _p(out))
    return out


def e2m1_value(code: int, L=None) -> float:
    return (L or lib()).oracle_e2m1_value(code)


def e4m3_value(code: int, L=None) -> float:
    return (L or lib()).oracle_e4m3_value(code)
