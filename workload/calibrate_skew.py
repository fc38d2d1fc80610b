"""Calibrate the router bias of the skewed long-prefill workload.

The skewed workload shifts every token by a seeded mean vector m and adds
beta * m/|m| to the router columns of 16 hot experts (8 in each of two groups).
This script bisects beta, routing the first 2048 tokens with the CPU oracle,
until the hot experts' mean load is 4x the mean load T*K/E, and stores beta in
skew_beta.json. It calls only the oracle and the generators; run it from the
repository root:  python -m workload.calibrate_skew
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import workload as W  # noqa: E402

TARGET = 4.0
N_TOK = 2048
SEED = 0


def hot_ratio(beta: float, x: np.ndarray, cfg) -> float:
    wr = W.gen_wr(cfg, SEED, beta=beta)
    r = oracle.route(cfg.with_tokens(N_TOK), x, wr)
    counts = np.bincount(r["idx"].ravel(), minlength=cfg.E)
    mean = N_TOK * cfg.top_k / cfg.E
    return float(counts[list(cfg.hot_experts)].mean() / mean)


def main():
    cfg = W.CONFIGS["skewed"]
    x = W.gen_x(cfg, SEED, 0, N_TOK)
    lo, hi = 0.0, 1.0
    while hot_ratio(hi, x, cfg) < TARGET:
        hi *= 2
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if hot_ratio(mid, x, cfg) < TARGET:
            lo = mid
        else:
            hi = mid
    beta = 0.5 * (lo + hi)
    ratio = hot_ratio(beta, x, cfg)
    out = {"beta": beta, "hot_load_ratio": ratio, "tokens": N_TOK, "seed": SEED,
           "hot_experts": list(cfg.hot_experts), "target": TARGET}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "skew_beta.json"), "w") as f:
        json.dump(out, f, indent=1)
    print(out)


if __name__ == "__main__":
    main()
