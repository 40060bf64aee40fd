"""Fits the router-logit lifts of the Zipf workloads -- test infrastructure.

The prefill workloads skew the router so that the per-expert pair counts follow Zipf(s = 1.1):
the router's last column adds a lift to every token's logit of the expert of rank r
(synth.zipf_logit_offsets), aiming at target_r, the water-filled Zipf counts
(synth.zipf_targets).  Closeness is the total variation TV = sum_r |count_r - target_r| /
(2 T k) of the seed-0 workload's counts under the oracle's fp64 routing.

1. Single scale: lift_r = tau * ln(target_r / T).  A coarse grid of tau, then a golden-section
   search of the bracket around the best grid point (4096-token workload); the result is
   synth.ZIPF_TAU, copied there by hand.
2. Per rank: starting from step 1, damped fixed-point passes lift_r += alpha * ln((target_r +
   1/2) / (count_r + 1/2)); the pass with the smallest TV is kept.  Written, with the realized
   counts, to block_quantized_moe_router_gb300/zipf_lifts.json for the named prefill workloads
   (the input recipe reads it; nothing reads this script at run time).

    python tests/zipf_fit.py [--tau] [pre4096 pre32768 ...]
"""
from __future__ import annotations

import math
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.join(ROOT, "tests"))

import oracle  # noqa: E402
from block_quantized_moe_router_gb300 import synth  # noqa: E402


def realized_counts(cfg, tau=None, lifts=None, seed=0):
    """Per-rank pair counts of the oracle's routing of the workload built with these lifts."""
    inp = synth.make_inputs(cfg, seed=seed, with_weights=False, zipf_tau=tau, zipf_lifts=lifts)
    r = oracle.route(T=cfg.T, E=cfg.E, k=cfg.k, scoring=cfg.scoring, renorm=cfg.renorm,
                     scaling=cfg.scaling, x_bf16=synth.bf16_bits(inp["x"]),
                     w_router_bf16=synth.bf16_bits(inp["w_router"]), bias=inp["bias"].numpy())
    per_expert = np.bincount(r["ids"].ravel(), minlength=cfg.E)
    by_rank = np.empty(cfg.E, dtype=np.int64)
    by_rank[synth.zipf_rank_of_expert(cfg, seed)] = per_expert
    return by_rank


def total_variation(cfg, counts):
    tgt = synth.zipf_targets(cfg.T, cfg.k, cfg.E, cfg.zipf_s)
    return float(np.abs(counts - tgt).sum() / (2.0 * cfg.T * cfg.k))


def fit(cfg, lo=0.25, hi=6.0, step=0.25, iters=14, verbose=True):
    memo = {}

    def tv(tau):
        tau = round(tau, 6)
        if tau not in memo:
            memo[tau] = total_variation(cfg, realized_counts(cfg, tau=tau))
            if verbose:
                print(f"  tau {tau:.4f}  TV {memo[tau]:.4f}", flush=True)
        return memo[tau]

    grid = np.arange(lo, hi + 1e-9, step)
    vals = [tv(t) for t in grid]
    i = int(np.argmin(vals))
    a, b = grid[max(0, i - 1)], grid[min(len(grid) - 1, i + 1)]
    g = (math.sqrt(5) - 1) / 2
    c, d = b - g * (b - a), a + g * (b - a)
    for _ in range(iters):
        if tv(c) <= tv(d):
            b, d = d, c
            c = b - g * (b - a)
        else:
            a, c = c, d
            d = a + g * (b - a)
    best = min(memo, key=memo.get)
    return best, memo[best]


def refine(cfg, tau, passes=28, alpha=0.7, verbose=True):
    """Per-rank lifts by damped fixed-point passes, started from the single-scale form."""
    tgt = synth.zipf_targets(cfg.T, cfg.k, cfg.E, cfg.zipf_s)
    lifts = tau * np.log(tgt / cfg.T)
    best = (float("inf"), None, None)
    for it in range(passes):
        counts = realized_counts(cfg, lifts=lifts)
        tv = total_variation(cfg, counts)
        if verbose:
            print(f"  pass {it:2d}  TV {tv:.4f}  head {counts[:3].tolist()}", flush=True)
        if tv < best[0]:
            best = (tv, lifts.copy(), counts.copy())
        lifts = np.clip(lifts + alpha * np.log((tgt + 0.5) / (counts + 0.5)), -30.0, 30.0)
    return best


if __name__ == "__main__":
    args = [a for a in sys.argv[1:] if not a.startswith("--")]
    if "--tau" in sys.argv:
        cfg = synth.CONFIGS["pre4096"]
        tau, val = fit(cfg)
        print(f"best single scale tau {tau:.4f}: TV {val:.4f}")
    import json
    path = synth._ZIPF_LIFTS_FILE
    table = json.load(open(path)) if os.path.exists(path) else {}
    for name in args or ["pre4096"]:
        cfg = synth.CONFIGS[name]
        tv, lifts, counts = refine(cfg, synth.ZIPF_TAU)
        tgt = synth.zipf_targets(cfg.T, cfg.k, cfg.E, cfg.zipf_s)
        print(f"{name}: TV {tv:.4f}")
        for r in (0, 1, 2, 3, 4, 9, 49, 127, 255):
            print(f"  rank {r + 1:3d}: target {tgt[r]:8.1f}  realized {counts[r]:6d}")
        table[name] = {"tv": round(tv, 5), "lifts": [round(float(v), 6) for v in lifts],
                       "realized_counts_by_rank": [int(c) for c in counts],
                       "note": "per-rank router-logit lifts written by tests/zipf_fit.py"}
        with open(path, "w") as fh:
            json.dump(table, fh, indent=0)
