"""Calibrate the two free constants of the synthetic input recipe with the oracle.

Run: ``python -m oracle.calibrate_inputs``. It prints the router weight scale
and the prefill bias skew that ``datagen`` stores as constants; nothing else
reads its output.

1. Router scale s for the d=4096 decode workloads: W_r = bf16(s * N(0, 0.02^2)),
   chosen so that about 5% of N(0,1) tokens (seed 0, 16384 tokens) have a gap
   below 0.05 between their 8th and 9th largest fp32 router logit.
2. Zipf skew alpha for the T=4096 prefill workload: bias b_e = alpha * (-1.1 ln r_e)
   with r a seeded permutation of 1..256, chosen so that max/mean expert load
   is about 4.
Both use only the oracle's router and top-k selection.
"""
from __future__ import annotations

import numpy as np

import datagen
import oracle


def gap_fraction(scale: float, n_tokens: int, seed: int = 0, thresh: float = 0.05) -> float:
    w = datagen.WORKLOADS["decode_t1"]
    wr = datagen.normal_bf16(seed, datagen.tag(datagen.TAG_ROUTER, 0), (w.E, w.d),
                             datagen.WEIGHT_SIGMA * scale)
    x = datagen.tokens(w, n_tokens, seed=seed)
    lg = oracle.router_logits(x, wr)
    _, _, gap = oracle.select_topk(lg, w.k)
    return float(np.mean(gap < thresh))


def load_ratio(alpha: float, logits: np.ndarray, seed: int = 0) -> float:
    w = datagen.WORKLOADS["prefill_t4096"]
    bias = datagen.router_bias(w, seed=seed, alpha=alpha)
    lg = logits if bias is None else (logits + bias[None, :]).astype(np.float32)
    ids, _, _ = oracle.select_topk(lg, w.k)
    counts = np.bincount(ids.ravel(), minlength=w.E)
    return float(counts.max() / counts.mean())


def main() -> None:
    lo, hi = 5.0, 30.0
    for _ in range(12):
        mid = 0.5 * (lo + hi)
        f = gap_fraction(mid, 16384)
        print(f"scale {mid:.4f}: gap<0.05 fraction {f:.4f}", flush=True)
        if f > 0.05:
            lo = mid
        else:
            hi = mid
    s = round(0.5 * (lo + hi), 2)
    print(f"ROUTER_SCALE_D4096 = {s}  (fraction {gap_fraction(s, 16384):.4f})")

    w = datagen.WORKLOADS["prefill_t4096"]
    wr = datagen.normal_bf16(0, datagen.tag(datagen.TAG_ROUTER, 0), (w.E, w.d), datagen.WEIGHT_SIGMA * s)
    x = datagen.tokens(w, w.T)
    base = oracle.router_logits(x, wr)
    lo, hi = 0.0, 20.0
    for _ in range(14):
        mid = 0.5 * (lo + hi)
        r = load_ratio(mid, base)
        print(f"alpha {mid:.4f}: max/mean load {r:.3f}", flush=True)
        if r < 4.0:
            lo = mid
        else:
            hi = mid
    a = round(0.5 * (lo + hi), 2)
    print(f"ZIPF_ALPHA = {a}  (max/mean {load_ratio(a, base):.3f})")


if __name__ == "__main__":
    main()
