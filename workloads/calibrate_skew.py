"""Report the overflow share of the skewed-overflow workload for a few Zipf
strengths, using the CPU oracle's router and slot assignment only.

The skewed shape (T=16384, d=1024, N=64, cf=1.0, gate-value priority) asks
for 10-30 % of the tokens to overflow.  ``SKEW_ZIPF_LAMBDA`` in
``workloads/__init__.py`` was frozen from this script's output on seed 0.

    python -m workloads.calibrate_skew
"""
import numpy as np

import oracle
from workloads import CONFIGS, make_inputs, zipf_bias


def drop_fraction(lam: float, seed: int = 0) -> tuple:
    w = CONFIGS["skew"].replace(zipf_lambda=lam)
    inp = make_inputs(w, seed, with_experts=False)
    r = oracle.route(inp.x, inp.W_g, zipf_bias(w))
    C = oracle.capacity(w.T, w.N, w.capacity_factor)
    _, drop, counts = oracle.assign_slots(r["expert_id"], r["gate"], w.N, C, w.priority_mode)
    return float(drop.mean()), float(counts.max() / (w.T / w.N))


if __name__ == "__main__":
    for lam in (0.05, 0.10, 0.12, 0.15, 0.20):
        d, s = drop_fraction(lam)
        print(f"lambda={lam:.2f}  dropped={d:.3f}  max/mean load={s:.2f}")
