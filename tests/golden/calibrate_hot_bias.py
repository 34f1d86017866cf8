"""Bisect the router-bias offset of the two hot experts of the E=16 GELU
workload (T=8192, d=4096, top-2) so that each receives about three times the
mean load, 3*T*k/E = 3072 assignments.  Calls only the oracle and the input
generator; prints the offset that the generator hard-codes (HOT2_BIAS).

    python tests/golden/calibrate_hot_bias.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402
from top_routing_expert_02_b300 import synth  # noqa: E402


def hot_load(L0, beta, E, k):
    b = np.zeros(E)
    b[:2] = beta
    idx, _, _ = oracle.route(L0 + b, k)
    return np.bincount(idx.ravel(), minlength=E)[:2].mean()


def main():
    cfg = synth.workload("e16_gelu_hot2")
    ri = synth.make_routing_inputs(cfg)
    L0 = oracle.router_logits(ri.x, ri.W, None)      # logits without bias
    target = 3.0 * cfg.T * cfg.k / cfg.E
    lo, hi = 0.0, 4.0
    while hi - lo > 0.01:
        mid = 0.5 * (lo + hi)
        if hot_load(L0, mid, cfg.E, cfg.k) < target:
            lo = mid
        else:
            hi = mid
    beta = round(hi, 2)
    print(f"HOT2_BIAS = {beta:.2f}  (mean hot load {hot_load(L0, beta, cfg.E, cfg.k):.1f}, target {target:.0f})")


if __name__ == "__main__":
    main()
