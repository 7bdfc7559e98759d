"""Writes the HYBRID thresholds gamma used by the layer configs.

gamma = median router probability of the routed (token, expert) pairs that
are missing from the available set, for the seed-0 tokens of each HYBRID
layer, rounded to three decimals.  Uses only the oracle's router steps and the
seeded inputs; prints the values to paste into workloads.CONFIGS.
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "..", ".."))
import oracle  # noqa: E402
from workloads import CONFIGS, make_tokens, make_weights  # noqa: E402


def missed_gates(cfg):
    W = make_weights(cfg, experts=[])
    x = make_tokens(cfg)
    l = oracle.logits(x, W.w_router, W.router_bias)
    lp = oracle.logits(x, W.w_prefetch)
    if cfg.n_resident > 0:
        resident, _ = oracle.batch_resident(lp, cfg.n_resident)
    else:
        resident = (1 << 64) - 1
    gates = []
    for t in range(x.shape[0]):
        a = oracle.softmax(l[t])
        routed = oracle.topk(l[t], cfg.k)
        avail = resident
        if cfg.use_prefetch_mask:
            dh, _ = oracle.delta_hat(W.w_ord, x[t], W.theta, cfg.tau)
            avail &= oracle.prefetch_set(cfg.k, dh, lp[t])
        gates += [a[e] for e in routed if not (avail >> int(e)) & 1]
    return np.array(gates)


if __name__ == "__main__":
    for name, cfg in CONFIGS.items():
        if cfg.policy != 3:
            continue
        g = missed_gates(cfg)
        print(f"{name}: misses={g.size} gamma={np.round(np.median(g), 3)}")
