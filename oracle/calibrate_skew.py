"""Bias strength for the skewed-routing workload (writes synth/_calibration.py).

The skewed prefill workload draws expert popularity from Zipf(1.2) over a seeded permutation:
b_e = alpha * (ln p_e - mean ln p), p_e proportional to rank(e)^-1.2. The pages ask for the
hottest expert to get about 10x the mean load; this script bisects alpha on the oracle router
(T=4096 tokens of the workload) until max load / mean load lies in [9.5, 10.5], and freezes it.

Run:  python -m oracle.calibrate_skew
"""
import dataclasses
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402


def hot_ratio(scores, cfg, alpha):
    b = synth.zipf_bias(cfg, alpha).numpy()
    idx, _ = oracle.select(scores, b, cfg.k, cfg.n_group, cfg.topk_group, cfg.route_scale)
    c = np.bincount(idx.reshape(-1), minlength=cfg.E)
    return c.max() / c.mean()


def main():
    cfg = synth.CONFIGS["dsv3_skew_prefill"]
    inp = synth.make_router_inputs(dataclasses.replace(cfg, bias="uniform"))   # x and gate only
    x = synth.bf16_bits(inp["x"])
    _, _, _, scores = oracle.route(x, inp["w_gate"].numpy(), np.zeros(cfg.E, np.float32), cfg.k,
                                   cfg.n_group, cfg.topk_group, cfg.route_scale, want_scores=True)
    lo, hi = 0.0, 1.0
    while hot_ratio(scores, cfg, hi) < 10.0:
        hi *= 2
    for _ in range(40):
        mid = (lo + hi) / 2
        r = hot_ratio(scores, cfg, mid)
        if 9.5 <= r <= 10.5:
            lo = hi = mid
            break
        if r < 10.0:
            lo = mid
        else:
            hi = mid
    alpha = float(np.float32((lo + hi) / 2))
    r = hot_ratio(scores, cfg, alpha)
    assert 9.5 <= r <= 10.5, r
    path = os.path.join(ROOT, "synth", "_calibration.py")
    with open(path, "w") as f:
        f.write("# Written by oracle/calibrate_skew.py; do not edit by hand.\n")
        f.write(f"# Oracle router at T={cfg.T}: hottest expert load / mean load = {r:.3f}\n")
        f.write(f"ZIPF_ALPHA = {alpha!r}\n")
    print(f"alpha={alpha} hot/mean={r:.3f}")


if __name__ == "__main__":
    main()
