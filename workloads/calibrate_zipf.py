"""Writes workloads/zipf_alpha.json: the Zipf logit-bias strength of the qwen3 shape.

The qwen3 workload adds b_e = alpha * (-1.2 * ln r_e) to the router logits so
that hot experts receive about ten times the mean load T*k/E. This script
draws the shape's x and W_r (seed 0), routes them with the CPU oracle, and
bisects alpha until the hottest expert's load is 10x the mean. Run once:

    python -m workloads.calibrate_zipf
"""
import json
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

from oracle import moe_oracle as O  # noqa: E402
import workloads as W  # noqa: E402


def max_over_mean(alpha, logits, cfg, ranks):
    bias = (alpha * (-1.2) * np.log(ranks)).astype(np.float32)
    idx, _ = O.route(logits, cfg, bias)
    counts = np.bincount(idx.ravel(), minlength=cfg.E)
    return counts.max() / (cfg.T * cfg.k / cfg.E)


def main(target=10.0):
    cfg = W.QWEN3
    inp = W.make_inputs(cfg.with_(bias_kind="none"), seed=0, weights=False, grad=False)
    logits = O.router_logits(inp["x"].double().numpy(), inp["W_r"].double().numpy())
    g = torch.Generator().manual_seed(0 + 7919)
    ranks = (torch.randperm(cfg.E, generator=g).double() + 1.0).numpy()
    lo, hi = 0.0, 8.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if max_over_mean(mid, logits, cfg, ranks) < target:
            lo = mid
        else:
            hi = mid
    alpha = round(hi, 6)
    ratio = max_over_mean(alpha, logits, cfg, ranks)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_alpha.json")
    with open(path, "w") as f:
        json.dump({"alpha": alpha, "max_over_mean_load": round(float(ratio), 4), "target": target,
                   "shape": "qwen3 T=16384 H=4096 E=128 k=8", "seed": 0}, f, indent=1)
    print(alpha, ratio)


if __name__ == "__main__":
    main()
