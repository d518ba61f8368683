"""Write tests/golden/entropy_temperatures.json.

For each of the three activation batches of the entropy-adaptive workload,
bisect the router's inverse temperature until the oracle's batch-mean
softmax entropy reaches the middle of one k band of the adaptive rule
(k=1: H < 1.2, k=2: 1.2 <= H < 2.5, k=3: H >= 2.5; page "Qwen3.5-MoE与
Qwen3-MoE架构差异深度解析", section 2.2).  Targets 0.6, 1.85 and 3.0 nats
keep every batch at least 0.5 nats away from a band edge.

Calls only the oracle and the seeded generator.  Run from the repo root:
    python tests/golden/make_entropy_temperatures.py
then copy the printed tuple into workloads.ENTROPY_INV_TEMPERATURES.
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import workloads  # noqa: E402

TARGETS = (0.6, 1.85, 3.0)


def mean_entropy(x, w, inv_t):
    return float(oracle.batch_mean_entropy(oracle.softmax_entropy(oracle.router_logits(x, w, None, inv_t))))


def main():
    cfg = workloads.CONFIGS["entropy"]
    layer_w = workloads.normal_f32(0, workloads.STREAM_ROUTER, (cfg.E, cfg.H), cfg.router_std)
    out = {"config": "entropy", "targets": list(TARGETS), "inv_temperatures": [], "mean_entropy": []}
    for b, target in enumerate(TARGETS):
        x = workloads.make_tokens(cfg, 0, b)
        lo, hi = 1e-3, 100.0   # entropy falls as the inverse temperature rises
        for _ in range(60):
            mid = float(np.sqrt(lo * hi))
            if mean_entropy(x, layer_w, mid) > target:
                lo = mid
            else:
                hi = mid
        inv_t = float(np.float32(round(np.sqrt(lo * hi), 6)))
        h = mean_entropy(x, layer_w, inv_t)
        out["inv_temperatures"].append(round(inv_t, 6))
        out["mean_entropy"].append(h)
        print(f"batch {b}: inv_temperature {inv_t:.6f} -> mean entropy {h:.6f} (target {target})")
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "entropy_temperatures.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=2)
    print("ENTROPY_INV_TEMPERATURES =", tuple(out["inv_temperatures"]))


if __name__ == "__main__":
    main()
