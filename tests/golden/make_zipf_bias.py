"""Calibrate the Zipf router-logit bias of the T=16384 skewed workload.

Writes tests/golden/zipf_bias.json.  Calls only the oracle (FP64 logits and
its top-k) and the seeded input generator: beta is bisected so that the
busiest expert receives 20x the mean load R/E (the workload asks for ~20x,
64 experts with no tokens, Zipf(1.1) over a random expert order).

Run:  python tests/golden/make_zipf_bias.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from top_routed_grouped_gb300 import inputs as I  # noqa: E402


def loads_for(logits, beta, cfg):
    b = I.zipf_bias(cfg.E, beta).double().numpy()
    ids = oracle.topk_select(logits + b, cfg.k)
    return np.bincount(ids.reshape(-1), minlength=cfg.E)


def main():
    cfg = I.CONFIGS["bf16_t16384_zipf"]
    x = I.normal((cfg.T, cfg.H), 0, I._STREAM["x"], 1.0, cfg.torch_dtype)
    wr = I.normal((cfg.E, cfg.H), 0, I._STREAM["w_router"], I.WEIGHT_STD)
    logits = oracle.router_logits(x, wr)
    mean = cfg.T * cfg.k / cfg.E
    target = 20.0 * mean
    lo, hi = 0.0, 4.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if loads_for(logits, mid, cfg).max() < target:
            lo = mid
        else:
            hi = mid
    beta = float(np.float32(hi))
    loads = loads_for(logits, beta, cfg)
    # The bias the kernels read is fp32: record loads with the fp32-rounded bias.
    out = {
        "workload": cfg.name, "T": cfg.T, "E": cfg.E, "k": cfg.k, "zipf_s": I.ZIPF_S,
        "n_empty_forced": I.ZIPF_EMPTY, "beta": beta, "mean_load": mean,
        "max_load": int(loads.max()), "max_over_mean": float(loads.max() / mean),
        "empty_experts": int((loads == 0).sum()), "active_experts": int((loads > 0).sum()),
        "loads_sorted_desc_top16": sorted(loads.tolist(), reverse=True)[:16],
        "note": "routing by oracle FP64 logits of x (seed 0) and W_router (seed 0) plus the fp32 bias",
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "zipf_bias.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
