"""Writes mixtral_router_scale.json: the w_router scale of the Mixtral-shaped
workload (T=4096, d=4096, N=8, top-2) at which the token-mean of the largest
full-softmax router probability is 0.40 ("top-1 share about 0.4").

Calls only the oracle router (and the seeded input generator for the inputs).
Run from the repository root:  python tests/golden/make_mixtral_router_scale.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

from mixture_experts_layer_94_b300 import inputs  # noqa: E402
from oracle import oracle  # noqa: E402

TARGET = 0.40


def top1_share(hidden, w_router, scale):
    r = oracle.router(hidden, w_router * scale, K=2, score_fn=oracle.SOFTMAX)
    return float(r["probs"].max(axis=1).mean())


def main():
    cfg = inputs.MIXTRAL.with_(router_scale=1.0)
    ri = inputs.make_router_inputs(cfg, seed=0)
    hidden = ri["hidden"].float().numpy()
    w_router = ri["w_router"].numpy()
    lo, hi = 0.5, 3.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if top1_share(hidden, w_router, mid) < TARGET:
            lo = mid
        else:
            hi = mid
    scale = round(0.5 * (lo + hi), 4)
    out = {
        "workload": "Mixtral-8x7B-shaped prefill, T=4096, d=4096, N=8, top-2, seed 0",
        "quantity": "w_router scale s with mean_t max_e softmax(s * logits)_e = 0.40",
        "reading": "'top-1 share about 0.4' read as the token-mean of the largest "
                   "full-softmax router probability",
        "router_scale": scale,
        "top1_share_at_scale": round(top1_share(hidden, w_router, scale), 5),
        "top1_share_at_1": round(top1_share(hidden, w_router, 1.0), 5),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "mixtral_router_scale.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(json.dumps(out, indent=1))


if __name__ == "__main__":
    main()
