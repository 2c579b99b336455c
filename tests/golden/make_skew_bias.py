"""Write tests/golden/skew_bias.json: the expert-0 logit bias that gives each
router-skew target (maxvio) on the seeded synthetic router inputs.

    python tests/golden/make_skew_bias.py

maxvio (MoonEP page, "What problem it solves") is max_e load_e / (T*K/E) - 1.
The bias beta is added to expert 0's logit before softmax and selection; it is
found by bisection on the CPU oracle's routing of the seed-0 inputs (x ~ N(0,1),
W_r ~ N(0, 0.02), bf16 storage), so that the oracle's maxvio lands within 2% of
the target.  Because a token sends at most one of its K picks to an expert,
maxvio <= E/K - 1; targets above that are recorded as unreachable, and "max"
stands for the largest skew the bias reaches.  A target below the router's
natural skew is met with beta = 0 and the natural value recorded.

Only the oracle and the input generator are called here.
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from token_dispatch_gb300 import synth  # noqa: E402

TARGETS = {
    synth.MIXTRAL_BF16.name: [0.2],
    synth.FINEGRAINED_BF16.name: [0.2, 1.0, 5.0, 10.0, 20.0],
    synth.EPBENCH_BF16.name: [0.2, 1.0, 10.0, 20.0],
}


def maxvio_at(logits, beta, K, E, T):
    l = logits.copy()
    l[:, 0] += beta
    idx = O.topk_experts(l, K)
    return O.maxvio(O.expert_histogram(idx, E), T, K, E)


def solve(shape):
    x, wr = synth.router_inputs(shape)
    logits = O.router_logits(x.ref, wr.ref)
    T, E, K = shape.T, shape.E, shape.K
    natural = maxvio_at(logits, 0.0, K, E, T)
    ceiling = E / K - 1
    out = {"natural_maxvio": natural, "ceiling": ceiling}
    for target in TARGETS[shape.name]:
        key = f"{target:g}"
        if target > ceiling:
            hi = 1.0
            while maxvio_at(logits, hi, K, E, T) < ceiling - 1e-12 and hi < 1e4:
                hi *= 2
            out[key] = {"beta": hi, "maxvio_oracle": maxvio_at(logits, hi, K, E, T),
                        "note": f"unreachable: maxvio <= E/K - 1 = {ceiling:.4g}; largest skew instead"}
            continue
        if target <= natural:
            out[key] = {"beta": 0.0, "maxvio_oracle": natural, "note": "natural skew already at or above target"}
            continue
        lo, hi = 0.0, 1.0
        while maxvio_at(logits, hi, K, E, T) < target:
            hi *= 2
        best = (hi, maxvio_at(logits, hi, K, E, T))
        for _ in range(60):
            mid = 0.5 * (lo + hi)
            v = maxvio_at(logits, mid, K, E, T)
            if abs(v - target) < abs(best[1] - target):
                best = (mid, v)
            if abs(v - target) <= 0.02 * target:
                break
            if v < target:
                lo = mid
            else:
                hi = mid
        out[key] = {"beta": best[0], "maxvio_oracle": best[1]}
    return out


def main():
    table = {name: solve(synth.WORKLOADS[name]) for name in TARGETS}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "skew_bias.json")
    with open(path, "w") as fh:
        json.dump(table, fh, indent=1, sort_keys=True)
    print(json.dumps(table, indent=1))


if __name__ == "__main__":
    main()
