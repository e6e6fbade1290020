"""Writes ``spec_inputs/draft_noise_table.json``: the draft-logit noise level
sigma that gives a target acceptance rate alpha for Gaussian target logits.

The synthetic draft logits are ``q_logits = L + sigma * z`` (z ~ N(0, 1)),
the target logits L ~ N(0, s^2) per token.  At temperature T the pair
(L / T, q_logits / T) depends only on s / T and sigma / T, so the table is
keyed by the scaled logit spread s / T and stores sigma / T.  alpha is the
acceptance mass sum_v min(p(v), q(v)) of "Speculative Decoding: Two Models,
One Voice" (Tool 1), computed with the oracle's softmax and emitted-law
functions and averaged over rows; sigma is found by bisection.

Run:  python -m oracle.calibrate_draft_noise
"""
import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(os.path.dirname(HERE), "spec_inputs", "draft_noise_table.json")

V = 128256
ROWS = 6
SPREADS = [1.0, 1.28, 1.81, 1.83]          # s / T of the configurations
ALPHAS = [0.5, 0.55, 0.6, 0.65, 0.7, 0.75, 0.8, 0.85, 0.9]


def mean_alpha(spread, noise, seed=0):
    rng = np.random.default_rng(seed)
    total = 0.0
    for _ in range(ROWS):
        L = spread * rng.standard_normal(V)
        ql = L + noise * rng.standard_normal(V)
        total += oracle.emitted_law(oracle.softmax(L), oracle.softmax(ql))[1]
    return total / ROWS


def solve(spread, alpha):
    lo, hi = 1e-4, 20.0            # alpha falls as the noise grows
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if mean_alpha(spread, mid) > alpha:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def main():
    table = {"V": V, "rows_per_estimate": ROWS,
             "key": "scaled target-logit spread s/T",
             "value": "scaled draft noise sigma/T for each alpha",
             "alphas": ALPHAS, "spreads": {}}
    for s in SPREADS:
        table["spreads"][f"{s:.2f}"] = [round(solve(s, a), 5) for a in ALPHAS]
        print(s, table["spreads"][f"{s:.2f}"], flush=True)
    with open(OUT, "w") as f:
        json.dump(table, f, indent=1)


if __name__ == "__main__":
    main()
