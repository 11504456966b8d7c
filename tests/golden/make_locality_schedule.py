"""Write tests/golden/locality_schedule.json: the correlation of the decode token stream.

The decode-loop workload feeds one Mixtral-shape layer a stream of tokens per
sequence whose consecutive rows are correlated (``moe_inputs.make_token_stream``,
correlation rho), so that consecutive tokens share experts more often than
chance. The lecture page ("Mixtral of Experts", router walkthrough) reports, at
layer 15, that the top-2 expert sets of tokens i and i+1 share an expert 62 %
(ArXiv) and 67 % (DM Mathematics) of the time, against 46 % for a uniform
random router, and that the first choices agree about 28 % of the time (12.5 %
at random). This script bisects rho with the fp64 oracle's router on the
decode workload's router matrix until the shared-expert rate is 0.62 +/- 0.005
(the ArXiv figure), and stores rho with both measured rates. The input package
never evaluates the router; it only replays rho.

Usage: python tests/golden/make_locality_schedule.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from moe_inputs import CONFIGS, make_token_stream, make_tokens, to_f64  # noqa: E402

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "locality_schedule.json")
TARGET = 0.62          # ArXiv, layer 15
CAL_B, CAL_S = 64, 65  # calibration: 64 sequences x 64 transitions
SEED = 5360            # the decode-loop workload's token seed


def rates(x, wg):
    """(shared-expert rate, same-first-choice rate) of consecutive tokens in a [S][B][d] stream."""
    S, B, d = x.shape
    idx, _, _ = oracle.top_k_gates(oracle.router_logits(to_f64(x.reshape(S * B, d)), to_f64(wg)), 2)
    idx = idx.reshape(S, B, 2)
    a, b = idx[:-1], idx[1:]
    shared = (a[..., :, None] == b[..., None, :]).any(axis=(-1, -2))
    first = a[..., 0] == b[..., 0]
    return float(shared.mean()), float(first.mean())


def main():
    c = CONFIGS[1]
    _, wg = make_tokens(1, c["d"], c["E"], c["dtype"], c["seed"])
    lo, hi = 0.0, 0.999
    for _ in range(30):
        rho = 0.5 * (lo + hi)
        sh, fi = rates(make_token_stream(CAL_B, CAL_S, c["d"], rho, SEED), wg)
        print(f"rho {rho:.4f}: shared {sh:.4f} first {fi:.4f}")
        if abs(sh - TARGET) <= 0.005:
            break
        if sh < TARGET:
            lo = rho
        else:
            hi = rho
    sh0, fi0 = rates(make_token_stream(CAL_B, CAL_S, c["d"], 0.0, SEED), wg)
    out = {"_about": __doc__.strip().splitlines()[0], "rho": rho, "seed": SEED, "router": "config 1 w_gate",
           "calibration": {"sequences": CAL_B, "transitions_per_sequence": CAL_S - 1},
           "shared_expert_rate": sh, "same_first_choice_rate": fi,
           "independent_tokens": {"shared_expert_rate": sh0, "same_first_choice_rate": fi0},
           "pages": {"shared_expert_rate": [0.62, 0.67], "same_first_choice_rate": 0.28,
                     "uniform_random_router": {"shared_expert_rate": 13 / 28,
                                               "same_first_choice_rate": 0.125}}}
    with open(PATH, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", PATH, out)


if __name__ == "__main__":
    main()
