"""Write tests/golden/input_schedule.json: margin redraws and the skew constant.

The five named workloads draw their token rows from ``moe_inputs``. Two of the
recipe's steps need router decisions, which the input package must not compute,
so this script takes them once with the fp64 oracle and stores the outcome:

* Margin: a token whose sorted router scores s0 >= s1 >= s2 have
  s0 - s1 < 1e-3 or s1 - s2 < 1e-3 is redrawn (attempt 1, 2, ...) until both
  gaps are at least 1e-3. Gaps are measured on the stored (bf16 or fp32) values
  widened to fp64. The stored list is [token, final attempt].
* Skew (the T=8192 workload): x = z + c*u; c is bisected until experts 0 and 1
  hold 0.60 +/- 0.01 of the 2T slots, and the first seed in 5304, 5404, ...
  whose least-used expert holds under 2% of the slots is kept.

Usage: python tests/golden/make_input_schedule.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from moe_inputs import CONFIGS, make_tokens, to_f64  # noqa: E402
from moe_inputs.gen import SCHEDULE_PATH  # noqa: E402

MARGIN = 1e-3


def gaps(x, wg):
    l = oracle.router_logits(to_f64(x), to_f64(wg))
    s = -np.sort(-l, axis=1)
    return s[:, 0] - s[:, 1], s[:, 1] - s[:, 2]


def shares(x, wg, E):
    idx, _, _ = oracle.top_k_gates(oracle.router_logits(to_f64(x), to_f64(wg)), 2)
    return np.bincount(idx.ravel(), minlength=E) / idx.size


def margin_redraws(cfg, seed, skew_c):
    T, d, E, dt = cfg["T"], cfg["d"], cfg["E"], cfg["dtype"]
    attempt = {}
    while True:
        red = sorted(attempt.items())
        x, wg = make_tokens(T, d, E, dt, seed, skew_c, red)
        g1, g2 = gaps(x, wg)
        bad = np.nonzero((g1 < MARGIN) | (g2 < MARGIN))[0]
        if bad.size == 0:
            return [[int(t), int(a)] for t, a in red]
        for t in bad:
            attempt[int(t)] = attempt.get(int(t), 0) + 1


def calibrate_skew(cfg):
    T, d, E, dt = cfg["T"], cfg["d"], cfg["E"], cfg["dtype"]
    for trial in range(20):
        seed = cfg["seed"] + 100 * trial
        lo, hi = 0.0, 1024.0
        c = None
        for _ in range(40):
            mid = 0.5 * (lo + hi)
            x, wg = make_tokens(T, d, E, dt, seed, mid)
            sh = shares(x, wg, E)
            top = sh[0] + sh[1]
            if abs(top - 0.60) <= 0.005:
                c = mid
                break
            if top < 0.60:
                lo = mid
            else:
                hi = mid
        if c is None:
            continue
        if sh.min() < 0.02:
            return seed, c, sh
        print(f"seed {seed}: c={c:.3f} shares={np.round(sh, 4)} (min share not < 2%)")
    raise RuntimeError("no seed gave a starved expert")


def main():
    out = {"_about": __doc__.strip().splitlines()[0]}
    for k, cfg in CONFIGS.items():
        seed, skew_c = cfg["seed"], None
        entry = {}
        if cfg["skew"]:
            seed, skew_c, sh = calibrate_skew(cfg)
            entry["skew_c"] = skew_c
            entry["shares_before_redraw"] = [round(float(v), 5) for v in sh]
        red = margin_redraws(cfg, seed, skew_c)
        x, wg = make_tokens(cfg["T"], cfg["d"], cfg["E"], cfg["dtype"], seed, skew_c, red)
        g1, g2 = gaps(x, wg)
        sh = shares(x, wg, cfg["E"])
        entry.update(seed=seed, redraws=red, min_gap=float(min(g1.min(), g2.min())),
                     shares=[round(float(v), 5) for v in sh])
        out[str(k)] = entry
        print(k, cfg["name"], "seed", seed, "redrawn", len(red), "min gap", entry["min_gap"],
              "shares", entry["shares"])
    with open(SCHEDULE_PATH, "w") as f:
        json.dump(out, f, indent=1)
    print("wrote", SCHEDULE_PATH)


if __name__ == "__main__":
    main()
