"""The decode token stream with router locality (CPU).

``make_token_stream`` draws each sequence as a first-order autoregression of
N(0, 1) rows; tests/golden/locality_schedule.json stores the correlation rho at
which consecutive tokens' top-2 expert sets share an expert at the lecture
page's layer-15 rate (62 %, "Mixtral of Experts" lecture, router walkthrough).
"""
import json
from pathlib import Path

import numpy as np

import oracle
from moe_inputs import CONFIGS, make_token_stream, make_tokens, to_f64

SCHED = json.loads((Path(__file__).resolve().parent / "golden" / "locality_schedule.json").read_text())


def _rates(x, wg):
    S, B, d = x.shape
    idx, _, _ = oracle.top_k_gates(oracle.router_logits(to_f64(x.reshape(S * B, d)), to_f64(wg)), 2)
    idx = idx.reshape(S, B, 2)
    a, b = idx[:-1], idx[1:]
    return float((a[..., :, None] == b[..., None, :]).any(axis=(-1, -2)).mean()), float((a[..., 0] == b[..., 0]).mean())


def test_stream_rows_are_standard_normal_with_lag_one_correlation_rho():
    rho = 0.6
    x = make_token_stream(8, 400, 256, rho, seed=3, dtype="f32").numpy().astype(np.float64)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1.0) < 0.02
    lag1 = np.mean(x[1:] * x[:-1])
    assert abs(lag1 - rho) < 0.02
    # rho = 0: rows independent
    z = make_token_stream(8, 400, 256, 0.0, seed=3, dtype="f32").numpy().astype(np.float64)
    assert abs(np.mean(z[1:] * z[:-1])) < 0.01


def test_stored_rho_reproduces_the_pages_shared_expert_rate():
    c = CONFIGS[1]
    _, wg = make_tokens(1, c["d"], c["E"], c["dtype"], c["seed"])
    x = make_token_stream(64, 65, c["d"], SCHED["rho"], SCHED["seed"])
    shared, first = _rates(x, wg)
    assert abs(shared - 0.62) <= 0.01                       # lecture: 62 % at layer 15 (ArXiv)
    assert shared == SCHED["shared_expert_rate"] and first == SCHED["same_first_choice_rate"]
    assert first > 0.125                                    # above a uniform random router's 1/8


def test_independent_stream_matches_a_random_routers_rates():
    """With rho = 0 the router's choices of consecutive tokens are independent: two top-2 sets of a
    near-uniform router share an expert with probability 1 - C(6,2)/C(8,2) = 13/28 (the page's 46 %),
    and the first choices agree with probability 1/8."""
    c = CONFIGS[1]
    _, wg = make_tokens(1, c["d"], c["E"], c["dtype"], c["seed"])
    x = make_token_stream(64, 65, c["d"], 0.0, seed=99)
    shared, first = _rates(x, wg)
    n = 64 * 64
    assert abs(shared - 13 / 28) <= 4 * np.sqrt(0.25 / n) + 0.02
    assert abs(first - 1 / 8) <= 4 * np.sqrt(0.11 / n) + 0.01
