"""Decode-time expert cache (weight-streaming path with part of each call's expert weights kept in L2).

The cache only changes the L2 priority of weight loads, never the arithmetic:
a decode loop over a token stream with router locality gives the same bits
with and without it, and matches the fp64 oracle step by step.
"""
import json
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, make_token_stream, make_tokens, make_weights, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import TOL, assert_status_ok

pytestmark = pytest.mark.gpu

SCHED = json.loads((Path(__file__).resolve().parent / "golden" / "locality_schedule.json").read_text())


def _loop(x, wg, w, keep_kb, B):
    """One moe_layer_forward per step on the first B rows of each step of x [S][Bmax][d]."""
    moe.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, keep_kb)
    try:
        ys = [moe.layer_forward(x[s, :B].contiguous(), wg, *w) for s in range(x.shape[0])]
        torch.cuda.synchronize()
    finally:
        moe.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, 0)
    assert_status_ok()
    return torch.stack(ys)


def _check_oracle(x, wg, w_host, ys, B):
    S, _, d = x.shape
    xx = x[:, :B].reshape(S * B, d).cpu()
    l = oracle.router_logits(to_f64(xx), to_f64(wg.cpu()))
    srt = -np.sort(-l, axis=1)
    ok = (srt[:, 0] - srt[:, 1] >= 1e-3) & (srt[:, 1] - srt[:, 2] >= 1e-3)   # tokens clear of near-ties
    assert ok.mean() > 0.9
    ref = oracle.layer_forward(to_f64(xx[ok]), to_f64(wg.cpu()), *(to_f64(t) for t in w_host))["y"]
    got = to_f64(ys.reshape(S * B, d).cpu()[ok])
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(got - ref)) <= TOL["bf16"] * np.max(np.abs(ref))


@pytest.mark.parametrize("B", [1, 2, 4])
def test_decode_loop_small_layer_same_bits_with_the_cache(B):
    d, F = 512, 1024
    w_host = make_weights(d, F, 8, "bf16", seed=41)
    _, wg = make_tokens(1, d, 8, "bf16", seed=42)
    w = tuple(t.cuda() for t in w_host)
    wg = wg.cuda()
    x = make_token_stream(4, 8, d, SCHED["rho"], seed=43).cuda()
    y0 = _loop(x, wg, w, 0, B)
    for keep_kb in (256, 4096, 131072):   # a few rows per expert, most of them, more than every expert holds
        assert torch.equal(_loop(x, wg, w, keep_kb, B), y0)
    _check_oracle(x, wg, w_host, y0, B)


def test_decode_loop_mixtral_shape_with_the_cache():
    c = CONFIGS[1]
    w_host = make_weights(c["d"], c["ffn"], c["E"], c["dtype"], c["weight_seed"])
    _, wg = make_tokens(1, c["d"], c["E"], c["dtype"], c["seed"])
    w = tuple(t.cuda() for t in w_host)
    wg = wg.cuda()
    x = make_token_stream(4, 3, c["d"], SCHED["rho"], SCHED["seed"]).cuda()
    y0 = _loop(x, wg, w, 0, 2)
    y1 = _loop(x, wg, w, 96 * 1024, 2)
    assert torch.equal(y0, y1)
    _check_oracle(x, wg, w_host, y1, 2)
