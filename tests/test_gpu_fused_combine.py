"""The combine fused into the CTA-pair down projection (MOE_KNOB_FUSE_COMBINE, the default).

The slot of a token in the higher-numbered of its two experts waits until the
unit holding the token's other slot has stored its y_slot row, adds it to its
own value and writes the token's row of y. Two fp32 operands add the same in
either order, so y must equal the separate combine pass bit for bit: on every
shape here (many units per pair, half tiles, an empty expert, all tokens on one
expert pair, units claimed from a counter, serialised launches, the largest
named batch), and it must match the oracle on the small ones.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import make_config, make_layer, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import assert_status_ok, check_y, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _pairs():
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 1)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 2)
    moe.moe_get_device_status()
    yield
    for k, v in ((moe.MOE_KNOB_FFN_PATH, 0), (moe.MOE_KNOB_TILE_CTAS, 0), (moe.MOE_KNOB_FUSE_COMBINE, 1),
                 (moe.MOE_KNOB_TILE_SCHED, 0), (moe.MOE_KNOB_GRID, 0), (moe.MOE_KNOB_PDL, 1)):
        moe.moe_set_knob(k, v)


def _margin_layer(T, d, ffn, seed):
    red = {}
    while True:
        L = make_layer(T, d, ffn, 8, "bf16", seed=seed, weight_seed=seed + 1000, redraws=sorted(red.items()))
        s = -np.sort(-oracle.router_logits(to_f64(L.x), to_f64(L.w_gate)), axis=1)
        bad = np.nonzero((s[:, 0] - s[:, 1] < 1e-3) | (s[:, 1] - s[:, 2] < 1e-3))[0]
        if bad.size == 0:
            return L
        for t in bad:
            red[int(t)] = red.get(int(t), 0) + 1


def _forward(dev):
    y = moe.layer_forward(dev["x"], dev["w_gate"], dev["w1"], dev["w3"], dev["w2"])
    torch.cuda.synchronize()
    return y


def _fused_and_separate(dev, calls=2):
    moe.moe_set_knob(moe.MOE_KNOB_FUSE_COMBINE, 0)
    ref = _forward(dev)
    moe.moe_set_knob(moe.MOE_KNOB_FUSE_COMBINE, 1)
    outs = [_forward(dev) for _ in range(calls)]
    assert_status_ok()
    return ref, outs


@pytest.mark.parametrize("T,d,ffn,grid", [
    (700, 256, 512, 6),       # 3 pairs, many units each: partners often in another pair's later work
    (1100, 256, 256, 0),      # groups of about 275 rows: last tiles of at most 128 rows run as half tiles
    (3000, 512, 1024, 0),     # several row tiles per expert, ragged last tiles
    (300, 256, 256, 2),       # one pair does everything in order
])
def test_fused_combine_equals_separate(T, d, ffn, grid):
    moe.moe_set_knob(moe.MOE_KNOB_GRID, grid)
    L = _margin_layer(T, d, ffn, seed=70 + T + grid)
    dev = upload(L)
    ref, outs = _fused_and_separate(dev)
    for y in outs:
        assert torch.equal(y, ref)
    check_y(L, ref.cpu())


def test_fused_combine_claimed_units_and_serialised_launches():
    L = _margin_layer(1500, 256, 512, seed=171)
    dev = upload(L)
    moe.moe_set_knob(moe.MOE_KNOB_FUSE_COMBINE, 0)
    ref = _forward(dev)
    moe.moe_set_knob(moe.MOE_KNOB_FUSE_COMBINE, 1)
    for sched, pdl in ((3, 1), (0, 0), (3, 0)):
        moe.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, sched)
        moe.moe_set_knob(moe.MOE_KNOB_PDL, pdl)
        assert torch.equal(_forward(dev), ref)
    assert_status_ok()


def test_fused_combine_empty_expert_and_one_expert_pair():
    """Every token picks experts (5, 3): six experts are empty and every finishing slot waits on expert 3."""
    T = 600
    L = make_layer(T, 256, 256, 8, "bf16", seed=5)
    x = L.x.float()
    x[:, 0] = 16.0
    L.x = x.to(torch.bfloat16)
    wg = L.w_gate.float()
    wg[:, 0] = 0.0
    wg[5, 0] = 1.0
    wg[3, 0] = 0.5
    L.w_gate = wg.to(torch.bfloat16)
    dev = upload(L)
    ref, outs = _fused_and_separate(dev)
    for y in outs:
        assert torch.equal(y, ref)


def test_fused_combine_largest_named_batch():
    """T = 16384 at the Mixtral shape: bit-identical to the separate combine."""
    L = make_config(3)
    dev = upload(L)
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 0)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 0)
    ref, outs = _fused_and_separate(dev, calls=2)
    for y in outs:
        assert torch.equal(y, ref)
