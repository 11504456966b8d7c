"""CTA-pair token tiles with units claimed from a counter (MOE_KNOB_TILE_SCHED = 3: both projections).

Which pair computes a unit does not enter its arithmetic, so the claimed
schedule must give the same bits as the static one (pair p takes units p,
p + pairs, ...), on every shape, on repeated calls (the counters are zeroed
before each launch) and with serialised launches; the small shapes are also
checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import make_config, make_layer, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import assert_status_ok, check_y, check_y_slot, run_staged, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _pair_tiles():
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 1)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 2)
    moe.moe_get_device_status()
    yield
    for k, v in ((moe.MOE_KNOB_FFN_PATH, 0), (moe.MOE_KNOB_TILE_CTAS, 0), (moe.MOE_KNOB_TILE_SCHED, 0),
                 (moe.MOE_KNOB_GRID, 0), (moe.MOE_KNOB_PDL, 1)):
        moe.moe_set_knob(k, v)


def _margin_layer(T, d, ffn, seed):
    """A layer whose tokens keep a 1e-3 gap between their 2nd and 3rd router scores (and 1st and 2nd)."""
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


def _both(dev, calls=2):
    """y of the static schedule, then of each projection claiming its units and both, `calls` calls in a row."""
    moe.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, 0)
    ref = _forward(dev)
    outs = []
    for sched in (1, 2, 3):
        moe.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, sched)
        outs += [_forward(dev) for _ in range(calls)]
    assert_status_ok()
    return ref, outs


@pytest.mark.parametrize("T,d,ffn,grid", [
    (700, 256, 512, 6),       # 3 pairs: each claims many units, the ring wraps many times
    (700, 256, 512, 0),       # one pair per two SMs
    (3000, 512, 1024, 0),     # several row tiles per expert, ragged last tiles
    (300, 256, 256, 2),       # one pair does everything
])
def test_claimed_units_equal_static(T, d, ffn, grid):
    moe.moe_set_knob(moe.MOE_KNOB_GRID, grid)
    L = _margin_layer(T, d, ffn, seed=40 + T + grid)
    dev = upload(L)
    ref, outs = _both(dev)
    for y in outs:
        assert torch.equal(y, ref)
    check_y(L, ref.cpu())


def test_claimed_units_staged_and_serialised():
    """The staged expert FFN (the tile kernels alone on the stream) and launches without PDL."""
    L = _margin_layer(1500, 256, 512, seed=77)
    dev = upload(L)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, 0)
    ref = run_staged(L, dev)
    assert_status_ok()
    moe.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, 3)
    for pdl in (1, 0):
        moe.moe_set_knob(moe.MOE_KNOB_PDL, pdl)
        got = run_staged(L, dev)
        assert_status_ok()
        assert torch.equal(torch.as_tensor(got["y_slot"]), torch.as_tensor(ref["y_slot"]))
        assert torch.equal(torch.as_tensor(got["y"]), torch.as_tensor(ref["y"]))
    check_y_slot(L, ref)


def test_claimed_units_training_step():
    """The training forward (which also writes u and v from the up-projection epilogue) and the backward's
    four GEMMs (dh, dx and the weight gradients), each way."""
    L = make_layer(900, 256, 512, 8, "bf16", seed=91)
    dev = upload(L)
    g = torch.Generator().manual_seed(5)
    dy = torch.randn(dev["x"].shape, generator=g).to(torch.bfloat16).cuda()
    res = []
    for sched in (0, 3, 4, 7):
        moe.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, sched)
        y, state = moe.layer_forward_train(dev["x"], dev["w_gate"], dev["w1"], dev["w3"], dev["w2"])
        grads = moe.layer_backward(dev["x"], dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], dy, state)
        torch.cuda.synchronize()
        res.append((y, *grads))
    assert_status_ok()
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert torch.equal(a, b)


@pytest.mark.parametrize("k", [2, 3])
def test_claimed_units_named_workloads(k):
    """Mixtral shape, T = 4096 and 16384: bit-identical to the static schedule."""
    L = make_config(k)
    dev = upload(L)
    ref, outs = _both(dev, calls=2)
    for y in outs:
        assert torch.equal(y, ref)
