"""The router on the tensor cores (MOE_KNOB_ROUTER_TC, bf16 batches above 256 tokens).

The scores of a 128-token tile are one tcgen05 product with W_g, so the sums
run in the hardware's order: the scores are held to the tensor-core bound of
gpu_harness.logit_bound, the choices to the oracle's exactly (every token of
these batches keeps a 1e-3 gap around its second score), and both agree with
the CUDA-core router's choices. Ragged batches (T not a multiple of 128) and
the largest named batch are covered.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import make_config, make_layer, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import assert_status_ok, check_router, logit_bound, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _router_default():
    moe.moe_get_device_status()
    yield
    moe.moe_set_knob(moe.MOE_KNOB_ROUTER_TC, 1)


def _margin_layer(T, d, seed):
    red = {}
    while True:
        L = make_layer(T, d, 256, 8, "bf16", seed=seed, weight_seed=seed + 1000, redraws=sorted(red.items()))
        s = -np.sort(-oracle.router_logits(to_f64(L.x), to_f64(L.w_gate)), axis=1)
        bad = np.nonzero((s[:, 0] - s[:, 1] < 1e-3) | (s[:, 1] - s[:, 2] < 1e-3))[0]
        if bad.size == 0:
            return L
        for t in bad:
            red[int(t)] = red.get(int(t), 0) + 1


def _route(dev, T):
    s = moe.shape_of(dev["x"], dev["w1"])
    out = dict(idx=torch.full((T, 2), -1, dtype=torch.int32, device="cuda"),
               w=torch.full((T, 2), -1.0, device="cuda"),
               logits=torch.full((T, 8), float("nan"), device="cuda"))
    moe.moe_route_top2(s, dev["x"], dev["w_gate"], out["idx"], out["w"], out["logits"])
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in out.items()}


@pytest.mark.parametrize("T,d", [(257, 256), (300, 512), (1000, 256), (4096, 1024), (5000, 4096)])
def test_tensor_core_router_matches_oracle_and_cuda_cores(T, d):
    L = _margin_layer(T, d, seed=T + d)
    dev = upload(L)
    got = {}
    for tc in (1, 0):
        moe.moe_set_knob(moe.MOE_KNOB_ROUTER_TC, tc)
        got[tc] = _route(dev, T)
        assert_status_ok()
        check_router(L, got[tc], tc=bool(tc))
    assert torch.equal(got[0]["idx"], got[1]["idx"])
    # each score within the two bounds of each other
    x64, wg64 = to_f64(L.x), to_f64(L.w_gate)
    both = logit_bound(x64, wg64, d, tc=True) + logit_bound(x64, wg64, d, tc=False)
    diff = np.abs(got[1]["logits"].numpy().astype(np.float64) - got[0]["logits"].numpy())
    assert np.all(diff <= both)


def test_tensor_core_router_largest_named_batch():
    """T = 16384 at the Mixtral shape (128 tiles of 128 tokens): every token's choice is the oracle's."""
    L = make_config(3)
    dev = {"x": L.x.cuda(), "w_gate": L.w_gate.cuda(), "w1": torch.empty((8, 14336, 4096), dtype=torch.bfloat16,
                                                                            device="meta")}
    got = _route(dev, L.T)
    assert_status_ok()
    _, _, l_ref = check_router(L, got, tc=True)
    # The worst-case bound of the tensor-core sums (about 2e-3 here) exceeds half the 1e-3 gap that the
    # workloads keep around every token's second score, so the equal choices rest on the measured error:
    # it must stay far below that half gap.
    err = np.abs(got["logits"].numpy().astype(np.float64) - l_ref)
    assert err.max() <= 1e-4, f"largest score error {err.max():.3g}"
