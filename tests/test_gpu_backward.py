"""Backward pass of the layer on the GPU (through the C ABI) against the fp64 backward oracle.

The oracle's gradients are pinned to central finite differences of the forward
definition (test_oracle_backward_pins.py). The GPU keeps u, v, h, g*dy and
du, dv in bf16 between its contractions (fp32 accumulation), so each gradient
is held to max|err| <= 2e-2 * max|ref| (BWD_TOL; measured 1.5e-3 to 4.2e-3); indices are exact and an
expert with no tokens must get exactly zero.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, make_config, make_layer, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import TOL, assert_status_ok, upload

pytestmark = pytest.mark.gpu

BWD_TOL = 2e-2
NAMES = ("dx", "dw_gate", "dw1", "dw3", "dw2")


@pytest.fixture(autouse=True)
def _reset_knobs():
    for k, v in ((moe.MOE_KNOB_FFN_PATH, 0), (moe.MOE_KNOB_GRID, 0), (moe.MOE_KNOB_TILE_CTAS, 0)):
        moe.moe_set_knob(k, v)
    moe.moe_get_device_status()
    yield
    for k, v in ((moe.MOE_KNOB_FFN_PATH, 0), (moe.MOE_KNOB_GRID, 0), (moe.MOE_KNOB_TILE_CTAS, 0)):
        moe.moe_set_knob(k, v)


def _margin_layer(T, d, ffn, seed):
    red = {}
    while True:
        L = make_layer(T, d, ffn, 8, "bf16", seed=seed, weight_seed=seed + 1000, redraws=sorted(red.items()))
        l = oracle.router_logits(to_f64(L.x), to_f64(L.w_gate))
        s = -np.sort(-l, axis=1)
        bad = np.nonzero((s[:, 0] - s[:, 1] < 1e-3) | (s[:, 1] - s[:, 2] < 1e-3))[0]
        if bad.size == 0:
            return L
        for t in bad:
            red[int(t)] = red.get(int(t), 0) + 1


def _dy(L, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((L.T, L.d), generator=g).to(torch.bfloat16)


def _gpu_grads(L, dev, dy, aux_coef):
    y, state = moe.layer_forward_train(dev["x"], dev["w_gate"], dev["w1"], dev["w3"], dev["w2"])
    g = moe.layer_backward(dev["x"], dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], dy.cuda(), state,
                           aux_coef=aux_coef)
    torch.cuda.synchronize()
    assert_status_ok()
    return y, dict(zip(NAMES, (t.float().cpu().numpy() for t in g)))


def _check(got, ref, names=NAMES):
    for n in names:
        r = ref[n]
        err = np.max(np.abs(got[n] - r)) if r.size else 0.0
        scale = np.max(np.abs(r)) if r.size else 1.0
        assert err <= BWD_TOL * scale, f"{n}: max error {err:.3e} > {BWD_TOL} * {scale:.3e}"


@pytest.mark.parametrize("T,d,ffn,aux", [(300, 512, 768, 0.0), (300, 512, 768, 0.5), (1000, 256, 256, 0.0),
                                         (40, 256, 512, 0.3), (1, 256, 256, 0.0)])
def test_backward_matches_oracle(T, d, ffn, aux):
    L = _margin_layer(T, d, ffn, seed=500 + T)
    dev = upload(L)
    dy = _dy(L, T)
    y, got = _gpu_grads(L, dev, dy, aux)
    ref = oracle.layer_backward(to_f64(L.x), to_f64(L.w_gate), to_f64(L.w1), to_f64(L.w3), to_f64(L.w2),
                                to_f64(dy), aux_coef=aux)
    _check(got, ref)
    # experts without tokens get exactly zero
    idx = ref["idx"]
    for e in set(range(8)) - set(np.unique(idx).tolist()):
        for n in ("dw1", "dw3", "dw2"):
            assert not got[n][e].any(), (n, e)
    # the training forward gives the forward's y bit for bit
    y_ref = moe.layer_forward(dev["x"], dev["w_gate"], dev["w1"], dev["w3"], dev["w2"])
    assert torch.equal(y, y_ref)


def test_backward_is_deterministic():
    L = _margin_layer(700, 256, 512, seed=31)
    dev = upload(L)
    dy = _dy(L, 3)
    _, a = _gpu_grads(L, dev, dy, 0.2)
    _, b = _gpu_grads(L, dev, dy, 0.2)
    for n in NAMES:
        assert np.array_equal(a[n], b[n]), n


def test_backward_with_empty_experts_and_skew():
    """Every token on experts (5, 3): six experts get zero gradients, one group holds all rows."""
    T = 260
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
    dy = _dy(L, 9)
    _, got = _gpu_grads(L, dev, dy, 0.1)
    ref = oracle.layer_backward(to_f64(L.x), to_f64(L.w_gate), to_f64(L.w1), to_f64(L.w3), to_f64(L.w2),
                                to_f64(dy), aux_coef=0.1)
    assert np.all(ref["idx"] == [5, 3])
    _check(got, ref)
    for e in (0, 1, 2, 4, 6, 7):
        for n in ("dw1", "dw3", "dw2"):
            assert not got[n][e].any()


def test_backward_mixtral_shape_sampled():
    """Prefill batch (T=4096) at the Mixtral shape: dx on sampled tokens, and sampled rows of one expert's
    weight gradients, against the oracle restricted to what those entries depend on."""
    L = make_config(2)
    dev = upload(L)
    dy = _dy(L, 2024)
    _, got = _gpu_grads(L, dev, dy, 0.0)
    X, Wg = to_f64(L.x), to_f64(L.w_gate)
    rng = np.random.default_rng(2)
    tok = np.sort(rng.choice(L.T, size=24, replace=False))
    # dx of a token depends only on that token when aux_coef = 0
    sub = oracle.layer_backward(X[tok], Wg, to_f64(L.w1), to_f64(L.w3), to_f64(L.w2), to_f64(dy)[tok])
    dx_ref = sub["dx"]
    assert np.max(np.abs(got["dx"][tok] - dx_ref)) <= BWD_TOL * np.max(np.abs(dx_ref))
    # one expert's gradients need all of its tokens: expert 6, sampled rows
    l = oracle.router_logits(X, Wg)
    idx, g, _ = oracle.top_k_gates(l, 2)
    e = 6
    sel_t, sel_j = np.nonzero(idx == e)
    Xe = X[sel_t]
    W1, W3, W2 = (to_f64(w[e]) for w in (L.w1, L.w3, L.w2))
    u, v = Xe @ W1.T, Xe @ W3.T
    s = 1.0 / (1.0 + np.exp(-u))
    h = u * s * v
    do = g[sel_t, sel_j][:, None] * to_f64(dy)[sel_t]
    rows_d = rng.choice(L.d, size=16, replace=False)
    rows_f = rng.choice(L.ffn, size=16, replace=False)
    dw2_ref = do[:, rows_d].T @ h
    dh = do @ W2
    du = dh * v * oracle.silu_grad(u)
    dv = dh * u * s
    dw1_ref = du[:, rows_f].T @ Xe
    dw3_ref = dv[:, rows_f].T @ Xe
    for name, gotv, refv in (("dw2", got["dw2"][e][rows_d], dw2_ref), ("dw1", got["dw1"][e][rows_f], dw1_ref),
                             ("dw3", got["dw3"][e][rows_f], dw3_ref)):
        err = np.max(np.abs(gotv - refv))
        assert err <= BWD_TOL * np.max(np.abs(refv)), (name, err, np.max(np.abs(refv)))
