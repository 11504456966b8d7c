"""Pins of the fp64 backward oracle against central finite differences of the forward oracle.

The backward module applies the chain rule by hand; these checks differentiate
the forward definition numerically instead, so they share none of its
formulas. Tiny layers are drawn with a wide router margin so that no
perturbation changes which experts a token selects (the selection and the
routed counts f_i are piecewise constant).
"""
import numpy as np
import pytest

import oracle
import oracle.moe_backward as mb

EPS = 1e-5


def _tiny(seed, T=6, d=5, ffn=3, E=8, margin=0.05):
    rng = np.random.default_rng(seed)
    while True:
        x = rng.standard_normal((T, d))
        wg = rng.standard_normal((E, d)) / np.sqrt(d)
        l = x @ wg.T
        s = -np.sort(-l, axis=1)
        if np.all(s[:, 0] - s[:, 1] > margin) and np.all(s[:, 1] - s[:, 2] > margin):
            break
    w1 = rng.standard_normal((E, ffn, d)) / np.sqrt(d)
    w3 = rng.standard_normal((E, ffn, d)) / np.sqrt(d)
    w2 = rng.standard_normal((E, d, ffn)) / np.sqrt(ffn)
    dy = rng.standard_normal((T, d))
    return dict(x=x, w_gate=wg, w1=w1, w3=w3, w2=w2), dy


def _loss(p, dy, aux_coef, f_fixed):
    out = oracle.layer_forward(p["x"], p["w_gate"], p["w1"], p["w3"], p["w2"])
    L = float(np.sum(dy * out["y"]))
    if aux_coef:
        st = oracle.aux_stats(out["logits"], out["idx"], p["w_gate"].shape[0])
        assert np.array_equal(st["f"], f_fixed)  # the perturbation kept the routing
        L += aux_coef * st["l_aux"]
    return L


def _fd(p, dy, name, direction, aux_coef, f_fixed):
    hi = dict(p)
    lo = dict(p)
    hi[name] = p[name] + EPS * direction
    lo[name] = p[name] - EPS * direction
    return (_loss(hi, dy, aux_coef, f_fixed) - _loss(lo, dy, aux_coef, f_fixed)) / (2 * EPS)


GRAD = {"x": "dx", "w_gate": "dw_gate", "w1": "dw1", "w3": "dw3", "w2": "dw2"}


@pytest.mark.parametrize("seed", [1, 2, 3])
@pytest.mark.parametrize("aux_coef", [0.0, 0.7])
def test_directional_derivatives_match_finite_differences(seed, aux_coef):
    p, dy = _tiny(seed)
    g = oracle.layer_backward(p["x"], p["w_gate"], p["w1"], p["w3"], p["w2"], dy, aux_coef=aux_coef)
    out = oracle.layer_forward(p["x"], p["w_gate"], p["w1"], p["w3"], p["w2"])
    f_fixed = oracle.aux_stats(out["logits"], out["idx"], 8)["f"]
    rng = np.random.default_rng(100 + seed)
    for name, gname in GRAD.items():
        for _ in range(3):
            D = rng.standard_normal(p[name].shape)
            fd = _fd(p, dy, name, D, aux_coef, f_fixed)
            an = float(np.sum(g[gname] * D))
            assert abs(fd - an) <= 1e-7 * max(1.0, abs(fd)), (name, fd, an)


def test_every_entry_of_the_router_and_input_gradient():
    p, dy = _tiny(7, T=4, d=3, ffn=2)
    g = oracle.layer_backward(p["x"], p["w_gate"], p["w1"], p["w3"], p["w2"], dy, aux_coef=0.3)
    out = oracle.layer_forward(p["x"], p["w_gate"], p["w1"], p["w3"], p["w2"])
    f_fixed = oracle.aux_stats(out["logits"], out["idx"], 8)["f"]
    for name in ("x", "w_gate"):
        num = np.zeros_like(p[name])
        for i in np.ndindex(p[name].shape):
            D = np.zeros_like(p[name])
            D[i] = 1.0
            num[i] = _fd(p, dy, name, D, 0.3, f_fixed)
        np.testing.assert_allclose(g[GRAD[name]], num, rtol=0, atol=1e-8)


def test_silu_grad_matches_finite_differences():
    z = np.linspace(-12, 12, 241)
    num = (oracle.silu(z + EPS) - oracle.silu(z - EPS)) / (2 * EPS)
    np.testing.assert_allclose(oracle.silu_grad(z), num, rtol=0, atol=1e-9)
    assert oracle.silu_grad(0.0) == 0.5


def test_two_way_softmax_gradient_closed_form():
    rng = np.random.default_rng(5)
    la, lb = rng.standard_normal(50) + 1.0, rng.standard_normal(50) - 1.0
    ga = 1.0 / (1.0 + np.exp(lb - la))
    g = np.stack([ga, 1 - ga], axis=1)
    dg = rng.standard_normal((50, 2))
    dl = oracle.topk_softmax_backward(g, dg)
    closed = g[:, 0] * g[:, 1] * (dg[:, 0] - dg[:, 1])
    np.testing.assert_allclose(dl[:, 0], closed, rtol=0, atol=1e-15)
    np.testing.assert_allclose(dl[:, 1], -closed, rtol=0, atol=1e-15)
    # numerically: d/dla of ga*dga + gb*dgb
    f = lambda a, b: (1 / (1 + np.exp(b - a))) * dg[:, 0] + (1 - 1 / (1 + np.exp(b - a))) * dg[:, 1]
    num = (f(la + EPS, lb) - f(la - EPS, lb)) / (2 * EPS)
    np.testing.assert_allclose(dl[:, 0], num, rtol=0, atol=1e-9)


def test_aux_gradient_matches_finite_differences_and_sums_to_zero():
    rng = np.random.default_rng(9)
    l = rng.standard_normal((7, 8))
    idx, _, _ = oracle.top_k_gates(l, 2)
    grad = oracle.aux_score_grad(l, idx, 8)
    np.testing.assert_allclose(grad.sum(axis=1), 0.0, atol=1e-15)
    for t, j in [(0, 0), (3, 5), (6, 7)]:
        d = np.zeros_like(l)
        d[t, j] = EPS
        num = (oracle.aux_stats(l + d, idx, 8)["l_aux"] - oracle.aux_stats(l - d, idx, 8)["l_aux"]) / (2 * EPS)
        assert abs(num - grad[t, j]) < 1e-9


def test_structure_of_the_gradients():
    p, dy = _tiny(11, T=5)
    # steer every token to experts 2 and 6 so the other six get no rows
    p["w_gate"][[2, 6]] += 4.0 * np.sign(p["x"].sum(axis=0))
    p["x"] = np.abs(p["x"]) + 0.5
    p["w_gate"][[2, 6]] = np.abs(p["w_gate"][[2, 6]]) + np.array([[0.3], [0.0]])
    g = oracle.layer_backward(p["x"], p["w_gate"], p["w1"], p["w3"], p["w2"], dy)
    assert set(np.unique(g["idx"])) == {2, 6}
    for e in set(range(8)) - {2, 6}:
        assert not g["dw1"][e].any() and not g["dw3"][e].any() and not g["dw2"][e].any()
        assert not g["dl"][:, e].any()  # no aux term: only kept scores get gradient
    np.testing.assert_allclose(g["dl"].sum(axis=1), 0.0, atol=1e-14)


def test_planted_mistakes_are_caught(monkeypatch):
    """Each plausible slip in the backward module fails the finite-difference check."""
    p, dy = _tiny(3)
    out = oracle.layer_forward(p["x"], p["w_gate"], p["w1"], p["w3"], p["w2"])
    f_fixed = oracle.aux_stats(out["logits"], out["idx"], 8)["f"]
    D = {n: np.random.default_rng(4).standard_normal(p[n].shape) for n in GRAD}
    fd = {n: _fd(p, dy, n, D[n], 0.5, f_fixed) for n in GRAD}

    def mismatch():
        g = mb.layer_backward(p["x"], p["w_gate"], p["w1"], p["w3"], p["w2"], dy, aux_coef=0.5)
        return any(abs(float(np.sum(g[GRAD[n]] * D[n])) - fd[n]) > 1e-6 * max(1, abs(fd[n])) for n in GRAD)

    assert not mismatch()
    orig_aux = mb.aux_score_grad
    plants = {
        "silu_grad": lambda z: mb._sigmoid(np.asarray(z, dtype=np.float64)),  # SiLU' taken as sigmoid
        "topk_softmax_backward": lambda g, dg: g * dg,                         # Jacobian's second term dropped
        "aux_score_grad": lambda l, idx, E: -orig_aux(l, idx, E),              # wrong sign
    }
    for name, bad in plants.items():
        with monkeypatch.context() as m:
            m.setattr(mb, name, bad)
            assert mismatch(), name
