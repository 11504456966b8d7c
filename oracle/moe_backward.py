"""Plain fp64 CPU oracle of the backward pass of the top-2 sparse MoE layer.

TEST INFRASTRUCTURE, under the same rules as ``moe_oracle``: only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may use it; it
shares no code with the CUDA path.

The pages train the router and the experts end to end and add the
load-balancing term to the loss (tokentrails.org "Mixtral", step "Load
balancing": L_aux = N . sum_i f_i P_i; "Mixtral of Experts" lecture, router
walkthrough: the router is a learned linear layer). They print no backward
pass, so this module is the chain rule applied to the forward definition in
``moe_oracle`` for the scalar

    L = sum_t <dy_t, y_t> + aux_coef * L_aux,

i.e. the gradients a caller receives for an upstream gradient dy. Readings
where the pages are silent:

* the top-k selection is piecewise constant: scores outside a token's top k
  get no gradient through the mixture, and the selection itself is not
  differentiated;
* f_i (a count of routed slots) is piecewise constant, so L_aux reaches the
  scores only through P_i;
* the k kept weights are the softmax of the k kept scores, whose Jacobian gives
  dl_j = g_j (dg_j - sum_i g_i dg_i) for the kept j (for k = 2:
  dl_a = -dl_b = g_a g_b (dg_a - dg_b));
* SiLU'(z) = s (1 + z (1 - s)) with s = sigmoid(z), from SiLU(z) = z s.

These are pinned in the tests by central finite differences of the forward
oracle on tiny layers, which use none of the formulas above.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import _f64, router_logits, top_k_gates


def _sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def silu_grad(z) -> np.ndarray:
    """d/dz [z sigmoid(z)] = s + z s (1 - s)."""
    z = _f64(z)
    s = _sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def topk_softmax_backward(g, dg) -> np.ndarray:
    """Scores' gradient through g = softmax(kept scores): dl_j = g_j (dg_j - sum_i g_i dg_i)."""
    g, dg = _f64(g), _f64(dg)
    return g * (dg - np.sum(g * dg, axis=1, keepdims=True))


def aux_score_grad(logits, idx, E: int) -> np.ndarray:
    """d L_aux / d l[t][j] = (E / T) p_tj (f_j - sum_i f_i p_ti), with f held fixed."""
    l = _f64(logits)
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    if T == 0:
        return np.zeros_like(l)
    f = np.array([np.count_nonzero(idx == i) for i in range(E)], dtype=np.float64) / (k * T)
    m = l.max(axis=1, keepdims=True)
    p = np.exp(l - m)
    p = p / p.sum(axis=1, keepdims=True)
    c = (p * f[None, :]).sum(axis=1, keepdims=True)
    return (E / T) * p * (f[None, :] - c)


def layer_backward(x, w_gate, w1, w3, w2, dy, aux_coef: float = 0.0, k: int = 2) -> dict:
    """Gradients of L = sum <dy, y> + aux_coef * L_aux with respect to x, W_g, W1, W3, W2.

    Weights are [out][in] as in the forward: w_gate [E][d], w1, w3 [E][ffn][d],
    w2 [E][d][ffn]. Returns dx [T][d], dw_gate [E][d], dw1, dw3 [E][ffn][d],
    dw2 [E][d][ffn], and the scores' gradient dl [T][E] and the kept weights'
    gradient dg [T][k].
    """
    X = _f64(x)
    dY = _f64(dy)
    Wg = _f64(w_gate)
    T, d = X.shape
    E = Wg.shape[0]
    logits = router_logits(X, Wg)
    idx, g, _ = top_k_gates(logits, k)
    dx = np.zeros((T, d))
    dw1 = np.zeros(np.shape(w1))
    dw3 = np.zeros(np.shape(w3))
    dw2 = np.zeros(np.shape(w2))
    dg = np.zeros((T, k))
    for e in range(E):
        sel_t, sel_j = np.nonzero(idx == e)
        if sel_t.size == 0:
            continue  # an expert no token selected gets no gradient
        W1, W3, W2 = _f64(w1[e]), _f64(w3[e]), _f64(w2[e])
        Xe = X[sel_t]
        u = Xe @ W1.T
        v = Xe @ W3.T
        s = _sigmoid(u)
        h = u * s * v
        o = h @ W2.T
        dg[sel_t, sel_j] = np.sum(dY[sel_t] * o, axis=1)
        do = g[sel_t, sel_j][:, None] * dY[sel_t]
        dw2[e] = do.T @ h
        dh = do @ W2
        du = dh * v * silu_grad(u)
        dv = dh * u * s
        dw1[e] = du.T @ Xe
        dw3[e] = dv.T @ Xe
        np.add.at(dx, sel_t, du @ W1 + dv @ W3)
    dl = np.zeros((T, E))
    dl_kept = topk_softmax_backward(g, dg)
    for j in range(k):
        np.add.at(dl, (np.arange(T), idx[:, j]), dl_kept[:, j])
    if aux_coef != 0.0:
        dl = dl + aux_coef * aux_score_grad(logits, idx, E)
    dw_gate = dl.T @ X
    dx = dx + dl @ Wg
    return dict(dx=dx, dw_gate=dw_gate, dw1=dw1, dw3=dw3, dw2=dw2, dl=dl, dg=dg, idx=idx, g=g)
