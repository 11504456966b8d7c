"""Plain fp64 CPU oracle of the Mixtral top-2 sparse MoE feed-forward layer.

TEST INFRASTRUCTURE. This module is the slow, obviously-correct definition that
the CUDA path is checked against. Only the tests, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import it; the CUDA library and its
Python binding never do. It shares no code, table or helper with the CUDA path.

Every function computes in float64 from inputs widened exactly from their stored
type (bf16 or fp32). numpy's ``@`` (matrix product), ``exp``, ``argsort`` and
``cumsum`` are used as library primitives; there is no blocking, fusion or
reordering beyond the definitions cited below.

Sources (web pages about "Mixtral of Experts", arXiv 2401.04088):

* "Mixtral of Experts" lecture (ennepo.ai), the router walkthrough: the router
  is a linear layer giving one score per expert; a top-two mask sets the other
  six scores to -inf; a softmax over all eight then leaves two probabilities
  that sum to one; the output is the weighted sum of the two experts' outputs,
  and the other six experts are not touched.
* "Mixtral 8x7B" summary (flashpapers.ai), "How It Works": y = sum_i G(x)_i E_i(x)
  with G(x) = Softmax(TopK(x . W_g)), K = 2; an expert with G(x)_i = 0 is skipped.
* "Mixtral" lineage page (tokentrails.org), steps "The router"
  (g = softmax(top-2(x . W_g))), "Two experts per token"
  (y = g_a E_a(x) + g_b E_b(x); some experts get no tokens), "Load balancing"
  (L_aux = N . sum_i f_i P_i), and its code sketch (expert = w2(silu(w1 x) * w3 x);
  softmax over all 8, top-2, renormalise = softmax over the top 2).
* "Mixtral of Experts" breakdown (fdeinterviews.com), "The paper in one minute":
  each expert is a SwiGLU block; its layer diagram prints 176M parameters per
  expert and 41.9M attention parameters per layer.

Readings where the pages are silent:

* ties in the top-k go to the lower expert index, and the k selected slots are
  ordered by score, highest first;
* SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z)), the textbook definition;
* no biases, no capacity limit (every token gets exactly k experts);
* the expert-contiguous slot order (expert ascending, then token ascending) is
  this library's own data structure; the pages define no permutation;
* f_i = (slots routed to i) / (k T), P_i = mean over tokens of the full E-way
  softmax of the router scores, N = E.

Parity status: router, top-k gates, mixture, permutation and aux statistics are
pinned by brute force, closed forms and special cases in the tests; the expert
FFN is pinned by hand-computed tiny cases. Full-size layer outputs have no
printed worked example on the pages, so beyond those pins they are checked by
the definition only.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def router_logits(x, w_gate) -> np.ndarray:
    """Router scores l[t][e] = x_t . W_g[:, e] (lecture: 'one score per expert').

    ``w_gate`` is stored [E][d], so row e holds column e of the page's W_g.
    """
    return _f64(x) @ _f64(w_gate).T


def top_k_gates(logits, k: int = 2):
    """TopK mask followed by a softmax over all E scores.

    Lecture router walkthrough / flashpapers "How It Works": keep the k largest
    scores, set the others to -inf, softmax. Returns

    * ``idx``  [T][k] int64: selected experts, highest score first, equal scores
      in ascending expert index;
    * ``g``    [T][k] float64: their softmax weights;
    * ``G``    [T][E] float64: the dense gate vector G(x), exactly 0 off the top k.
    """
    l = _f64(logits)
    T, E = l.shape
    if not 1 <= k <= E:
        raise ValueError("k must be in [1, E]")
    # Stable sort of the negated scores: descending score, and among equal
    # scores the original (ascending) expert order is kept.
    order = np.argsort(-l, axis=1, kind="stable")
    idx = order[:, :k].astype(np.int64)
    rows = np.arange(T)[:, None]
    masked = np.full_like(l, -np.inf)
    masked[rows, idx] = l[rows, idx]
    if T == 0:
        return idx, np.zeros((0, k)), np.zeros((0, E))
    m = masked.max(axis=1, keepdims=True)
    p = np.exp(masked - m)  # exp(-inf) = 0 for the masked scores
    G = p / p.sum(axis=1, keepdims=True)
    g = G[rows, idx]
    return idx, g, G


def permute(idx, g, E: int) -> dict:
    """Expert-contiguous slot order (this library's own grouping structure).

    A slot is one (token t, choice j) pair. Slots are ordered by expert
    ascending, then token ascending. Returns counts[E], offsets[E+1] (exclusive
    prefix sum), perm_token[kT] (token of each row), slot_row[T][k] (row of slot
    (t, j)) and perm_w[kT] (gate weight of each row).
    """
    idx = np.asarray(idx, dtype=np.int64)
    g = _f64(g)
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for e in range(E):
        counts[e] = np.count_nonzero(idx == e)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    nxt = offsets[:-1].copy()
    slot_row = np.empty((T, k), dtype=np.int64)
    perm_token = np.empty(T * k, dtype=np.int64)
    perm_w = np.empty(T * k, dtype=np.float64)
    for t in range(T):  # visiting tokens in ascending order ranks them stably
        for j in range(k):
            e = idx[t, j]
            r = nxt[e]
            nxt[e] += 1
            slot_row[t, j] = r
            perm_token[r] = t
            perm_w[r] = g[t, j]
    return dict(counts=counts, offsets=offsets, perm_token=perm_token,
                slot_row=slot_row, perm_w=perm_w)


def silu(z) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z))."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_forward(x_rows, w1_e, w3_e, w2_e) -> np.ndarray:
    """One SwiGLU expert on a set of token rows: E(x) = W2 (SiLU(W1 x) * (W3 x)).

    Code sketch of the lineage page ('each expert is a SwiGLU MLP'); breakdown
    'The paper in one minute'. Weights are [out][in]: w1_e, w3_e [ffn][d],
    w2_e [d][ffn]. Returns [n][d].
    """
    X = _f64(x_rows)
    u = X @ _f64(w1_e).T
    v = X @ _f64(w3_e).T
    h = silu(u) * v
    return h @ _f64(w2_e).T


def expert_ffn_slots(x_perm, offsets, perm_w, w1, w3, w2) -> np.ndarray:
    """Scaled expert outputs in expert-contiguous order.

    y_slot[r] = perm_w[r] * E_e(x_perm[r]) for offsets[e] <= r < offsets[e+1].
    Experts with no rows are skipped ('six experts contribute nothing; their
    parameters are not touched').
    """
    xp = _f64(x_perm)
    offsets = np.asarray(offsets, dtype=np.int64)
    pw = _f64(perm_w)
    E = len(offsets) - 1
    y_slot = np.zeros((xp.shape[0], xp.shape[1]), dtype=np.float64)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y_slot[a:b] = pw[a:b, None] * expert_forward(xp[a:b], w1[e], w3[e], w2[e])
    return y_slot


def combine(y_slot, slot_row) -> np.ndarray:
    """y[t] = sum over j of y_slot[slot_row[t][j]], taken in choice order j = 0, 1, ..."""
    ys = _f64(y_slot)
    slot_row = np.asarray(slot_row, dtype=np.int64)
    T, k = slot_row.shape
    y = ys[slot_row[:, 0]].copy() if T else np.zeros((0, ys.shape[1]))
    for j in range(1, k):
        y = y + ys[slot_row[:, j]]
    return y


def layer_forward(x, w_gate, w1, w3, w2, k: int = 2) -> dict:
    """The MoE layer: y_t = sum_j g_tj E_{idx_tj}(x_t) (flashpapers 'How It Works';
    lineage step 'Two experts per token').

    Each expert runs only on the tokens that selected it; an expert that no
    token selected is never read. Returns y [T][d] with the router's logits,
    idx, g and dense G.
    """
    X = _f64(x)
    logits = router_logits(X, w_gate)
    idx, g, G = top_k_gates(logits, k)
    T, d = X.shape
    E = logits.shape[1]
    outs = np.zeros((T, k, d), dtype=np.float64)
    for e in range(E):
        sel_t, sel_j = np.nonzero(idx == e)
        if sel_t.size == 0:
            continue
        outs[sel_t, sel_j] = expert_forward(X[sel_t], w1[e], w3[e], w2[e])
    y = np.zeros((T, d), dtype=np.float64)
    for j in range(k):
        y = y + g[:, j, None] * outs[:, j]
    return dict(y=y, logits=logits, idx=idx, g=g, G=G)


def layer_forward_tokens(x, w_gate, w1, w3, w2, tokens, k: int = 2) -> np.ndarray:
    """``layer_forward`` restricted to the listed token rows (routing is per token)."""
    tokens = np.asarray(tokens, dtype=np.int64)
    return layer_forward(_f64(x)[tokens], w_gate, w1, w3, w2, k)["y"]


def aux_stats(logits, idx, E: int) -> dict:
    """Load-balancing statistics (lineage step 'Load balancing' and its code).

    f_i = share of the k*T slots routed to expert i, P_i = mean over tokens of
    the full E-way softmax of the router scores, L_aux = E * sum_i f_i P_i.
    """
    l = _f64(logits)
    idx = np.asarray(idx, dtype=np.int64)
    T, k = idx.shape
    f = np.array([np.count_nonzero(idx == i) for i in range(E)], dtype=np.float64) / (k * T)
    m = l.max(axis=1, keepdims=True)
    p = np.exp(l - m)
    p = p / p.sum(axis=1, keepdims=True)
    P = p.mean(axis=0)
    return dict(f=f, P=P, l_aux=float(E * np.sum(f * P)))


def mixtral_param_counts(d: int = 4096, ffn: int = 14336, E: int = 8, k: int = 2,
                         layers: int = 32, n_heads: int = 32, n_kv_heads: int = 8) -> dict:
    """Parameter accounting of the decoder stack without embeddings and norms.

    Shapes from the royalroad notes 'Architecture' and the lineage page's shape
    table: 32 layers, d=4096, 14336 per expert, 32 query / 8 KV heads, 8 experts,
    2 active. No biases.
    """
    head_dim = d // n_heads
    expert = 3 * d * ffn
    attention = d * (n_heads * head_dim) * 2 + d * (n_kv_heads * head_dim) * 2
    router = d * E
    stored = layers * (E * expert + attention + router)
    active = layers * (k * expert + attention + router)
    return dict(expert=expert, attention=attention, router=router,
                stored_wo_embed=stored, active_wo_embed=active,
                flops_per_slot=6 * d * ffn)
