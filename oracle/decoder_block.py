"""Plain fp64 CPU oracle of one Mixtral decoder block around the MoE layer.

TEST INFRASTRUCTURE, like the rest of this package: only the tests,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` may use it. It
shares no code with the CUDA path. Every function computes in float64 from
inputs widened exactly from their stored type; numpy's ``@``, ``exp``, ``cos``
and ``sin`` are the library primitives.

Sources:

* "Mixtral" lineage page (tokentrails.org), step "GPT-2 vs Mixtral": Mixtral
  keeps LLaMA's normalisation, rotary positions and grouped-query attention
  and swaps only the MLP for the MoE layer; its Code gives the two residual
  branches, attention on the normalised input and then the MoE layer on the
  normalised result.
* "Mixtral of Experts" notes (royalroad.pages.dev), Proposed Method /
  Architecture: d = 4096, 32 attention heads, 8 KV heads, context 32768.
* "Mixtral of Experts" breakdown (fdeinterviews.com), layer diagram: 41.9M
  attention parameters per layer, which fixes the head width at d / 32 = 128
  and the K and V projections at 8 * 128 rows each.

Readings where the pages are silent:

* RMSNorm(x) = g * x / sqrt(mean(x^2) + eps) with a learned gain g per
  channel, no bias, eps = 1e-5 (the RMSNorm paper's form);
* RoPE as its paper defines it: channel pairs (2i, 2i+1) of every head are
  rotated by the angle pos * base^(-2i / head_dim), base 10000, pos the
  token's index inside its sequence (0 for the first token);
* attention scores q . k / sqrt(head_dim), causal (a query sees its own and
  earlier positions), no sliding window, no biases;
* grouped-query attention: query head h reads KV head h // (Hq / Hkv);
* the fused projection stores Wq, Wk and Wv one above the other,
  [(Hq + 2 Hkv) head_dim][d], nn.Linear convention; Wo is [d][Hq head_dim];
* a batch is B independent sequences of S tokens each, token-major [B S][d].

Parity status: every function here is pinned in tests/test_oracle_block_pins.py
by closed forms (constant vectors, rotations by known angles, single-key and
two-key attention, equal keys) and by invariants (causality, independence of
the sequences of a batch, the residual paths); the decode step is pinned
against the whole-sequence block (the last token of a sequence computed both
ways) and by a single-key closed form.
"""
from __future__ import annotations

import numpy as np

from .moe_oracle import layer_forward


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def rms_norm(x, g, eps: float = 1e-5) -> np.ndarray:
    """g * x / sqrt(mean over channels of x^2 + eps), row by row."""
    X = _f64(x)
    ms = np.mean(X * X, axis=-1, keepdims=True)
    return _f64(g) * X / np.sqrt(ms + eps)


def rope(x, pos, base: float = 10000.0) -> np.ndarray:
    """Rotary position embedding of x [..., heads, head_dim] at positions pos [...].

    Pair i = (x[2i], x[2i+1]) of every head turns by pos * base^(-2i/head_dim):
    (a, b) -> (a cos t - b sin t, a sin t + b cos t).
    """
    X = _f64(x)
    hd = X.shape[-1]
    if hd % 2:
        raise ValueError("head_dim must be even")
    i = np.arange(hd // 2, dtype=np.float64)
    theta = base ** (-2.0 * i / hd)
    t = _f64(pos)[..., None, None] * theta          # [..., 1, hd/2]
    a, b = X[..., 0::2], X[..., 1::2]
    out = np.empty_like(X)
    out[..., 0::2] = a * np.cos(t) - b * np.sin(t)
    out[..., 1::2] = a * np.sin(t) + b * np.cos(t)
    return out


def causal_gqa_attention(q, k, v) -> np.ndarray:
    """One sequence: q [S][Hq][hd], k and v [S][Hkv][hd] -> [S][Hq][hd].

    out[t, h] = sum_{j <= t} softmax_j(q[t,h] . k[j,g] / sqrt(hd)) v[j,g] with
    g = h // (Hq / Hkv).
    """
    Q, K, V = _f64(q), _f64(k), _f64(v)
    S, Hq, hd = Q.shape
    Hkv = K.shape[1]
    if Hq % Hkv:
        raise ValueError("query heads must be a multiple of the KV heads")
    group = Hq // Hkv
    out = np.zeros((S, Hq, hd), dtype=np.float64)
    future = np.triu(np.ones((S, S), dtype=bool), 1)   # key after the query
    for h in range(Hq):
        kv = h // group
        s = (Q[:, h, :] @ K[:, kv, :].T) / np.sqrt(hd)
        s[future] = -np.inf
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ V[:, kv, :]
    return out


def attention_sublayer(x, g_attn, wqkv, wo, seq_len: int, n_heads: int, n_kv_heads: int,
                       eps: float = 1e-5, base: float = 10000.0) -> dict:
    """h = x + Wo . attention(RoPE(Wq xn), RoPE(Wk xn), Wv xn), xn = RMSNorm(x).

    x is [B*S][d], B sequences of ``seq_len`` tokens. Returns the intermediates
    (xn, q, k, v after RoPE, attn [T][Hq*hd], o = attn Wo^T) and h.
    """
    X = _f64(x)
    T, d = X.shape
    if seq_len <= 0 or T % seq_len:
        raise ValueError("the tokens must split into sequences of seq_len")
    W = _f64(wqkv)
    hd = W.shape[0] // (n_heads + 2 * n_kv_heads)
    xn = rms_norm(X, g_attn, eps)
    qkv = xn @ W.T
    q = qkv[:, :n_heads * hd].reshape(T, n_heads, hd)
    k = qkv[:, n_heads * hd:(n_heads + n_kv_heads) * hd].reshape(T, n_kv_heads, hd)
    v = qkv[:, (n_heads + n_kv_heads) * hd:].reshape(T, n_kv_heads, hd)
    pos = np.arange(T) % seq_len
    q = rope(q, pos, base)
    k = rope(k, pos, base)
    attn = np.zeros((T, n_heads, hd), dtype=np.float64)
    for b in range(T // seq_len):
        r = slice(b * seq_len, (b + 1) * seq_len)
        attn[r] = causal_gqa_attention(q[r], k[r], v[r])
    attn = attn.reshape(T, n_heads * hd)
    o = attn @ _f64(wo).T
    return dict(xn=xn, q=q, k=k, v=v, attn=attn, o=o, h=X + o)


def decoder_block(x, p: dict, seq_len: int, n_heads: int, n_kv_heads: int, eps: float = 1e-5,
                  base: float = 10000.0, k: int = 2) -> dict:
    """out = h + MoE(RMSNorm(h)), h = x + attention(RMSNorm(x)) (lineage page, Code).

    ``p`` holds g_attn [d], wqkv, wo, g_ffn [d], w_gate, w1, w3, w2.
    """
    a = attention_sublayer(x, p["g_attn"], p["wqkv"], p["wo"], seq_len, n_heads, n_kv_heads, eps, base)
    hn = rms_norm(a["h"], p["g_ffn"], eps)
    m = layer_forward(hn, p["w_gate"], p["w1"], p["w3"], p["w2"], k)
    return dict(a, hn=hn, moe=m, out=a["h"] + m["y"])


def attention_one_query(q, k, v) -> np.ndarray:
    """One new token per sequence: q [Hq][hd] against keys k, v [n][Hkv][hd] (all
    positions up to and including the token's own) -> [Hq][hd]."""
    Q, K, V = _f64(q), _f64(k), _f64(v)
    Hq, hd = Q.shape
    group = Hq // K.shape[1]
    out = np.zeros((Hq, hd), dtype=np.float64)
    for h in range(Hq):
        s = K[:, h // group, :] @ Q[h] / np.sqrt(hd)
        w = np.exp(s - s.max())
        out[h] = (w / w.sum()) @ V[:, h // group, :]
    return out


def decoder_block_decode(x_new, k_prefix, v_prefix, p: dict, n_heads: int, n_kv_heads: int,
                         eps: float = 1e-5, base: float = 10000.0, k: int = 2) -> dict:
    """One decode step of the block for B sequences, one new token each.

    x_new [B][d]; k_prefix[b], v_prefix[b] [L_b][Hkv][hd] hold the keys (after
    RoPE) and values of the sequence's earlier tokens, so the new token sits at
    position L_b. Returns out [B][d] and the new token's k, v (to append).
    """
    X = _f64(x_new)
    B, d = X.shape
    W = _f64(p["wqkv"])
    hd = W.shape[0] // (n_heads + 2 * n_kv_heads)
    xn = rms_norm(X, p["g_attn"], eps)
    qkv = xn @ W.T
    attn = np.zeros((B, n_heads * hd), dtype=np.float64)
    k_new = np.zeros((B, n_kv_heads, hd))
    v_new = np.zeros((B, n_kv_heads, hd))
    for b in range(B):
        pos = np.array([len(k_prefix[b])])
        q = rope(qkv[b, :n_heads * hd].reshape(1, n_heads, hd), pos, base)[0]
        k_new[b] = rope(qkv[b, n_heads * hd:(n_heads + n_kv_heads) * hd].reshape(1, n_kv_heads, hd), pos, base)[0]
        v_new[b] = qkv[b, (n_heads + n_kv_heads) * hd:].reshape(n_kv_heads, hd)
        keys = np.concatenate([_f64(k_prefix[b]).reshape(-1, n_kv_heads, hd), k_new[b][None]])
        vals = np.concatenate([_f64(v_prefix[b]).reshape(-1, n_kv_heads, hd), v_new[b][None]])
        attn[b] = attention_one_query(q, keys, vals).reshape(-1)
    h = X + attn @ _f64(p["wo"]).T
    hn = rms_norm(h, p["g_ffn"], eps)
    m = layer_forward(hn, p["w_gate"], p["w1"], p["w3"], p["w2"], k)
    return dict(h=h, hn=hn, attn=attn, moe=m, out=h + m["y"], k_new=k_new, v_new=v_new)
