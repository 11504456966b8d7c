"""Pins of the fp64 oracle against what the pages and mathematics fix (no GPU).

Each test ties one oracle function to something other than itself: brute force
on tiny inputs, closed forms, special cases that reduce to a plain softmax
mixture, hand-derived worked examples (tests/golden/hand_examples.json) and the
figures printed on the pages (tests/golden/mixtral_page_numbers.json).
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import moe_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _example_a():
    ex = _golden("hand_examples.json")["example_A"]
    arr = {k: np.array(ex[k], dtype=np.float64) for k in ("x", "w_gate", "w1", "w3", "w2")}
    return ex, arr


# ---------------------------------------------------------------- top-k ---

def _brute_force_topk(l, k):
    """Select by pairwise comparison: expert a beats b when (l_a, -a) > (l_b, -b)."""
    E = len(l)
    beats = lambda a, b: (l[a] > l[b]) or (l[a] == l[b] and a < b)  # noqa: E731
    winners = [S for S in itertools.combinations(range(E), k)
               if all(beats(s, e) for s in S for e in range(E) if e not in S)]
    assert len(winners) == 1
    S = list(winners[0])
    # order inside the set: highest first (ties: lower index first)
    ordered = []
    while S:
        best = [s for s in S if all(s == o or beats(s, o) for o in S)][0]
        ordered.append(best)
        S.remove(best)
    return ordered


@pytest.mark.parametrize("k", [1, 2, 3])
def test_topk_matches_brute_force_enumeration(k):
    rng = np.random.default_rng(11)
    # integer scores in a small range make exact ties common
    l_int = rng.integers(-3, 4, size=(3000, 8)).astype(np.float64)
    l_cont = rng.standard_normal((3000, 8))
    for l in (l_int, l_cont):
        idx, _, _ = oracle.top_k_gates(l, k)
        for t in range(l.shape[0]):
            assert list(idx[t]) == _brute_force_topk(l[t], k)


def test_topk_ties_go_to_lower_index():
    l = np.array([[1.0, 5.0, 5.0, 5.0, 0.0, 0.0, 0.0, 0.0],
                  [0.0] * 8,
                  [2.0, 1.0, 2.0, 1.0, 2.0, 1.0, 2.0, 1.0]])
    idx, g, _ = oracle.top_k_gates(l, 2)
    assert idx.tolist() == [[1, 2], [0, 1], [0, 2]]
    assert np.all(g == 0.5)


# ---------------------------------------------------------------- gates ---

def test_gates_closed_form_and_invariants():
    rng = np.random.default_rng(3)
    l = rng.standard_normal((5000, 8)) * 3
    idx, g, G = oracle.top_k_gates(l, 2)
    la = l[np.arange(len(l)), idx[:, 0]]
    lb = l[np.arange(len(l)), idx[:, 1]]
    sig = 1.0 / (1.0 + np.exp(lb - la))  # the two-way softmax is a logistic function of the gap
    np.testing.assert_allclose(g[:, 0], sig, rtol=0, atol=4e-16)
    np.testing.assert_allclose(g[:, 1], 1.0 - sig, rtol=0, atol=4e-16)
    assert np.all((g > 0) & (g < 1))
    assert np.all(g[:, 0] >= g[:, 1])
    np.testing.assert_allclose(g.sum(1), 1.0, rtol=0, atol=4.5e-16)
    # the other E - k entries of G(x) are exactly zero
    mask = np.ones_like(G, dtype=bool)
    mask[np.arange(len(l))[:, None], idx] = False
    assert np.all(G[mask] == 0.0)


def test_gates_equal_softmax_all_then_renormalise():
    """Lineage page code sketch: softmax over all 8, top-2, renormalise."""
    rng = np.random.default_rng(4)
    l = rng.standard_normal((2000, 8)) * 2
    idx, g, _ = oracle.top_k_gates(l, 2)
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    order = np.array([sorted(range(8), key=lambda e: (-p[t, e], e))[:2] for t in range(len(l))])
    w = p[np.arange(len(l))[:, None], order]
    w /= w.sum(1, keepdims=True)
    assert np.array_equal(order, idx)
    np.testing.assert_allclose(g, w, rtol=1e-14, atol=0)


# ------------------------------------------------------------ mixtures ---

def _rand_layer(rng, T=12, d=6, F=5, E=8):
    x = rng.standard_normal((T, d))
    wg = rng.standard_normal((E, d))
    w1 = rng.standard_normal((E, F, d)) / np.sqrt(d)
    w3 = rng.standard_normal((E, F, d)) / np.sqrt(d)
    w2 = rng.standard_normal((E, d, F)) / np.sqrt(F)
    return x, wg, w1, w3, w2


def _dense_expert(x, w1, w3, w2):
    u = w1 @ x
    v = w3 @ x
    return w2 @ (u * v / (1.0 + math.e ** (-u)))


def test_k_equals_E_is_the_dense_softmax_mixture():
    rng = np.random.default_rng(5)
    x, wg, w1, w3, w2 = _rand_layer(rng)
    out = oracle.layer_forward(x, wg, w1, w3, w2, k=8)
    for t in range(x.shape[0]):
        scores = [float(np.dot(x[t], wg[e])) for e in range(8)]
        z = [math.exp(s - max(scores)) for s in scores]
        sm = [v / sum(z) for v in z]
        ref = sum(sm[e] * _dense_expert(x[t], w1[e], w3[e], w2[e]) for e in range(8))
        np.testing.assert_allclose(out["y"][t], ref, rtol=1e-12, atol=1e-13)


def test_k1_is_the_selected_expert_alone():
    rng = np.random.default_rng(6)
    x, wg, w1, w3, w2 = _rand_layer(rng)
    out = oracle.layer_forward(x, wg, w1, w3, w2, k=1)
    assert np.all(out["g"] == 1.0)
    for t in range(x.shape[0]):
        a = int(np.argmax(x[t] @ wg.T))
        np.testing.assert_allclose(out["y"][t], _dense_expert(x[t], w1[a], w3[a], w2[a]),
                                   rtol=1e-13, atol=1e-14)


def test_top2_equals_dense_sum_with_zero_gates():
    rng = np.random.default_rng(7)
    x, wg, w1, w3, w2 = _rand_layer(rng)
    out = oracle.layer_forward(x, wg, w1, w3, w2, k=2)
    for t in range(x.shape[0]):
        ref = sum(out["G"][t, e] * _dense_expert(x[t], w1[e], w3[e], w2[e]) for e in range(8))
        np.testing.assert_allclose(out["y"][t], ref, rtol=1e-12, atol=1e-13)


def test_unselected_expert_weights_are_never_read():
    """Poisoning an expert that no token selects leaves y bit-identical."""
    rng = np.random.default_rng(8)
    x, wg, w1, w3, w2 = _rand_layer(rng, T=40)
    x[:, 0] = 10.0
    wg[5, 0] = -10.0  # expert 5 scores about -100 for every token
    base = oracle.layer_forward(x, wg, w1, w3, w2)
    assert not np.any(base["idx"] == 5)
    for w in (w1, w3, w2):
        w[5] = np.nan
    poisoned = oracle.layer_forward(x, wg, w1, w3, w2)
    assert np.array_equal(base["y"], poisoned["y"])
    assert np.all(np.isfinite(poisoned["y"]))


# -------------------------------------------------------------- experts ---

def test_silu_special_values():
    ln4 = math.log(4.0)
    v = oracle.silu(np.array([0.0, ln4, -ln4, math.log(9.0), 40.0, -40.0, -1000.0]))
    assert v[0] == 0.0
    assert v[1] == pytest.approx(0.8 * ln4, rel=1e-15)
    assert v[2] == pytest.approx(-0.2 * ln4, rel=1e-15)
    assert v[3] == pytest.approx(0.9 * math.log(9.0), rel=1e-15)
    assert v[4] == pytest.approx(40.0, rel=1e-16)
    assert v[5] == pytest.approx(-40.0 * math.exp(-40.0), rel=1e-14)
    assert v[6] == 0.0


def test_hand_example_top2():
    ex, a = _example_a()
    out = oracle.layer_forward(a["x"], a["w_gate"], a["w1"], a["w3"], a["w2"], k=2)
    exp = ex["expected"]
    assert out["idx"].tolist() == exp["idx"]
    np.testing.assert_allclose(out["g"], exp["g"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out["y"], exp["y"], rtol=1e-14, atol=1e-15)


def test_hand_example_top1():
    _, a = _example_a()
    exb = _golden("hand_examples.json")["example_B_top1"]
    out = oracle.layer_forward(a["x"], a["w_gate"], a["w1"], a["w3"], a["w2"], k=1)
    assert out["idx"].tolist() == exb["expected"]["idx"]
    np.testing.assert_allclose(out["y"], exb["expected"]["y"], rtol=1e-14, atol=1e-15)


def test_hand_example_through_the_permuted_path():
    """Router -> permutation -> scaled expert rows -> combine gives the same y."""
    ex, a = _example_a()
    l = oracle.router_logits(a["x"], a["w_gate"])
    idx, g, _ = oracle.top_k_gates(l, 2)
    p = oracle.permute(idx, g, 4)
    assert p["counts"].tolist() == ex["expected"]["counts"]
    x_perm = a["x"][p["perm_token"]]
    y_slot = oracle.expert_ffn_slots(x_perm, p["offsets"], p["perm_w"], a["w1"], a["w3"], a["w2"])
    y = oracle.combine(y_slot, p["slot_row"])
    np.testing.assert_allclose(y, ex["expected"]["y"], rtol=1e-14, atol=1e-15)
    aux = oracle.aux_stats(l, idx, 4)
    assert aux["l_aux"] == pytest.approx(ex["expected"]["l_aux"], rel=1e-15)


# ---------------------------------------------------------- permutation ---

@pytest.mark.parametrize("T", [0, 1, 7, 200])
def test_permutation_invariants_and_brute_force(T):
    rng = np.random.default_rng(T + 1)
    E = 8
    l = rng.standard_normal((T, E))
    l[:, 6] -= 100.0  # expert 6 never selected: an empty group
    idx, g, _ = oracle.top_k_gates(l, 2)
    p = oracle.permute(idx, g, E)
    counts, offsets = p["counts"], p["offsets"]
    assert counts.sum() == 2 * T and counts[6] == 0
    assert offsets[0] == 0 and np.array_equal(np.diff(offsets), counts)
    # brute force: sort the (expert, token, choice) triples
    triples = sorted((int(idx[t, j]), t, j) for t in range(T) for j in range(2))
    for r, (e, t, j) in enumerate(triples):
        assert p["perm_token"][r] == t
        assert p["slot_row"][t, j] == r
        assert p["perm_w"][r] == g[t, j]
        assert offsets[e] <= r < offsets[e + 1]
    # each token's two rows are distinct and map back to it
    if T:
        assert np.all(p["slot_row"][:, 0] != p["slot_row"][:, 1])
        assert np.array_equal(p["perm_token"][p["slot_row"][:, 0]], np.arange(T))


# ------------------------------------------------------------ aux stats ---

def test_aux_closed_forms():
    cf = _golden("hand_examples.json")["aux_closed_forms"]
    T = 64
    # uniform: every expert holds T/4 slots and all scores are equal
    idx = np.array([[(2 * t) % 8, (2 * t + 1) % 8] for t in range(T)])
    aux = oracle.aux_stats(np.zeros((T, 8)), idx, 8)
    np.testing.assert_allclose(aux["f"], cf["uniform"]["f"], rtol=0, atol=1e-16)
    np.testing.assert_allclose(aux["P"], cf["uniform"]["P"], rtol=0, atol=1e-16)
    assert aux["l_aux"] == pytest.approx(cf["uniform"]["l_aux"], rel=1e-15)
    # all slots on experts 0 and 1, probability split evenly between them
    l = np.full((T, 8), -1e4)
    l[:, :2] = 3.0
    idx = np.tile([0, 1], (T, 1))
    aux = oracle.aux_stats(l, idx, 8)
    np.testing.assert_allclose(aux["f"], cf["two_experts"]["f"], atol=1e-16)
    np.testing.assert_allclose(aux["P"], cf["two_experts"]["P"], atol=1e-16)
    assert aux["l_aux"] == pytest.approx(cf["two_experts"]["l_aux"], rel=1e-15)


def test_aux_brute_force_tiny():
    rng = np.random.default_rng(9)
    T, E = 5, 8
    l = rng.standard_normal((T, E))
    idx, _, _ = oracle.top_k_gates(l, 2)
    aux = oracle.aux_stats(l, idx, E)
    f = [0.0] * E
    for t in range(T):
        for j in range(2):
            f[int(idx[t, j])] += 1.0 / (2 * T)
    P = [0.0] * E
    for t in range(T):
        den = sum(math.exp(v) for v in l[t])
        for e in range(E):
            P[e] += math.exp(l[t, e]) / den / T
    np.testing.assert_allclose(aux["f"], f, rtol=1e-15)
    np.testing.assert_allclose(aux["P"], P, rtol=1e-13)
    assert aux["l_aux"] == pytest.approx(E * sum(a * b for a, b in zip(f, P)), rel=1e-13)


# ------------------------------------------------------- page figures ---

def test_parameter_counts_match_the_pages():
    pg = _golden("mixtral_page_numbers.json")
    pc = oracle.mixtral_param_counts(d=pg["d_model"]["value"], ffn=pg["ffn_per_expert"]["value"],
                                     E=pg["n_experts"]["value"], k=pg["top_k"]["value"],
                                     layers=pg["layers"]["value"], n_heads=pg["attention_heads"]["value"],
                                     n_kv_heads=pg["kv_heads"]["value"])
    assert pc["expert"] == 176_160_768
    assert abs(pc["expert"] - pg["params_per_expert"]["value"]) <= pg["params_per_expert"]["rounding"]
    assert abs(pc["attention"] - pg["attention_params_per_layer"]["value"]) <= pg["attention_params_per_layer"]["rounding"]
    # Embeddings are not given on the pages; they are shared by the stored and
    # the active count, so both leave the same remainder up to the printing.
    rest_stored = pg["params_stored"]["value"] - pc["stored_wo_embed"]
    rest_active = pg["params_active"]["value"] - pc["active_wo_embed"]
    tol = pg["params_stored"]["rounding"] + pg["params_active"]["rounding"]
    assert 0 < rest_stored < 0.5e9
    assert abs(rest_stored - rest_active) <= tol
    share = pg["n_experts"]["value"] * pg["layers"]["value"] * pc["expert"] / pg["params_stored"]["value"]
    assert abs(share - pg["expert_share_of_params"]["value"]) <= pg["expert_share_of_params"]["rounding"] + 0.01
    gib = pg["params_stored"]["value"] * 2 / 2**30
    assert abs(gib - pg["weights_gib_16bit"]["value"]) <= pg["weights_gib_16bit"]["rounding"]
    gflops = 2 * pg["params_active"]["value"] / 1e9
    assert abs(gflops - pg["gflops_per_token"]["value"]) <= pg["gflops_per_token"]["rounding"]
    assert pc["flops_per_slot"] == 2 * pc["expert"]


# ------------------------------------------- the pins catch planted bugs ---

def _planted(monkeypatch, name, fn):
    monkeypatch.setattr(moe_oracle, name, fn)


def test_pins_catch_swapped_w1_w3(monkeypatch):
    orig = moe_oracle.expert_forward
    _planted(monkeypatch, "expert_forward", lambda x, w1, w3, w2: orig(x, w3, w1, w2))
    with pytest.raises(AssertionError):
        test_hand_example_top2()


def test_pins_catch_ties_to_higher_index(monkeypatch):
    def bad(logits, k=2):
        l = np.asarray(logits, np.float64)
        rev = l[:, ::-1]
        idx, g, G = orig(rev, k)
        return (l.shape[1] - 1 - idx), g, G[:, ::-1]
    orig = moe_oracle.top_k_gates
    _planted(monkeypatch, "top_k_gates", bad)
    with pytest.raises(AssertionError):
        test_hand_example_top2()


def test_pins_catch_wrong_f_normalisation(monkeypatch):
    orig = moe_oracle.aux_stats

    def bad(logits, idx, E):
        r = orig(logits, idx, E)
        r["f"] = r["f"] * 2  # counts / T instead of counts / (2T)
        r["l_aux"] = float(E * np.sum(r["f"] * r["P"]))
        return r
    _planted(monkeypatch, "aux_stats", bad)
    monkeypatch.setattr(oracle, "aux_stats", bad)
    with pytest.raises(AssertionError):
        test_aux_closed_forms()


def test_pins_catch_sigmoid_in_place_of_silu(monkeypatch):
    _planted(monkeypatch, "silu", lambda z: 1.0 / (1.0 + np.exp(-np.asarray(z, np.float64))))
    with pytest.raises(AssertionError):
        test_hand_example_top2()
