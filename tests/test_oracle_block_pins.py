"""Pins of the decoder-block oracle (oracle/decoder_block.py) without a GPU.

Each test ties an oracle function to something other than its own formula:
closed forms at special inputs (constant vectors, rotations by known angles,
one and two keys, keys that are all equal), invariants (causality, sequences of
a batch not mixing, the two residual paths), the attention parameter count
printed on the pages (tests/golden/mixtral_page_numbers.json) and the MoE layer
oracle, pinned on its own in test_oracle_pins.py.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# -------------------------------------------------------------- RMSNorm ---

def test_rms_norm_of_a_constant_vector():
    d, c, eps = 8, -3.0, 1e-5
    g = np.arange(1, d + 1, dtype=np.float64)
    out = oracle.rms_norm(np.full((1, d), c), g, eps)
    assert np.allclose(out[0], g * c / math.sqrt(c * c + eps), rtol=1e-15, atol=0)


def test_rms_norm_gives_unit_rms_and_ignores_scale_without_eps():
    x = _rng(1).standard_normal((5, 64))
    out = oracle.rms_norm(x, np.ones(64), eps=0.0)
    assert np.allclose(np.sqrt(np.mean(out ** 2, axis=1)), 1.0, rtol=1e-14)
    assert np.allclose(oracle.rms_norm(7.5 * x, np.ones(64), eps=0.0), out, rtol=1e-13)
    # the gain multiplies channel by channel
    g = _rng(2).standard_normal(64)
    assert np.allclose(oracle.rms_norm(x, g, eps=0.0), out * g, rtol=1e-13)


# ----------------------------------------------------------------- RoPE ---

def test_rope_turns_the_first_pair_by_the_position():
    # pair 0 turns by pos * base^0 = pos radians, whatever the base
    x = np.array([[[1.0, 0.0]]])
    out = oracle.rope(x, np.array([0.5]), base=123.0)
    assert np.allclose(out[0, 0], [math.cos(0.5), math.sin(0.5)], rtol=1e-15)
    # position 0 leaves every pair in place
    y = _rng(3).standard_normal((1, 4, 16))
    assert np.array_equal(oracle.rope(y, np.array([0]), 10000.0), y)


def test_rope_second_pair_angle():
    # head_dim 4, base 100: pair 1 turns by pos * 100^(-2/4) = pos / 10
    x = np.array([[[0.0, 0.0, 0.0, 1.0]]])
    out = oracle.rope(x, np.array([10.0]), base=100.0)
    assert np.allclose(out[0, 0], [0.0, 0.0, -math.sin(1.0), math.cos(1.0)], rtol=1e-14, atol=1e-15)


def test_rope_keeps_pair_norms_composes_and_depends_on_relative_position():
    r = _rng(4)
    q = r.standard_normal((3, 2, 8))
    k = r.standard_normal((3, 2, 8))
    pos = np.array([0.0, 5.0, 17.0])
    rq = oracle.rope(q, pos)
    n = lambda a: a[..., 0::2] ** 2 + a[..., 1::2] ** 2  # noqa: E731
    assert np.allclose(n(rq), n(q), rtol=1e-13)
    assert np.allclose(oracle.rope(oracle.rope(q, pos), pos + 3.0), oracle.rope(q, 2 * pos + 3.0), rtol=1e-12,
                       atol=1e-12)
    # <R(m) q, R(n) k> depends on m - n only
    a = np.sum(oracle.rope(q, np.array([4.0] * 3)) * oracle.rope(k, np.array([1.0] * 3)), axis=-1)
    b = np.sum(oracle.rope(q, np.array([13.0] * 3)) * oracle.rope(k, np.array([10.0] * 3)), axis=-1)
    assert np.allclose(a, b, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------ attention ---

def test_attention_first_query_returns_the_first_value_of_its_kv_head():
    r = _rng(5)
    q, k, v = r.standard_normal((6, 4, 8)), r.standard_normal((6, 2, 8)), r.standard_normal((6, 2, 8))
    out = oracle.causal_gqa_attention(q, k, v)
    for h in range(4):
        assert np.allclose(out[0, h], v[0, h // 2], rtol=1e-15)


def test_attention_with_equal_keys_is_the_running_mean_of_values():
    r = _rng(6)
    S = 7
    q, v = r.standard_normal((S, 4, 8)), r.standard_normal((S, 1, 8))
    k = np.tile(r.standard_normal((1, 1, 8)), (S, 1, 1))
    out = oracle.causal_gqa_attention(q, k, v)
    for t in range(S):
        assert np.allclose(out[t], v[:t + 1, 0].mean(axis=0), rtol=1e-13)


def test_attention_two_keys_closed_form_fixes_the_scale():
    # head_dim 4, so scores are divided by 2: s0 = 0, s1 = a * 2 / 2 = a
    a = 0.7
    q = np.zeros((2, 1, 4))
    q[1, 0, 0] = a
    k = np.zeros((2, 1, 4))
    k[1, 0, 0] = 2.0
    v = np.array([[[1.0, 2.0, 3.0, 4.0]], [[-1.0, 0.5, 0.0, 2.0]]])
    out = oracle.causal_gqa_attention(q, k, v)
    w1 = math.exp(a) / (1.0 + math.exp(a))
    assert np.allclose(out[1, 0], (1 - w1) * v[0, 0] + w1 * v[1, 0], rtol=1e-14)


def test_attention_follows_a_dominant_earlier_key():
    r = _rng(7)
    S, hd = 9, 16
    q = r.standard_normal((S, 1, hd))
    k = 0.01 * r.standard_normal((S, 1, hd))
    v = r.standard_normal((S, 1, hd))
    k[3, 0] = 40.0 * q[8, 0] / np.linalg.norm(q[8, 0])
    out = oracle.causal_gqa_attention(q, k, v)
    assert np.allclose(out[8, 0], v[3, 0], atol=1e-6)


def test_gqa_equals_attention_with_each_kv_head_repeated_for_its_query_group():
    r = _rng(8)
    q, k, v = r.standard_normal((5, 6, 4)), r.standard_normal((5, 2, 4)), r.standard_normal((5, 2, 4))
    a = oracle.causal_gqa_attention(q, k, v)
    b = oracle.causal_gqa_attention(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1))
    assert np.allclose(a, b, rtol=1e-14)


def test_attention_is_causal():
    r = _rng(9)
    q, k, v = r.standard_normal((10, 2, 8)), r.standard_normal((10, 1, 8)), r.standard_normal((10, 1, 8))
    a = oracle.causal_gqa_attention(q, k, v)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    for z in (q2, k2, v2):
        z[6:] = r.standard_normal(z[6:].shape)
    b = oracle.causal_gqa_attention(q2, k2, v2)
    assert np.array_equal(a[:6], b[:6]) and not np.allclose(a[6:], b[6:])


# ------------------------------------------------------- the sublayers ---

def test_attention_parameter_count_matches_the_page():
    pg = json.load(open(os.path.join(GOLDEN, "mixtral_page_numbers.json")))
    d, H, Hkv = pg["d_model"]["value"], pg["attention_heads"]["value"], pg["kv_heads"]["value"]
    hd = d // H
    wqkv_rows = (H + 2 * Hkv) * hd
    count = wqkv_rows * d + d * H * hd
    assert abs(count - pg["attention_params_per_layer"]["value"]) <= pg["attention_params_per_layer"]["rounding"]


def _small_block(seed, T, d=16, H=4, Hkv=2, hd=4, ffn=8, E=8):
    r = _rng(seed)
    p = dict(g_attn=1.0 + 0.1 * r.standard_normal(d),
             wqkv=r.standard_normal(((H + 2 * Hkv) * hd, d)) / math.sqrt(d),
             wo=r.standard_normal((d, H * hd)) / math.sqrt(H * hd),
             g_ffn=1.0 + 0.1 * r.standard_normal(d),
             w_gate=r.standard_normal((E, d)) / math.sqrt(d),
             w1=r.standard_normal((E, ffn, d)) / math.sqrt(d),
             w3=r.standard_normal((E, ffn, d)) / math.sqrt(d),
             w2=r.standard_normal((E, d, ffn)) / math.sqrt(ffn))
    return r.standard_normal((T, d)), p


def test_rope_rotates_queries_and_keys_but_not_values():
    # d = 2, one head of width 2 (angle of pair 0 = position). Every token has
    # rms 1 with first channel 1, so the query and key are the same at every
    # position and the score between positions t and j is s^2 cos(t - j) / sqrt(2);
    # the value reads the second channel, the token's sign.
    sgn = np.array([1.0, -1.0, -1.0, 1.0, 1.0, -1.0])
    x = np.stack([np.ones(6), sgn], axis=1)
    s = 1.3
    wqkv = np.array([[s, 0.0], [0.0, 0.0],     # q = (s, 0)
                     [s, 0.0], [0.0, 0.0],     # k = (s, 0)
                     [0.0, 1.0], [0.0, 0.0]])  # v = (sign, 0)
    wo = np.eye(2)
    a = oracle.attention_sublayer(x, np.ones(2), wqkv, wo, seq_len=6, n_heads=1, n_kv_heads=1, eps=0.0)
    for t in range(6):
        w = np.array([math.exp(s * s * math.cos(t - j) / math.sqrt(2.0)) for j in range(t + 1)])
        expect = float(np.dot(w, sgn[:t + 1]) / w.sum())
        assert abs(a["o"][t, 0] - expect) < 1e-13 and abs(a["o"][t, 1]) < 1e-15
    assert np.allclose(a["h"], x + a["o"], rtol=0, atol=0)


def test_sublayer_with_zero_keys_averages_unrotated_values():
    x, p = _small_block(10, 6)
    hd, H, Hkv = 4, 4, 2
    w = p["wqkv"].copy()
    w[H * hd:(H + Hkv) * hd] = 0.0
    a = oracle.attention_sublayer(x, p["g_attn"], w, p["wo"], 6, H, Hkv)
    xn = oracle.rms_norm(x, p["g_attn"])
    vals = (xn @ w[(H + Hkv) * hd:].T).reshape(6, Hkv, hd)
    for t in range(6):
        m = vals[:t + 1].mean(axis=0)                     # [Hkv][hd]
        attn = np.concatenate([m[h // 2] for h in range(H)])
        assert np.allclose(a["o"][t], p["wo"] @ attn, rtol=1e-12, atol=1e-14)


def test_sequences_of_a_batch_do_not_mix_and_positions_restart():
    x, p = _small_block(11, 12)
    both = oracle.decoder_block(x, p, seq_len=6, n_heads=4, n_kv_heads=2)
    for b in range(2):
        one = oracle.decoder_block(x[6 * b:6 * (b + 1)], p, seq_len=6, n_heads=4, n_kv_heads=2)
        assert np.allclose(both["out"][6 * b:6 * (b + 1)], one["out"], rtol=1e-13, atol=1e-13)
    # one 12-token sequence is a different computation
    long = oracle.decoder_block(x, p, seq_len=12, n_heads=4, n_kv_heads=2)
    assert np.allclose(long["out"][:6], both["out"][:6], rtol=1e-13)
    assert not np.allclose(long["out"][6:], both["out"][6:])


def test_block_residual_paths():
    x, p = _small_block(12, 8)
    q = dict(p, wo=np.zeros_like(p["wo"]), w2=np.zeros_like(p["w2"]))
    assert np.array_equal(oracle.decoder_block(x, q, 8, 4, 2)["out"], x)
    # with no attention output the block is x + MoE(RMSNorm(x))
    q = dict(p, wo=np.zeros_like(p["wo"]))
    ref = x + oracle.layer_forward(oracle.rms_norm(x, p["g_ffn"]), p["w_gate"], p["w1"], p["w3"], p["w2"])["y"]
    assert np.allclose(oracle.decoder_block(x, q, 8, 4, 2)["out"], ref, rtol=1e-14, atol=1e-14)


def test_block_is_causal():
    x, p = _small_block(13, 10)
    a = oracle.decoder_block(x, p, 10, 4, 2)["out"]
    x2 = x.copy()
    x2[7:] += 1.0
    b = oracle.decoder_block(x2, p, 10, 4, 2)["out"]
    assert np.array_equal(a[:7], b[:7])


@pytest.mark.parametrize("bad", ["seq", "heads"])
def test_block_rejects_bad_shapes(bad):
    x, p = _small_block(14, 6)
    with pytest.raises(ValueError):
        if bad == "seq":
            oracle.attention_sublayer(x, p["g_attn"], p["wqkv"], p["wo"], 4, 4, 2)
        else:
            oracle.causal_gqa_attention(np.zeros((2, 3, 4)), np.zeros((2, 2, 4)), np.zeros((2, 2, 4)))


# ----------------------------------------------------------- decode step ---

def test_decode_step_equals_the_last_token_of_the_whole_sequence():
    # the prefix's keys and values come from the whole-sequence sublayer; the
    # decode step then recomputes the last token incrementally
    for L in (1, 5, 9):
        x, p = _small_block(20 + L, 2 * (L + 1))
        full = oracle.decoder_block(x, p, L + 1, 4, 2)
        kp = [full["k"][b * (L + 1):b * (L + 1) + L] for b in range(2)]
        vp = [full["v"][b * (L + 1):b * (L + 1) + L] for b in range(2)]
        step = oracle.decoder_block_decode(x[[L, 2 * L + 1]], kp, vp, p, 4, 2)
        assert np.allclose(step["out"], full["out"][[L, 2 * L + 1]], rtol=1e-12, atol=1e-12)
        assert np.allclose(step["k_new"], full["k"][[L, 2 * L + 1]], rtol=1e-12, atol=1e-12)


def test_decode_step_of_a_first_token_attends_to_itself_only():
    x, p = _small_block(30, 3)
    step = oracle.decoder_block_decode(x, [np.zeros((0, 2, 4))] * 3, [np.zeros((0, 2, 4))] * 3, p, 4, 2)
    # one key: the attention output is the token's own value, per KV head
    for b in range(3):
        v = step["v_new"][b]
        assert np.allclose(step["attn"][b].reshape(4, 4), v[[0, 0, 1, 1]], rtol=1e-14)


def test_one_query_attention_two_key_closed_form():
    q = np.zeros((1, 4))
    q[0, 0] = 0.9
    k = np.zeros((2, 1, 4))
    k[1, 0, 0] = 2.0
    v = np.array([[[1.0, 0.0, 0.0, 0.0]], [[0.0, 1.0, 0.0, 0.0]]])
    out = oracle.attention_one_query(q, k, v)
    w1 = math.exp(0.9) / (1 + math.exp(0.9))
    assert np.allclose(out[0], [1 - w1, w1, 0, 0], rtol=1e-14)


# ------------------------------------------- the pins catch planted bugs ---

import importlib  # noqa: E402

_db = importlib.import_module("oracle.decoder_block")  # the module (the package exports a function of that name)


def _plant(monkeypatch, name, fn):
    monkeypatch.setattr(_db, name, fn)
    monkeypatch.setattr(oracle, name, fn)


def test_pins_catch_kv_head_map_by_remainder(monkeypatch):
    orig = _db.causal_gqa_attention

    def bad(q, k, v):  # query head h reads KV head h % Hkv instead of h // (Hq / Hkv)
        g = q.shape[1] // k.shape[1]
        return orig(q, np.tile(k, (1, g, 1)), np.tile(v, (1, g, 1)))
    _plant(monkeypatch, "causal_gqa_attention", bad)
    with pytest.raises(AssertionError):
        test_attention_first_query_returns_the_first_value_of_its_kv_head()


def test_pins_catch_scale_one_over_head_dim(monkeypatch):
    orig = _db.causal_gqa_attention
    _plant(monkeypatch, "causal_gqa_attention", lambda q, k, v: orig(q / math.sqrt(q.shape[-1]), k, v))
    with pytest.raises(AssertionError):
        test_attention_two_keys_closed_form_fixes_the_scale()


def test_pins_catch_rotation_the_other_way(monkeypatch):
    orig = _db.rope
    _plant(monkeypatch, "rope", lambda x, pos, base=10000.0: orig(x, -np.asarray(pos, np.float64), base))
    with pytest.raises(AssertionError):
        test_rope_turns_the_first_pair_by_the_position()
    # turning q and k both the other way keeps every score (cos is even): only the direct pin sees it
    test_rope_rotates_queries_and_keys_but_not_values()


def test_pins_catch_rmsnorm_without_eps(monkeypatch):
    orig = _db.rms_norm
    _plant(monkeypatch, "rms_norm", lambda x, g, eps=1e-5: orig(x, g, 0.0))
    with pytest.raises(AssertionError):
        test_rms_norm_of_a_constant_vector()


def test_pins_catch_unrotated_keys_in_the_decode_step(monkeypatch):
    # a decode step that forgets to turn the new key: the last token no longer matches the whole sequence
    orig = _db.rope
    calls = {"n": 0}

    def bad(x, pos, base=10000.0):
        calls["n"] += 1
        return orig(x, pos, base) if calls["n"] % 2 == 1 else np.asarray(x, np.float64)  # q turned, k not
    x, p = _small_block(40, 8)
    full = oracle.decoder_block(x, p, 4, 4, 2)
    kp = [full["k"][b * 4:b * 4 + 3] for b in range(2)]
    vp = [full["v"][b * 4:b * 4 + 3] for b in range(2)]
    monkeypatch.setattr(_db, "rope", bad)
    step = oracle.decoder_block_decode(x[[3, 7]], kp, vp, p, 4, 2)
    assert not np.allclose(step["out"], full["out"][[3, 7]], rtol=1e-12, atol=1e-12)
