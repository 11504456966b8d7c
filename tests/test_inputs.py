"""Host tests of the seeded input generator and of the stored input schedule."""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import CONFIGS, load_schedule, make_config, make_layer, make_tokens, to_f64
from moe_inputs import gen


def test_draws_do_not_depend_on_thread_count(monkeypatch):
    n = 3 * gen.CHUNK + 17
    monkeypatch.setattr(gen, "_threads", lambda: 1)
    a = gen.normal_f32(9, 3, n, 0.5)
    monkeypatch.setattr(gen, "_threads", lambda: 5)
    b = gen.normal_f32(9, 3, n, 0.5)
    assert np.array_equal(a, b)
    assert abs(a.std() - 0.5) < 1e-3 and abs(a.mean()) < 1e-3


def test_layer_shapes_storage_and_scales():
    L = make_layer(300, 256, 512, 8, "bf16", seed=3, weight_seed=4)
    assert L.x.shape == (300, 256) and L.w_gate.shape == (8, 256)
    assert L.w1.shape == (8, 512, 256) and L.w3.shape == (8, 512, 256) and L.w2.shape == (8, 256, 512)
    assert all(t.dtype == torch.bfloat16 and t.is_contiguous() for t in (L.x, L.w_gate, L.w1, L.w3, L.w2))
    assert abs(float(L.w1.float().std()) - 1 / 16) < 2e-3
    assert abs(float(L.w2.float().std()) - 1 / np.sqrt(512)) < 2e-3
    assert abs(float(L.x.float().std()) - 1.0) < 2e-2
    # bf16 rounding is round-to-nearest-even of the float32 draw
    f = gen.normal_f32(3, gen.STREAM_X, 300 * 256, 1.0)
    assert torch.equal(torch.from_numpy(f).to(torch.bfloat16).view(300, 256), L.x)


def test_same_seed_same_tensors_and_weights_shared_by_seed():
    a = make_layer(20, 128, 256, 8, "f32", seed=1, weight_seed=7)
    b = make_layer(20, 128, 256, 8, "f32", seed=2, weight_seed=7)
    assert torch.equal(a.w1, b.w1) and torch.equal(a.w2, b.w2)
    assert not torch.equal(a.x, b.x)
    c = make_layer(20, 128, 256, 8, "f32", seed=1, weight_seed=7)
    assert torch.equal(a.x, c.x) and torch.equal(a.w_gate, c.w_gate)


def test_redraw_replaces_only_listed_rows():
    x0, wg0 = make_tokens(10, 128, 8, "bf16", 5)
    x1, wg1 = make_tokens(10, 128, 8, "bf16", 5, redraws=[(3, 1), (7, 2)])
    diff = [t for t in range(10) if not torch.equal(x0[t], x1[t])]
    assert diff == [3, 7] and torch.equal(wg0, wg1)


@pytest.mark.parametrize("k", sorted(CONFIGS))
def test_schedule_gives_router_margin(k):
    """Every token of every named workload has both top-2 gaps >= 1e-3."""
    c = CONFIGS[k]
    s = load_schedule()[str(k)]
    x, wg = make_tokens(c["T"], c["d"], c["E"], c["dtype"], s["seed"], s.get("skew_c"),
                        [tuple(r) for r in s["redraws"]])
    l = oracle.router_logits(to_f64(x), to_f64(wg))
    srt = -np.sort(-l, axis=1)
    assert np.min(srt[:, 0] - srt[:, 1]) >= 1e-3
    assert np.min(srt[:, 1] - srt[:, 2]) >= 1e-3
    idx, _, _ = oracle.top_k_gates(l, 2)
    shares = np.bincount(idx.ravel(), minlength=8) / idx.size
    np.testing.assert_allclose(shares, s["shares"], atol=1e-5)
    if c["skew"]:
        assert abs(shares[0] + shares[1] - 0.60) <= 0.01
        assert shares.min() < 0.02
    elif c["T"] >= 4096:
        assert np.all(np.abs(shares - 0.125) < 0.01)  # near-uniform routing


def test_make_config_tiny_is_complete():
    L = make_config(0)
    assert (L.T, L.d, L.ffn, L.E, L.dtype) == (64, 128, 256, 8, "f32")
    assert L.x.dtype == torch.float32
