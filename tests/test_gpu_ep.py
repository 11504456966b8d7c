"""Expert parallelism on one GPU: N ranks' worth of the layer through the library's kernels.

`ep.emulate` keeps every rank's grouped rows in one device buffer, so dispatch
and return are row gathers; each rank runs moe_expert_ffn on its share of the
experts. Every rank's output must be the single-GPU layer's on its tokens.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import make_layer, to_f64
from sparse_mixture_experts_53_b300 import ep, moe

from gpu_harness import TOL, assert_status_ok

pytestmark = pytest.mark.gpu


class _pinned_tiles:
    """Token-tile expert GEMMs on single CTAs (1) or CTA pairs (2) for every row count."""

    def __init__(self, ctas):
        self.ctas = ctas

    def __enter__(self):
        moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 1)
        moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, self.ctas)

    def __exit__(self, *exc):
        moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 0)
        moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 0)


def _margin_tokens(T, d, seed, wg, skew=None):
    """Token rows with the 1e-3 router margin for the given router weights."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, d), generator=g)
    if skew is not None:
        x = x + skew
    x = x.to(torch.bfloat16)
    while True:
        l = oracle.router_logits(to_f64(x), to_f64(wg))
        s = -np.sort(-l, axis=1)
        bad = np.nonzero((s[:, 0] - s[:, 1] < 1e-3) | (s[:, 1] - s[:, 2] < 1e-3))[0]
        if bad.size == 0:
            return x
        x[torch.from_numpy(bad)] = torch.randn((bad.size, d), generator=g).to(torch.bfloat16)


def test_gather_rows_and_its_index_check():
    src = torch.randn((50, 64), device="cuda").to(torch.bfloat16)
    idx = torch.tensor([3, 0, 49, 7, 7], dtype=torch.int32, device="cuda")
    dst = torch.empty((5, 64), dtype=torch.bfloat16, device="cuda")
    moe.moe_gather_rows(src, idx, dst)
    torch.cuda.synchronize()
    assert torch.equal(dst, src[idx.long()])
    assert_status_ok()
    bad = torch.tensor([1, 50, -1], dtype=torch.int32, device="cuda")
    out = torch.full((3, 64), 1.0, dtype=torch.bfloat16, device="cuda")
    moe.moe_gather_rows(src, bad, out)
    code, _ = moe.moe_get_device_status()
    assert code == moe.MOE_ERR_DEVICE_CHECK
    assert torch.equal(out[0], src[1]) and not out[1:].float().any()


@pytest.mark.parametrize("E,T", [(1, 40), (2, 300), (4, 500), (4, 20)])
def test_expert_ffn_with_a_share_of_the_experts(E, T):
    L = make_layer(T, 256, 512, E, "bf16", seed=E * 100 + T)
    rng = np.random.default_rng(T)
    # top-2 routing gives an expert at most T of the 2T rows; the FFN relies on that bound
    counts = np.minimum(np.bincount(rng.integers(0, E, size=2 * T), minlength=E), T)
    off = np.concatenate([[0], np.cumsum(counts)])
    xp = L.x[rng.integers(0, T, size=2 * T)]
    pw = torch.rand(2 * T)
    s = moe.make_shape(T, 256, 512, moe.MOE_BF16, E=E)
    ys = torch.empty((2 * T, 256), device="cuda")
    moe.moe_expert_ffn(s, xp.cuda(), torch.from_numpy(off).int().cuda(), pw.cuda(), L.w1.cuda(), L.w3.cuda(),
                       L.w2.cuda(), ys, moe.workspace(s, ffn_only=True))
    torch.cuda.synchronize()
    assert_status_ok()
    ref = oracle.expert_ffn_slots(to_f64(xp), off, to_f64(pw), to_f64(L.w1), to_f64(L.w3), to_f64(L.w2))
    n = int(off[-1])  # rows past the last group are not written
    assert np.max(np.abs(ys.cpu().numpy()[:n] - ref[:n])) <= TOL["bf16"] * np.max(np.abs(ref[:n]))


@pytest.mark.parametrize("N,T,mode", [(2, 300, "contiguous"), (4, 300, "balanced"), (8, 200, "contiguous"),
                                      (4, 16, "contiguous"), (4, 300, "replicated"), (8, 200, "replicated")])
def test_emulated_ranks_equal_the_single_gpu_layer(N, T, mode):
    d, ffn = 512, 1024
    L = make_layer(N * T, d, ffn, 8, "bf16", seed=77 + N, weight_seed=88)
    xs = [_margin_tokens(T, d, 1000 * N + s, L.w_gate).cuda() for s in range(N)]
    dev = {k: getattr(L, k).cuda() for k in ("w_gate", "w1", "w3", "w2")}
    load = sum(np.bincount(oracle.top_k_gates(oracle.router_logits(to_f64(x.cpu()), to_f64(L.w_gate)), 2)[0].ravel(),
                           minlength=8) for x in xs)
    if mode == "replicated":
        # two hot experts' copies (a heavier load than these tokens'), so rows of one expert
        # from one source go to several ranks
        owner = ep.replicated_placement(np.array([900, 700, 50, 50, 50, 50, 50, 50]), N, 8 // N + 1)
        assert any(len(r) > 1 for r in owner)
    else:
        owner = ep.balanced_owners(load, N) if mode == "balanced" else ep.contiguous_owners(8, N)
    ys, plan, _ = ep.emulate(xs, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], owner)
    torch.cuda.synchronize()
    assert_status_ok()
    assert int(plan.rows_per_rank.sum()) == 2 * N * T
    for x, y in zip(xs, ys):
        ref = oracle.layer_forward(to_f64(x.cpu()), to_f64(L.w_gate), to_f64(L.w1), to_f64(L.w3), to_f64(L.w2))["y"]
        assert np.max(np.abs(y.float().cpu().numpy() - ref)) <= TOL["bf16"] * np.max(np.abs(ref))
    # Same rows, same weights, same K order: with the expert GEMM's kernel pinned (a rank's row
    # count would otherwise pick its own tile shape or split-K width), every rank's output equals
    # the single-GPU layer's bit for bit.
    for ctas in (1, 2):
        with _pinned_tiles(ctas):
            ys, _, _ = ep.emulate(xs, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], owner)
            for x, y in zip(xs, ys):
                single = moe.layer_forward(x, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"])
                torch.cuda.synchronize()
                assert_status_ok()
                assert torch.equal(y, single)


def test_skewed_routing_is_rebalanced_by_placement():
    d, ffn, N, T = 256, 512, 4, 256
    L = make_layer(N * T, d, ffn, 8, "bf16", seed=5, weight_seed=6)
    wg = L.w_gate.float()
    u = torch.randn(d, generator=torch.Generator().manual_seed(1))
    u = u / u.norm()
    wg[:2] += u / np.sqrt(d) * 40
    L.w_gate = wg.to(torch.bfloat16)
    xs = [_margin_tokens(T, d, s, L.w_gate, skew=1.5 * u).cuda() for s in range(N)]
    dev = {k: getattr(L, k).cuda() for k in ("w_gate", "w1", "w3", "w2")}
    _, p_c, _ = ep.emulate(xs, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], ep.contiguous_owners(8, N))
    load = p_c.counts.sum(0)
    ys, p_b, _ = ep.emulate(xs, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], ep.balanced_owners(load, N))
    assert_status_ok()
    assert load[:2].sum() > 0.4 * load.sum()  # the two steered experts are hot
    assert p_b.rows_per_rank.max() < p_c.rows_per_rank.max()
    # one more slot per rank: copies of the hot experts split their rows
    ys_r, p_r, _ = ep.emulate(xs, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"],
                              ep.replicated_placement(load, N, 8 // N + 1))
    assert_status_ok()
    assert p_r.rows_per_rank.max() < p_b.rows_per_rank.max()
    # the same rows through the same pinned kernel, split differently over the ranks: the same bits
    with _pinned_tiles(2):
        ys_b, _, _ = ep.emulate(xs, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], ep.balanced_owners(load, N))
        ys_r, _, _ = ep.emulate(xs, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"],
                                ep.replicated_placement(load, N, 8 // N + 1))
        torch.cuda.synchronize()
        assert_status_ok()
    for y_b, y_r in zip(ys_b, ys_r):
        assert torch.equal(y_b, y_r)
