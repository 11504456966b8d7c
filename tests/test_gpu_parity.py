"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Router indices and the permutation must match bit for bit (the workloads carry a
1e-3 score margin, far above the fp32 error bound checked in gpu_harness);
outputs must be within 2e-2 * max|y_ref| for bf16 storage and 1e-5 * max|y_ref|
for fp32 storage.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import make_config, make_layer, make_weights, to_f64, CONFIGS
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import (TOL, assert_status_ok, check_permutation, check_router, check_y, check_y_slot,
                         run_forward, run_staged, upload)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_knobs():
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 0)
    moe.moe_set_knob(moe.MOE_KNOB_KSLICE, 0)
    moe.moe_set_knob(moe.MOE_KNOB_GRID, 0)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 0)
    moe.moe_get_device_status()
    yield
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 0)
    moe.moe_set_knob(moe.MOE_KNOB_KSLICE, 0)
    moe.moe_set_knob(moe.MOE_KNOB_GRID, 0)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 0)


def _margin_layer(T, d, ffn, dtype, seed, weights=None, E=8):
    """A custom-shape layer whose tokens carry the 1e-3 router margin."""
    red = {}
    while True:
        L = make_layer(T, d, ffn, E, dtype, seed=seed, weight_seed=seed + 1000,
                       redraws=sorted(red.items()), weights=weights)
        l = oracle.router_logits(to_f64(L.x), to_f64(L.w_gate))
        s = -np.sort(-l, axis=1)
        bad = np.nonzero((s[:, 0] - s[:, 1] < 1e-3) | (s[:, 1] - s[:, 2] < 1e-3))[0]
        if bad.size == 0:
            return L
        for t in bad:
            red[int(t)] = red.get(int(t), 0) + 1


# ------------------------------------------------------------------ tiny fp32

def test_tiny_fp32_config_staged_and_whole():
    L = make_config(0)
    got = run_staged(L)
    assert_status_ok()
    idx_ref, _, l_ref = check_router(L, got)
    check_permutation(L, got, idx_ref)
    check_y_slot(L, got)
    check_y(L, got["y"])
    y = run_forward(L)
    assert_status_ok()
    check_y(L, y)
    assert torch.equal(y, got["y"])  # same kernels, same order: bit-identical
    aux = oracle.aux_stats(l_ref, idx_ref, 8)
    np.testing.assert_allclose(got["f"].numpy(), aux["f"], rtol=0, atol=1e-7)
    np.testing.assert_allclose(got["P"].numpy(), aux["P"], rtol=0, atol=2e-6)
    assert abs(float(got["l_aux"][0]) - aux["l_aux"]) <= 1e-5 * aux["l_aux"]


@pytest.mark.parametrize("T,d,ffn", [(1, 128, 256), (37, 96, 160), (300, 128, 256)])
def test_fp32_odd_shapes(T, d, ffn):
    L = _margin_layer(T, d, ffn, "f32", seed=40 + T)
    got = run_staged(L)
    assert_status_ok()
    idx_ref, _, _ = check_router(L, got)
    check_permutation(L, got, idx_ref)
    check_y_slot(L, got)
    check_y(L, got["y"])


# ------------------------------------------------------------- bf16, small

SMALL_BF16 = [
    # (T, d, ffn): several 128-row tiles per expert with ragged tails, several
    # column tiles, and K loops of several stages
    (300, 512, 1024),
    (1000, 256, 384),
    (130, 768, 640),
    (700, 1024, 768),
]


@pytest.mark.parametrize("ctas", [2, 1])
@pytest.mark.parametrize("T,d,ffn", SMALL_BF16)
def test_bf16_token_tile_path(T, d, ffn, ctas):
    """Token tiles on CTA pairs (256-token tiles, one MMA across two SMs) and on single CTAs."""
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 1)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, ctas)
    L = _margin_layer(T, d, ffn, "bf16", seed=7 + T)
    got = run_staged(L)
    assert_status_ok()
    idx_ref, _, _ = check_router(L, got)
    check_permutation(L, got, idx_ref)
    check_y_slot(L, got)
    check_y(L, got["y"])


@pytest.mark.parametrize("T,d,ffn,kslice", [(16, 512, 1024, 0), (16, 512, 1024, 128), (5, 256, 384, 64),
                                            (64, 512, 512, 256), (1, 256, 128, 0), (33, 1024, 256, 0)])
def test_bf16_weight_streaming_path(T, d, ffn, kslice):
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 2)
    moe.moe_set_knob(moe.MOE_KNOB_KSLICE, kslice)
    L = _margin_layer(T, d, ffn, "bf16", seed=100 + T + kslice)
    got = run_staged(L)
    assert_status_ok()
    idx_ref, _, _ = check_router(L, got)
    check_permutation(L, got, idx_ref)
    check_y_slot(L, got)
    check_y(L, got["y"])


@pytest.mark.parametrize("T", [16, 48])
def test_both_bf16_paths_agree(T):
    L = _margin_layer(T, 512, 1024, "bf16", seed=900 + T)
    dev = upload(L)
    outs = []
    for path in (1, 2):
        moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, path)
        outs.append(run_staged(L, dev))
        assert_status_ok()
    # the two paths sum in different orders; both round h to bf16
    a, b = outs[0]["y_slot"].numpy(), outs[1]["y_slot"].numpy()
    assert np.max(np.abs(a - b)) <= 1e-2 * np.max(np.abs(a))
    for o in outs:
        check_y(L, o["y"])


def test_small_grid_many_tiles_per_cta():
    """Few CTAs: each runs many tiles, cycling all stages and both accumulators."""
    moe.moe_set_knob(moe.MOE_KNOB_GRID, 3)
    for path, T, ctas in ((1, 700, 2), (1, 700, 1), (2, 40, 1)):
        moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, path)
        moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, ctas)
        L = _margin_layer(T, 256, 512, "bf16", seed=300 + T)
        got = run_staged(L)
        assert_status_ok()
        check_y_slot(L, got)
        check_y(L, got["y"])


# ----------------------------------------------------------- edge cases

def test_empty_batch():
    L = make_layer(0, 256, 128, 8, "bf16", seed=1)
    dev = upload(L)
    y, (f, P, l) = moe.layer_forward(dev["x"], dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], aux=True)
    torch.cuda.synchronize()
    assert y.shape == (0, 256)
    assert float(l[0]) == 0.0 and torch.all(f == 0) and torch.all(P == 0)
    assert_status_ok()


@pytest.mark.parametrize("path", [1, 2])
def test_all_tokens_on_one_expert_pair(path):
    """Every token picks experts (5, 3): six experts are empty, one group holds all rows."""
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, path)
    T = 40 if path == 2 else 260
    L = make_layer(T, 256, 256, 8, "bf16", seed=5)
    x = L.x.float()
    x[:, 0] = 16.0
    L.x = x.to(torch.bfloat16)
    wg = L.w_gate.float()
    wg[:, 0] = 0.0
    wg[5, 0] = 1.0
    wg[3, 0] = 0.5
    L.w_gate = wg.to(torch.bfloat16)
    got = run_staged(L)
    assert_status_ok()
    assert np.all(got["idx"].numpy() == [5, 3])
    assert got["counts"].tolist() == [0, 0, 0, T, 0, T, 0, 0]
    check_y_slot(L, got)
    check_y(L, got["y"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_exact_ties_go_to_the_lower_index(dtype):
    """Duplicated router rows give bit-equal scores; the lower expert index wins."""
    L = make_layer(64, 256, 128, 8, dtype, seed=11)
    wg = L.w_gate.clone()
    wg[6] = wg[2]
    wg[7] = wg[2]
    L.w_gate = wg
    got = run_staged(L)
    assert_status_ok()
    idx = got["idx"].numpy()
    # 2, 6 and 7 always score the same: 7 can never win, and 2 first means 6 second
    assert not np.any(idx == 7)
    assert np.all(idx[idx[:, 0] == 2, 1] == 6)
    l = oracle.router_logits(to_f64(L.x), to_f64(L.w_gate))
    idx_ref, _, _ = oracle.top_k_gates(l, 2)
    assert np.array_equal(idx, idx_ref)


@pytest.mark.parametrize("path", [1, 2])
def test_poisoned_unselected_expert_is_never_read(path):
    """NaN weights of an expert with no tokens leave y bit-identical."""
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, path)
    T = 24 if path == 2 else 200
    L = make_layer(T, 256, 256, 8, "bf16", seed=21)
    x = L.x.float()
    x[:, 0] = 10.0
    L.x = x.to(torch.bfloat16)
    wg = L.w_gate.float()
    wg[4, 0] = -10.0
    L.w_gate = wg.to(torch.bfloat16)
    dev = upload(L)
    clean = run_forward(L, dev)
    assert_status_ok()
    for k in ("w1", "w3", "w2"):
        dev[k][4] = float("nan")
    poisoned = run_forward(L, dev)
    assert_status_ok()
    assert torch.isfinite(poisoned.float()).all()
    assert torch.equal(clean, poisoned)


def test_deterministic_repeat():
    L = _margin_layer(500, 256, 256, "bf16", seed=77)
    dev = upload(L)
    a = run_forward(L, dev)
    b = run_forward(L, dev)
    assert torch.equal(a, b)


def test_out_of_range_index_is_reported_not_written():
    L = make_layer(8, 256, 128, 8, "bf16", seed=3)
    dev = upload(L)
    s = moe.make_shape(8, 256, 128, moe.MOE_BF16)
    idx = torch.tensor([[0, 1]] * 7 + [[9, 2]], dtype=torch.int32, device="cuda")
    w = torch.full((8, 2), 0.5, device="cuda")
    counts = torch.zeros(8, dtype=torch.int32, device="cuda")
    offsets = torch.zeros(9, dtype=torch.int32, device="cuda")
    perm_token = torch.full((16,), -1, dtype=torch.int32, device="cuda")
    slot_row = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    perm_w = torch.zeros(16, device="cuda")
    x_perm = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(s, idx, w, dev["x"], counts, offsets, perm_token, slot_row, perm_w, x_perm)
    code, _ = moe.moe_get_device_status()
    assert code == moe.MOE_ERR_DEVICE_CHECK
    assert slot_row[7, 0].item() == -1 and int(offsets[8]) == 15
    assert_status_ok()  # the status word was cleared by the read


# ------------------------------------------------ the five named workloads

@pytest.fixture(scope="module")
def mixtral_weights():
    c = CONFIGS[1]
    return make_weights(c["d"], c["ffn"], c["E"], c["dtype"], c["weight_seed"])


@pytest.fixture(scope="module")
def mixtral_dev_weights(mixtral_weights):
    return tuple(w.cuda() for w in mixtral_weights)


def _sample_tokens(idx, T, n, seed):
    """n seeded tokens plus every token routed to the least-used non-empty expert."""
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(n, T), replace=False).tolist())
    counts = np.bincount(idx.ravel(), minlength=8)
    nz = np.nonzero(counts)[0]
    rare = nz[np.argmin(counts[nz])]
    pick |= set(np.nonzero((idx == rare).any(1))[0].tolist())
    return np.array(sorted(pick))


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_named_workload_full_size(k, mixtral_weights, mixtral_dev_weights):
    L = make_config(k, weights=mixtral_weights)
    dev = {"x": L.x.cuda(), "w_gate": L.w_gate.cuda()}
    dev["w1"], dev["w3"], dev["w2"] = mixtral_dev_weights
    got = run_staged(L, dev)
    assert_status_ok()
    idx_ref, _, l_ref = check_router(L, got)
    check_permutation(L, got, idx_ref)
    y, (f, P, l_aux) = run_forward(L, dev, aux=True)
    assert_status_ok()
    assert torch.equal(y, got["y"])
    tokens = np.arange(L.T) if L.T <= 64 else _sample_tokens(idx_ref, L.T, 192, seed=k)
    check_y(L, y, tokens)
    aux = oracle.aux_stats(l_ref, idx_ref, 8)
    np.testing.assert_allclose(f.numpy(), aux["f"], rtol=0, atol=1e-7)
    np.testing.assert_allclose(P.numpy(), aux["P"], rtol=0, atol=2e-5)
    assert abs(float(l_aux[0]) - aux["l_aux"]) <= 1e-4 * aux["l_aux"]
    if k == 4:
        counts = got["counts"].numpy()
        assert counts.min() == 0  # the skewed workload leaves one expert empty


@pytest.mark.parametrize("k", [2, 4])
def test_named_workload_every_token(k, mixtral_weights, mixtral_dev_weights):
    """The prefill batch (T = 4096) and the skewed batch (T = 8192, one expert empty) as the benchmark runs
    them (whole-layer call, automatic kernel choice): y of every token against the fp64 oracle, and the
    staged calls bit for bit equal to the whole layer."""
    L = make_config(k, weights=mixtral_weights)
    dev = {"x": L.x.cuda(), "w_gate": L.w_gate.cuda()}
    dev["w1"], dev["w3"], dev["w2"] = mixtral_dev_weights
    y = run_forward(L, dev)
    assert_status_ok()
    check_y(L, y)
    got = run_staged(L, dev)
    assert_status_ok()
    assert torch.equal(y, got["y"])


def test_largest_batch_mixtral_shape(mixtral_weights, mixtral_dev_weights):
    """T = 65536 (four times the largest named workload, 131072 slot rows): routing and grouping bit for bit
    on every token, y on sampled tokens, the load-balancing statistics."""
    T, d = 65536, 4096
    c = CONFIGS[3]
    from moe_inputs import make_tokens
    x, wg = make_tokens(T, d, 8, "bf16", seed=65536)
    # redraw the rows with a near tie (fp64 gaps below 1e-3) from a seeded stream
    g = torch.Generator().manual_seed(65536)
    while True:
        l = oracle.router_logits(to_f64(x), to_f64(wg))
        srt = -np.sort(-l, axis=1)
        bad = np.nonzero((srt[:, 0] - srt[:, 1] < 1e-3) | (srt[:, 1] - srt[:, 2] < 1e-3))[0]
        if bad.size == 0:
            break
        x[torch.from_numpy(bad)] = torch.randn((bad.size, d), generator=g).to(torch.bfloat16)
    w1, w3, w2 = mixtral_weights
    L = make_layer(1, d, c["ffn"], 8, "bf16", seed=1, weights=mixtral_weights)
    L.T, L.x, L.w_gate = T, x, wg
    dev = {"x": x.cuda(), "w_gate": wg.cuda()}
    dev["w1"], dev["w3"], dev["w2"] = mixtral_dev_weights
    got = run_staged(L, dev)
    assert_status_ok()
    idx_ref, _, l_ref = check_router(L, got)
    check_permutation(L, got, idx_ref)
    y, (f, P, l_aux) = run_forward(L, dev, aux=True)
    assert_status_ok()
    assert torch.equal(y, got["y"])
    check_y(L, y, _sample_tokens(idx_ref, T, 96, seed=65536))
    aux = oracle.aux_stats(l_ref, idx_ref, 8)
    np.testing.assert_allclose(f.numpy(), aux["f"], rtol=0, atol=1e-7)
    np.testing.assert_allclose(P.numpy(), aux["P"], rtol=0, atol=2e-5)


@pytest.mark.parametrize("T", [16, 300])
def test_pdl_on_and_off_give_identical_results(T):
    """Programmatic dependent launch only overlaps launch set-up: results are bit-identical."""
    L = _margin_layer(T, 512, 1024, "bf16", seed=1200 + T)
    dev = upload(L)
    outs = []
    for pdl in (0, 1):
        moe.moe_set_knob(moe.MOE_KNOB_PDL, pdl)
        try:
            outs.append(run_forward(L, dev))
            outs.append(run_staged(L, dev)["y"])
        finally:
            moe.moe_set_knob(moe.MOE_KNOB_PDL, 1)
        assert_status_ok()
    for o in outs[1:]:
        assert torch.equal(outs[0], o)
    check_y(L, outs[0])


def test_single_and_paired_token_tiles_agree():
    """Same sums in the same K order: the 1-CTA and CTA-pair tiles give the same y_slot up to rounding."""
    L = _margin_layer(600, 512, 1024, "bf16", seed=1300)
    dev = upload(L)
    moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 1)
    outs = []
    for ctas in (1, 2):
        moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, ctas)
        outs.append(run_staged(L, dev))
        assert_status_ok()
    a = outs[0]["y_slot"].numpy()
    assert np.max(np.abs(a - outs[1]["y_slot"].numpy())) <= 1e-3 * np.max(np.abs(a))


def _permute_outputs(s, idx, w, x, ws):
    T, d = x.shape
    c = "cuda"
    out = dict(counts=torch.full((8,), -5, dtype=torch.int32, device=c),
               offsets=torch.full((9,), -5, dtype=torch.int32, device=c),
               perm_token=torch.full((2 * T,), -5, dtype=torch.int32, device=c),
               slot_row=torch.full((T, 2), -5, dtype=torch.int32, device=c),
               perm_w=torch.full((2 * T,), -5.0, device=c),
               x_perm=torch.zeros((2 * T, d), dtype=x.dtype, device=c))
    moe.moe_permute(s, idx, w, x, out["counts"], out["offsets"], out["perm_token"], out["slot_row"],
                    out["perm_w"], out["x_perm"], ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T,dtype,bad", [(2048, "bf16", False), (5000, "bf16", False), (4500, "f32", False),
                                         (9000, "bf16", True)])
def test_many_cta_grouping_equals_single_cta(T, dtype, bad):
    """Per-chunk counts + ranks on many CTAs give the unique stable order of the one-CTA kernel."""
    d = 256 if dtype == "bf16" else 37  # 37 fp32 = 148-byte rows: the separate row gather
    L = make_layer(T, d, 128, 8, dtype, seed=T)
    x = L.x.cuda()
    s = moe.make_shape(T, d, 128, moe.MOE_BF16 if dtype == "bf16" else moe.MOE_F32)
    rng = np.random.default_rng(T)
    sel = np.stack([rng.choice(8, size=2, replace=False) for _ in range(T)]).astype(np.int32)
    # skew: expert 3 takes many slots, expert 6 none
    sel[: T // 3, 0] = 3
    sel[: T // 3, 1] = np.where(sel[: T // 3, 1] == 3, 5, sel[: T // 3, 1])
    sel[sel == 6] = 7
    sel[sel[:, 0] == sel[:, 1], 1] = 0
    sel[sel[:, 0] == sel[:, 1], 1] = 1
    if bad:
        sel[T // 2, 1] = 11
    idx = torch.from_numpy(sel).cuda()
    w = torch.rand((T, 2), device="cuda")
    ws = torch.empty(moe.moe_permute_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    one = _permute_outputs(s, idx, w, x, None)
    code_one, _ = moe.moe_get_device_status()
    many = _permute_outputs(s, idx, w, x, ws)
    code_many, _ = moe.moe_get_device_status()
    for k in one:
        assert torch.equal(one[k], many[k]), k
    if bad:
        assert code_one == code_many == moe.MOE_ERR_DEVICE_CHECK
        assert int(many["slot_row"][T // 2, 1]) == -1
    else:
        assert code_one == code_many == moe.MOE_OK
        assert int(many["counts"][6]) == 0
        ref = oracle.permute(sel.astype(np.int64), w.cpu().numpy(), 8)
        for k in ("counts", "offsets", "perm_token", "slot_row"):
            assert np.array_equal(many[k].cpu().numpy().astype(np.int64), ref[k]), k
        assert torch.equal(many["x_perm"].cpu(), L.x[torch.from_numpy(ref["perm_token"])])


@pytest.mark.parametrize("T,bad", [(1, False), (7, False), (64, False), (256, False), (100, True)])
def test_small_batch_grouping_matches_oracle(T, bad):
    """Slots ranked on every CTA of the small-batch grouping: the oracle's unique stable order, bit for bit."""
    d = 512
    L = make_layer(T, d, 128, 8, "bf16", seed=400 + T)
    x = L.x.cuda()
    s = moe.make_shape(T, d, 128, moe.MOE_BF16)
    rng = np.random.default_rng(T)
    sel = np.stack([rng.choice(8, size=2, replace=False) for _ in range(T)]).astype(np.int32)
    sel[sel == 6] = 7  # expert 6 empty
    sel[sel[:, 0] == sel[:, 1], 1] = 0
    sel[sel[:, 0] == sel[:, 1], 1] = 1
    if bad:
        sel[T // 3, 0] = -2
    idx = torch.from_numpy(sel).cuda()
    w = torch.rand((T, 2), device="cuda")
    out = _permute_outputs(s, idx, w, x, None)
    code, _ = moe.moe_get_device_status()
    ok = (sel >= 0) & (sel < 8)
    ref = oracle.permute(np.where(ok, sel, 0).astype(np.int64), w.cpu().numpy(), 8)
    if bad:
        assert code == moe.MOE_ERR_DEVICE_CHECK
        assert int(out["slot_row"][T // 3, 0]) == -1
        assert int(out["offsets"][8]) == 2 * T - 1
        return
    assert code == moe.MOE_OK
    for k in ("counts", "offsets", "perm_token", "slot_row"):
        assert np.array_equal(out[k].cpu().numpy().astype(np.int64), ref[k]), k
    assert np.array_equal(out["perm_w"].cpu().numpy(), ref["perm_w"].astype(np.float32))
    assert torch.equal(out["x_perm"].cpu(), L.x[torch.from_numpy(ref["perm_token"])])


def test_device_wait_timeout_is_reported_and_the_device_stays_usable():
    """A wait on a barrier nothing arrives on gives up after its limit and latches MOE_ERR_TIMEOUT."""
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_selftest_wait_timeout(20_000_000, flag)  # 20 ms
    code, detail = moe.moe_get_device_status()
    assert code == moe.MOE_ERR_TIMEOUT and detail == 1202
    assert int(flag) == 1
    assert_status_ok()  # the read cleared the word
    moe.moe_selftest_wait_timeout(5_000_000, flag)
    assert moe.moe_check_device_status() == moe.MOE_ERR_TIMEOUT
    assert moe.moe_check_device_status() == moe.MOE_OK
    # and the device still runs the layer
    L = _margin_layer(40, 256, 256, "bf16", seed=4)
    got = run_staged(L)
    assert_status_ok()
    check_y(L, got["y"])


def test_debug_mode_returns_device_errors_from_the_launching_call():
    """With the debug knob on, a device-side error comes back from the call that launched the kernel."""
    moe.moe_set_knob(moe.MOE_KNOB_DEBUG, 1)
    try:
        flag = torch.zeros(1, dtype=torch.int32, device="cuda")
        with pytest.raises(moe.MoEError) as e:
            moe.moe_selftest_wait_timeout(5_000_000, flag)
        assert e.value.code == moe.MOE_ERR_TIMEOUT
        assert moe.moe_check_device_status() == moe.MOE_ERR_TIMEOUT  # still latched until read
        src = torch.randn((8, 64), device="cuda").to(torch.bfloat16)
        bad = torch.tensor([0, 9], dtype=torch.int32, device="cuda")
        out = torch.empty((2, 64), dtype=torch.bfloat16, device="cuda")
        with pytest.raises(moe.MoEError) as e:
            moe.moe_gather_rows(src, bad, out)
        assert e.value.code == moe.MOE_ERR_DEVICE_CHECK
        assert moe.moe_check_device_status() == moe.MOE_ERR_DEVICE_CHECK
        # a clean call passes in debug mode too
        good = torch.tensor([3, 7], dtype=torch.int32, device="cuda")
        moe.moe_gather_rows(src, good, out)
        assert torch.equal(out, src[good.long()])
    finally:
        moe.moe_set_knob(moe.MOE_KNOB_DEBUG, 0)
    assert_status_ok()
