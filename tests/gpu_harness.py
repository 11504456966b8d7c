"""Shared helpers of the GPU tests: upload a layer, run the ABI calls one by one
or as a whole, and compare with the oracle under the written tolerances."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from moe_inputs import to_f64
from sparse_mixture_experts_53_b300 import moe

# Written tolerances on y (and y_slot):
#   bf16 storage with fp32 accumulation: max|err| <= 2e-2 * max|y_ref|
#   fp32 storage (CUDA-core FFMA path):   max|err| <= 1e-5 * max|y_ref|
TOL = {"bf16": 2e-2, "f32": 1e-5}


def upload(layer, device="cuda"):
    return {k: getattr(layer, k).to(device).contiguous() for k in ("x", "w_gate", "w1", "w3", "w2")}


def shape_of(layer):
    code = moe.MOE_BF16 if layer.dtype == "bf16" else moe.MOE_F32
    return moe.make_shape(layer.T, layer.d, layer.ffn, code, E=layer.E)


def run_staged(layer, dev=None, stream=None):
    """Route -> permute -> expert FFN -> combine (+ aux) through the separate ABI calls."""
    dev = dev or upload(layer)
    s = shape_of(layer)
    T, d, E = layer.T, layer.d, layer.E
    c = "cuda"
    i32 = dict(dtype=torch.int32, device=c)
    f32 = dict(dtype=torch.float32, device=c)
    out = dict(
        idx=torch.full((T, 2), -7, **i32), w=torch.zeros((T, 2), **f32), logits=torch.zeros((T, E), **f32),
        counts=torch.zeros(E, **i32), offsets=torch.zeros(E + 1, **i32), perm_token=torch.full((2 * T,), -7, **i32),
        slot_row=torch.full((T, 2), -7, **i32), perm_w=torch.zeros(2 * T, **f32),
        x_perm=torch.zeros((2 * T, d), dtype=dev["x"].dtype, device=c), y_slot=torch.zeros((2 * T, d), **f32),
        y=torch.zeros((T, d), dtype=dev["x"].dtype, device=c),
        f=torch.zeros(E, **f32), P=torch.zeros(E, **f32), l_aux=torch.zeros(1, **f32))
    ws = moe.workspace(s, ffn_only=True)
    pws = torch.empty(max(16, moe.moe_permute_workspace_bytes(s)), dtype=torch.uint8, device=c)
    moe.moe_route_top2(s, dev["x"], dev["w_gate"], out["idx"], out["w"], out["logits"], stream)
    moe.moe_permute(s, out["idx"], out["w"], dev["x"], out["counts"], out["offsets"], out["perm_token"],
                    out["slot_row"], out["perm_w"], out["x_perm"], pws, stream)
    moe.moe_expert_ffn(s, out["x_perm"], out["offsets"], out["perm_w"], dev["w1"], dev["w3"], dev["w2"],
                       out["y_slot"], ws, stream)
    moe.moe_combine(s, out["y_slot"], out["slot_row"], out["y"], stream)
    moe.moe_aux_stats(s, out["logits"], out["counts"], out["f"], out["P"], out["l_aux"], stream)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in out.items()}


def run_forward(layer, dev=None, aux=False):
    dev = dev or upload(layer)
    res = moe.layer_forward(dev["x"], dev["w_gate"], dev["w1"], dev["w3"], dev["w2"], aux=aux)
    torch.cuda.synchronize()
    if aux:
        y, (f, P, l) = res
        return y.cpu(), (f.cpu(), P.cpu(), l.cpu())
    return res.cpu()


def assert_status_ok():
    code, detail = moe.moe_get_device_status()
    assert code == moe.MOE_OK, f"device status {moe.status_string(code)} (detail {detail})"


def logit_bound(x64, wg64, d, tc=False):
    """Worst-case fp32 error of the router's scores.

    CUDA cores: each lane sums d/32 products in order and a 5-level butterfly
    adds the 32 lane sums, so the error is at most (d/32 + 5) * 2^-24 *
    sum_j |x_j w_j| (products of stored values are exact in fp32 for bf16 inputs
    and rounded once for fp32 inputs).

    Tensor cores (bf16 batches above 256 tokens): d/16 MMA steps each add 16
    exact products to the fp32 accumulator. The order and the rounding inside a
    step are the hardware's, so each step is allowed an error of 2^-22 (twice
    the round-to-nearest unit: truncation when the addends are aligned) of the
    sum of magnitudes so far: at most (d/16 + 5) * 2^-22 * sum_j |x_j w_j|."""
    if tc:
        return (int(np.ceil(d / 16)) + 5) * 2.0 ** -22 * (np.abs(x64) @ np.abs(wg64).T)
    n = int(np.ceil(d / 32)) + 6
    return n * 2.0 ** -24 * (np.abs(x64) @ np.abs(wg64).T)


def router_on_tensor_cores(layer):
    """Whether the library's router ran on the tensor cores for this layer (MOE_KNOB_ROUTER_TC at its default)."""
    return layer.x.dtype == torch.bfloat16 and layer.T > 256 and layer.d % 64 == 0


def check_router(layer, got, tc=None):
    x64, wg64 = to_f64(layer.x), to_f64(layer.w_gate)
    l_ref = oracle.router_logits(x64, wg64)
    idx_ref, g_ref, _ = oracle.top_k_gates(l_ref, 2)
    assert np.array_equal(got["idx"].numpy(), idx_ref), "router indices differ from the oracle"
    bound = logit_bound(x64, wg64, layer.d, router_on_tensor_cores(layer) if tc is None else tc)
    err = np.abs(got["logits"].numpy().astype(np.float64) - l_ref)
    assert np.all(err <= bound + 1e-30), f"logit error {err.max()} above the fp32 bound"
    g = got["w"].numpy().astype(np.float64)
    # gate error: the sigmoid's slope is at most 1/4, plus a few fp32 roundings
    rows = np.arange(layer.T)
    gap_err = bound[rows, idx_ref[:, 0]] + bound[rows, idx_ref[:, 1]]
    assert np.all(np.abs(g - g_ref) <= 0.25 * gap_err[:, None] + 4 * 2.0 ** -24)
    assert np.all((g >= 0) & (g <= 1)) and np.all(g[:, 0] >= g[:, 1])
    assert np.all(np.abs(g.sum(1) - 1.0) <= 2.0 ** -22)
    return idx_ref, g_ref, l_ref


def check_permutation(layer, got, idx_ref):
    p = oracle.permute(idx_ref, got["w"].numpy(), layer.E)
    for k in ("counts", "offsets", "perm_token", "slot_row"):
        assert np.array_equal(got[k].numpy().astype(np.int64), p[k]), k
    # the gate weights travel unchanged; x rows are copied byte for byte
    r = np.arange(2 * layer.T)
    t = p["perm_token"]
    j = (p["slot_row"][t, 1] == r).astype(np.int64)
    assert np.array_equal(got["perm_w"].numpy(), got["w"].numpy()[t, j])
    assert torch.equal(got["x_perm"], layer.x[torch.from_numpy(p["perm_token"])])
    return p


def max_rel_err(got, ref):
    ref = np.asarray(ref, np.float64)
    got = np.asarray(got, np.float64)
    scale = np.max(np.abs(ref)) if ref.size else 1.0
    return float(np.max(np.abs(got - ref)) / scale) if ref.size else 0.0


_HOST_W = {}


def host_weights(layer):
    """float32 numpy views of the stored weights (exact), cached per layer object."""
    key = (id(layer.w1), id(layer.w3), id(layer.w2))
    if key not in _HOST_W:
        _HOST_W.clear()
        _HOST_W[key] = tuple(w.float().numpy() for w in (layer.w1, layer.w3, layer.w2))
    return _HOST_W[key]


def check_y_slot(layer, got, tol=None):
    tol = TOL[layer.dtype] if tol is None else tol
    ref = oracle.expert_ffn_slots(to_f64(got["x_perm"]), got["offsets"].numpy(),
                                  got["perm_w"].numpy().astype(np.float64), *host_weights(layer))
    err = max_rel_err(got["y_slot"].numpy(), ref)
    assert err <= tol, f"y_slot max error {err:.3e} > {tol:.1e} of max|ref|"
    return err


def check_y(layer, y, tokens=None, tol=None):
    tol = TOL[layer.dtype] if tol is None else tol
    if tokens is None:
        ref = oracle.layer_forward(to_f64(layer.x), to_f64(layer.w_gate), *host_weights(layer))["y"]
        got = to_f64(y)
    else:
        ref = oracle.layer_forward_tokens(to_f64(layer.x), to_f64(layer.w_gate), *host_weights(layer), tokens)
        got = to_f64(y[torch.as_tensor(tokens)])
    err = max_rel_err(got, ref)
    assert np.all(np.isfinite(got))
    assert err <= tol, f"y max error {err:.3e} > {tol:.1e} of max|y_ref|"
    return err
