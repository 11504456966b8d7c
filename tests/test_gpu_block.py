"""The decoder block around the MoE layer on the GPU against the fp64 oracle.

Each step of the block (RMSNorm with and without the residual add, the linear
layers, RoPE, attention, the residual add) is checked through its own ABI call
on seeded inputs, then the whole block (moe_block_forward) on a small model and
on the Mixtral shape. Written tolerances:

* bf16 outputs carry one rounding (relative error <= 2^-9) on top of fp32
  arithmetic: RMSNorm and RoPE elements within 2^-7 of the reference scale;
* the linear layer's fp32 output: max|err| <= 1e-4 * max|ref| (fp32
  accumulation of exact bf16 products);
* attention: P and the output are rounded to bf16: max|err| <= 1e-2 * max|ref|;
  the first query of a sequence sees one key, so its output is that key's
  value exactly;
* the block: the same 2e-2 * max|ref| as the MoE layer. A token whose oracle
  router scores put the 2nd and 3rd expert within 0.05 of each other may be
  routed either way by a bf16 pipeline; for such a token either mixture is
  accepted (both are computed by the oracle).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from moe_inputs import BLOCK_CONFIGS, make_block, make_block_config, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import assert_status_ok

pytestmark = pytest.mark.gpu

BF16_STEP = 2.0 ** -7
LINEAR_TOL = 1e-4
ATTN_TOL = 1e-2
BLOCK_TOL = 2e-2
ROUTE_GAP = 0.05


def _gen(seed):
    return torch.Generator().manual_seed(seed)


# ------------------------------------------------------------------ RMSNorm ---

@pytest.mark.parametrize("rows,d", [(1, 256), (300, 512), (37, 4096)])
def test_rmsnorm(rows, d):
    g = _gen(rows + d)
    x = torch.randn((rows, d), generator=g).to(torch.bfloat16)
    gain = (1 + 0.1 * torch.randn(d, generator=g)).to(torch.bfloat16)
    y = torch.empty_like(x, device="cuda")
    moe.moe_rmsnorm(x.cuda(), gain.cuda(), 1e-5, y)
    torch.cuda.synchronize()
    assert_status_ok()
    ref = oracle.rms_norm(to_f64(x), to_f64(gain), 1e-5)
    err = np.abs(to_f64(y.cpu()) - ref)
    assert np.all(err <= BF16_STEP * np.abs(ref) + 1e-6 * np.abs(ref).max())


@pytest.mark.parametrize("rows,d", [(300, 512), (5, 4096)])
def test_rmsnorm_after_residual_add(rows, d):
    g = _gen(7 * rows + d)
    x = torch.randn((rows, d), generator=g).to(torch.bfloat16)
    add = torch.randn((rows, d), generator=g)
    gain = (1 + 0.1 * torch.randn(d, generator=g)).to(torch.bfloat16)
    h = torch.empty_like(x, device="cuda")
    y = torch.empty_like(x, device="cuda")
    moe.moe_rmsnorm(x.cuda(), gain.cuda(), 1e-5, y, add=add.cuda(), h_out=h)
    torch.cuda.synchronize()
    assert_status_ok()
    h_ref = to_f64(x) + add.double().numpy()
    assert np.all(np.abs(to_f64(h.cpu()) - h_ref) <= 2.0 ** -8 * np.abs(h_ref))  # one bf16 rounding
    ref = oracle.rms_norm(h_ref, to_f64(gain), 1e-5)
    err = np.abs(to_f64(y.cpu()) - ref)
    assert np.all(err <= BF16_STEP * np.abs(ref) + 2.0 ** -8 * np.abs(ref).max())


# ------------------------------------------------------------------- linear ---

@pytest.mark.parametrize("rows,n_in,n_out", [(300, 512, 768), (1, 64, 256), (513, 4096, 1024)])
def test_linear(rows, n_in, n_out):
    g = _gen(rows + n_in + n_out)
    x = torch.randn((rows, n_in), generator=g).to(torch.bfloat16)
    w = (torch.randn((n_out, n_in), generator=g) / math.sqrt(n_in)).to(torch.bfloat16)
    y = torch.full((rows, n_out), float("nan"), device="cuda")
    moe.moe_linear(x.cuda(), w.cuda(), y)
    torch.cuda.synchronize()
    assert_status_ok()
    ref = to_f64(x) @ to_f64(w).T
    assert np.max(np.abs(y.cpu().double().numpy() - ref)) <= LINEAR_TOL * np.max(np.abs(ref))


def test_linear_rejects_untiled_widths():
    x = torch.zeros((4, 96), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((256, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_linear(x, w, torch.zeros((4, 256), device="cuda"))
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


# --------------------------------------------------------------------- RoPE ---

@pytest.mark.parametrize("B,S,Hq,Hkv,base", [(2, 150, 4, 2, 10000.0), (1, 33000, 2, 1, 1e6)])
def test_rope_split(B, S, Hq, Hkv, base):
    hd = 128
    s = moe.make_block_shape(B, S, 256, Hq, Hkv, 256, rope_base=base)
    T = B * S
    qkv = torch.randn((T, (Hq + 2 * Hkv) * hd), generator=_gen(S))
    q = torch.empty((T, Hq * hd), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((T, Hkv * hd), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    moe.moe_rope_split(s, qkv.cuda(), q, k, v)
    torch.cuda.synchronize()
    assert_status_ok()
    a = qkv.double().numpy()
    pos = np.arange(T) % S
    want = {
        "q": oracle.rope(a[:, :Hq * hd].reshape(T, Hq, hd), pos, base),
        "k": oracle.rope(a[:, Hq * hd:(Hq + Hkv) * hd].reshape(T, Hkv, hd), pos, base),
        "v": a[:, (Hq + Hkv) * hd:].reshape(T, Hkv, hd),
    }
    for name, got in (("q", q), ("k", k), ("v", v)):
        ref = want[name]
        out = to_f64(got.cpu()).reshape(ref.shape)
        # each element within 2^-7 of its pair's length (one rounding plus the angle's float error)
        pair = np.sqrt(ref[..., 0::2] ** 2 + ref[..., 1::2] ** 2).repeat(2, axis=-1)
        assert np.all(np.abs(out - ref) <= BF16_STEP * pair + 1e-30), name


# ---------------------------------------------------------------- attention ---

def _attn_inputs(B, S, Hq, Hkv, seed, q_scale=1.0):
    g = _gen(seed)
    T, hd = B * S, 128
    q = (q_scale * torch.randn((T, Hq * hd), generator=g)).to(torch.bfloat16)
    k = torch.randn((T, Hkv * hd), generator=g).to(torch.bfloat16)
    v = torch.randn((T, Hkv * hd), generator=g).to(torch.bfloat16)
    return q, k, v


@pytest.mark.parametrize("B,S,Hq,Hkv,q_scale", [(2, 200, 4, 2, 1.0), (1, 1000, 8, 2, 3.0), (3, 128, 2, 2, 1.0),
                                                (1, 1, 4, 1, 1.0), (2, 77, 4, 4, 2.0)])
def test_attention(B, S, Hq, Hkv, q_scale):
    hd = 128
    s = moe.make_block_shape(B, S, 256, Hq, Hkv, 256)
    q, k, v = _attn_inputs(B, S, Hq, Hkv, seed=B * 1000 + S, q_scale=q_scale)
    o = torch.full((B * S, Hq * hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_attention(s, q.cuda(), k.cuda(), v.cuda(), o)
    torch.cuda.synchronize()
    assert_status_ok()
    out = to_f64(o.cpu()).reshape(B, S, Hq, hd)
    Q, K, V = (to_f64(t).reshape(B, S, -1, hd) for t in (q, k, v))
    for b in range(B):
        ref = oracle.causal_gqa_attention(Q[b], K[b], V[b])
        assert np.max(np.abs(out[b] - ref)) <= ATTN_TOL * np.max(np.abs(ref)), b
        # the first query sees only the first key: its output is that value, exactly
        for h in range(Hq):
            assert np.array_equal(out[b, 0, h], V[b, 0, h // (Hq // Hkv)])


def test_attention_rejects_other_head_widths():
    s = moe.make_block_shape(1, 16, 256, 2, 1, 256, head_dim=64)
    t = torch.zeros((16, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_attention(s, t, t, t, t)
    assert e.value.code == moe.MOE_ERR_UNSUPPORTED


def test_residual_add():
    g = _gen(3)
    a = torch.randn(4096 + 8, generator=g).to(torch.bfloat16)
    b = torch.randn(4096 + 8, generator=g).to(torch.bfloat16)
    out = torch.empty_like(a, device="cuda")
    moe.moe_residual_add(a.cuda(), b.cuda(), out)
    torch.cuda.synchronize()
    ref = to_f64(a) + to_f64(b)
    assert np.all(np.abs(to_f64(out.cpu()) - ref) <= 2.0 ** -8 * np.abs(ref))


# -------------------------------------------------------------- whole block ---

def _upload(p):
    return {k: v.cuda() for k, v in p.items()}


def _oracle_block(p, B, S, Hq, Hkv, tokens=None):
    """Oracle h, hn and, for the listed tokens, both admissible outputs."""
    # the expert weights are widened one expert at a time (the Mixtral shape's would not fit as float64)
    f = {k: to_f64(v) for k, v in p.items() if k not in ("w1", "w3", "w2")}
    a = oracle.attention_sublayer(f["x"], f["attn_norm"], f["wqkv"], f["wo"], S, Hq, Hkv)
    hn = oracle.rms_norm(a["h"], f["ffn_norm"])
    tokens = np.arange(B * S) if tokens is None else np.asarray(tokens)
    l = oracle.router_logits(hn[tokens], f["w_gate"])
    order = np.argsort(-l, axis=1, kind="stable")
    outs, tight = [], []
    for i, t in enumerate(tokens):
        e1, e2, e3 = order[i, :3]
        tight.append(l[i, e2] - l[i, e3] < ROUTE_GAP)
        cand = []
        for pair in ((e1, e2), (e1, e3)) if tight[-1] else ((e1, e2),):
            z = l[i, list(pair)]
            w = np.exp(z - z.max())
            w = w / w.sum()
            y = sum(w[j] * oracle.expert_forward(hn[t:t + 1], to_f64(p["w1"][e]), to_f64(p["w3"][e]),
                                                 to_f64(p["w2"][e]))[0]
                    for j, e in enumerate(pair))
            cand.append(a["h"][t] + y)
        outs.append(cand)
    return a, outs, np.array(tight)


def _check_block(out, outs, tokens, scale):
    for i, t in enumerate(tokens):
        errs = [np.max(np.abs(out[t] - c)) for c in outs[i]]
        assert min(errs) <= BLOCK_TOL * scale, (t, errs)


def test_block_small_model_against_the_oracle():
    c = BLOCK_CONFIGS["small"]
    p = make_block_config("small")
    s = moe.make_block_shape(c["B"], c["S"], c["d"], c["n_heads"], c["n_kv_heads"], c["ffn"])
    dev = _upload(p)
    out = moe.block_forward(dev["x"], dev, s)
    torch.cuda.synchronize()
    assert_status_ok()
    a, outs, tight = _oracle_block(p, c["B"], c["S"], c["n_heads"], c["n_kv_heads"])
    got = to_f64(out.cpu())
    scale = max(np.max(np.abs(o[0])) for o in outs)
    _check_block(got, outs, range(c["B"] * c["S"]), scale)
    # router scores are ~N(0, 1): about one token in ten has its 2nd and 3rd expert within 0.05
    assert tight.mean() < 0.2


def test_block_equals_its_steps_and_keeps_sequences_apart():
    c = BLOCK_CONFIGS["small"]
    p = make_block_config("small")
    B, S, d = c["B"], c["S"], c["d"]
    Hq, Hkv, hd = c["n_heads"], c["n_kv_heads"], 128
    s = moe.make_block_shape(B, S, d, Hq, Hkv, c["ffn"])
    dev = _upload(p)
    out = moe.block_forward(dev["x"], dev, s)
    # the same steps through their own calls
    T = B * S
    bf = dict(dtype=torch.bfloat16, device="cuda")
    xn = torch.empty((T, d), **bf)
    qkv = torch.empty((T, (Hq + 2 * Hkv) * hd), device="cuda")
    q, k, v = (torch.empty((T, n * hd), **bf) for n in (Hq, Hkv, Hkv))
    attn = torch.empty((T, Hq * hd), **bf)
    o = torch.empty((T, d), device="cuda")
    h, hn = torch.empty((T, d), **bf), torch.empty((T, d), **bf)
    moe.moe_rmsnorm(dev["x"], dev["attn_norm"], 1e-5, xn)
    moe.moe_linear(xn, dev["wqkv"], qkv)
    moe.moe_rope_split(s, qkv, q, k, v)
    moe.moe_attention(s, q, k, v, attn)
    moe.moe_linear(attn, dev["wo"], o)
    moe.moe_rmsnorm(dev["x"], dev["ffn_norm"], 1e-5, hn, add=o, h_out=h)
    y = moe.layer_forward(hn, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"])
    steps = torch.empty_like(h)
    moe.moe_residual_add(h, y, steps)
    torch.cuda.synchronize()
    assert_status_ok()
    assert torch.equal(out, steps)
    # each sequence alone gives its rows of the batch; the router takes another kernel for 160 tokens
    # than for 320 (one CTA per token), so gate weights may differ in the last fp32 bit and an
    # output element by one bf16 step
    s1 = moe.make_block_shape(1, S, d, Hq, Hkv, c["ffn"])
    for b in range(B):
        one = moe.block_forward(dev["x"][b * S:(b + 1) * S].contiguous(), dev, s1)
        torch.cuda.synchronize()
        diff = (one.float() - out[b * S:(b + 1) * S].float()).abs().max().item()
        assert diff <= 2.0 ** -7 * out.float().abs().max().item()


def test_block_is_causal():
    c = BLOCK_CONFIGS["small"]
    p = make_block_config("small")
    S, d = c["S"], c["d"]
    s1 = moe.make_block_shape(1, S, d, c["n_heads"], c["n_kv_heads"], c["ffn"])
    dev = _upload(p)
    x = dev["x"][:S].contiguous()
    a = moe.block_forward(x, dev, s1)
    x2 = x.clone()
    x2[100:] = torch.randn((S - 100, d), generator=_gen(9)).to(torch.bfloat16).cuda()
    b = moe.block_forward(x2, dev, s1)
    torch.cuda.synchronize()
    assert_status_ok()
    assert (a[:100].float() - b[:100].float()).abs().max().item() <= 1e-3 * a.float().abs().max().item()
    assert not torch.equal(a[100:], b[100:])


def test_block_mixtral_shape_sampled_tokens():
    """Mixtral's block (d 4096, 32/8 heads, ffn 14336) on one 256-token sequence, 12 tokens checked."""
    d, Hq, Hkv, ffn, S = 4096, 32, 8, 14336, 256
    p = make_block(1, S, d, Hq, Hkv, ffn, seed=5330, weight_seed=5331)
    s = moe.make_block_shape(1, S, d, Hq, Hkv, ffn)
    dev = _upload(p)
    out = moe.block_forward(dev["x"], dev, s)
    torch.cuda.synchronize()
    assert_status_ok()
    tokens = [0, 1, 2, 63, 127, 128, 129, 200, 253, 254, 255, 31]
    _, outs, _ = _oracle_block(p, 1, S, Hq, Hkv, tokens)
    got = to_f64(out.cpu())
    scale = max(np.max(np.abs(o[0])) for o in outs)
    _check_block(got, outs, tokens, scale)


def test_block_rejects_bad_shapes_and_small_workspace():
    ok = moe.make_block_shape(1, 16, 512, 4, 2, 512)
    assert moe.moe_block_workspace_bytes(ok) > 0
    for bad in (moe.make_block_shape(1, 16, 512, 4, 3, 512),        # heads not a multiple of KV heads
                moe.make_block_shape(0, 16, 512, 4, 2, 512),        # no sequences
                moe.make_block_shape(1, 16, 512, 1, 1, 512)):       # projection 384 wide: not a 256 multiple
        assert moe.moe_block_workspace_bytes(bad) == 0
    p = _upload(make_block(1, 16, 512, 4, 2, 512, seed=3))
    out = torch.empty_like(p["x"])
    ws = torch.empty(moe.moe_block_workspace_bytes(ok) - 1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(moe.MoEError) as e:
        moe.moe_block_forward(ok, p["x"], moe.block_weights(p), out, ws)  # no caches
    assert e.value.code == moe.MOE_ERR_WORKSPACE
