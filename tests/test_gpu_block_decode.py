"""The decoder block's decode form on the GPU against the fp64 oracle.

One new token per sequence attends to a key/value cache. Checked here: the
weight-streaming linear layer (the decode batch's projections), RoPE with
device positions writing the caches, the split-key decode attention on ragged
cache lengths, the decode step against the oracle's incremental step on a
seeded cache, and prefill-then-decode against the oracle's whole-sequence
block (the last token of a sequence computed both ways). Tolerances as in
test_gpu_block.py: bf16 outputs within 2e-2 of the reference scale, decode
attention (fp32 P) within 1e-2, and the either-expert acceptance for router
near-ties inside the block.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from moe_inputs import BLOCK_CONFIGS, make_block, make_block_config, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import assert_status_ok
from test_gpu_block import BLOCK_TOL, ROUTE_GAP, _check_block

pytestmark = pytest.mark.gpu

HD = 128


def _gen(seed):
    return torch.Generator().manual_seed(seed)


@pytest.mark.parametrize("rows,n_in,n_out", [(16, 4096, 6144), (1, 512, 256), (64, 4096, 4096), (37, 1024, 768)])
def test_linear_weight_streaming(rows, n_in, n_out):
    g = _gen(rows * 7 + n_out)
    x = torch.randn((rows, n_in), generator=g).to(torch.bfloat16)
    w = (torch.randn((n_out, n_in), generator=g) / math.sqrt(n_in)).to(torch.bfloat16)
    n = moe.moe_linear_workspace_bytes(rows, n_in, n_out)
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    y = torch.full((rows, n_out), float("nan"), device="cuda")
    moe.moe_linear(x.cuda(), w.cuda(), y, ws=ws)
    torch.cuda.synchronize()
    assert_status_ok()
    ref = to_f64(x) @ to_f64(w).T
    assert np.max(np.abs(y.cpu().double().numpy() - ref)) <= 1e-4 * np.max(np.abs(ref))


def test_rope_split_writes_the_caches_at_their_positions():
    B, S, Hq, Hkv, cmax = 2, 150, 4, 2, 300
    s = moe.make_block_shape(B, S, 256, Hq, Hkv, 256, cache_max=cmax)
    qkv = torch.randn((B * S, (Hq + 2 * Hkv) * HD), generator=_gen(4))
    q = torch.empty((B * S, Hq * HD), dtype=torch.bfloat16, device="cuda")
    k, v = (torch.empty((B * S, Hkv * HD), dtype=torch.bfloat16, device="cuda") for _ in range(2))
    kc, vc = moe.kv_cache(s)
    moe.moe_rope_split(s, qkv.cuda(), q, k, v, k_cache=kc, v_cache=vc)
    torch.cuda.synchronize()
    assert_status_ok()
    # the cache holds the same bf16 values as the token-major outputs, head-major
    assert torch.equal(kc[:, :, :S].permute(0, 2, 1, 3).reshape(B * S, Hkv * HD), k)
    assert torch.equal(vc[:, :, :S].permute(0, 2, 1, 3).reshape(B * S, Hkv * HD), v)
    assert not kc[:, :, S:].any()
    # decode: one token per sequence at a device-held position
    s1 = moe.make_block_shape(B, 1, 256, Hq, Hkv, 256, cache_max=cmax)
    pos = torch.tensor([5, 299], dtype=torch.int32, device="cuda")
    qkv1 = torch.randn((B, (Hq + 2 * Hkv) * HD), generator=_gen(5))
    q1 = torch.empty((B, Hq * HD), dtype=torch.bfloat16, device="cuda")
    moe.moe_rope_split(s1, qkv1.cuda(), q1, None, None, pos=pos, k_cache=kc, v_cache=vc)
    torch.cuda.synchronize()
    assert_status_ok()
    a = qkv1.double().numpy()
    for b, p in enumerate((5, 299)):
        kref = oracle.rope(a[b, Hq * HD:(Hq + Hkv) * HD].reshape(1, Hkv, HD), np.array([p]))[0]
        got = to_f64(kc[b, :, p].cpu())
        pair = np.sqrt(kref[..., 0::2] ** 2 + kref[..., 1::2] ** 2).repeat(2, axis=-1)
        assert np.all(np.abs(got - kref) <= 2.0 ** -7 * pair + 1e-30)
        assert np.array_equal(to_f64(vc[b, :, p].cpu()), to_f64(torch.from_numpy(
            a[b, (Hq + Hkv) * HD:].reshape(Hkv, HD)).to(torch.bfloat16)))


@pytest.mark.parametrize("lens,Hq,Hkv,cmax", [((0, 1, 255, 256, 700), 32, 8, 1000), ((4095,), 8, 2, 4096),
                                               ((10, 300), 4, 4, 333), ((127, 128, 129), 16, 8, 300),
                                               ((50, 999), 16, 2, 1000), ((3, 2000), 32, 2, 2048),
                                               tuple([tuple(range(0, 3200, 100)), 8, 8, 3300]),
                                               ((100, 1000), 12, 4, 1100), ((77,), 24, 4, 200)])
def test_attention_decode_on_ragged_caches(lens, Hq, Hkv, cmax):
    B = len(lens)
    s = moe.make_block_shape(B, 1, 256, Hq, Hkv, 256, cache_max=cmax)
    g = _gen(sum(lens) + Hq)
    q = torch.randn((B, Hq * HD), generator=g).to(torch.bfloat16)
    kc = (torch.randn((B, Hkv, cmax, HD), generator=g)).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, cmax, HD), generator=g).to(torch.bfloat16)
    length = torch.tensor(lens, dtype=torch.int32)
    ws = torch.empty(moe.moe_attention_decode_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    o = torch.full((B, Hq * HD), float("nan"), dtype=torch.bfloat16, device="cuda")
    dlen = length.cuda()
    moe.moe_attention_decode(s, q.cuda(), kc.cuda(), vc.cuda(), dlen, o, ws)
    torch.cuda.synchronize()
    assert_status_ok()
    assert dlen.cpu().tolist() == [min(n + 1, cmax) for n in lens]  # advanced by one
    out = to_f64(o.cpu()).reshape(B, Hq, HD)
    for b, n in enumerate(lens):
        keys = to_f64(kc[b, :, :n + 1].permute(1, 0, 2))
        vals = to_f64(vc[b, :, :n + 1].permute(1, 0, 2))
        ref = oracle.attention_one_query(to_f64(q[b]).reshape(Hq, HD), keys, vals)
        assert np.max(np.abs(out[b] - ref)) <= 1e-2 * np.max(np.abs(ref)), (b, n)


def test_attention_decode_ignores_what_the_cache_holds_past_its_length():
    """Cache rows past a sequence's keys (never written: here NaN and Inf) must not reach the output;
    the result equals the one with zeros there, bit for bit, and the oracle's."""
    lens, Hq, Hkv, cmax = (5, 130, 255), 8, 2, 384
    B = len(lens)
    s = moe.make_block_shape(B, 1, 256, Hq, Hkv, 256, cache_max=cmax)
    g = _gen(31)
    q = torch.randn((B, Hq * HD), generator=g).to(torch.bfloat16).cuda()
    kc = torch.randn((B, Hkv, cmax, HD), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, cmax, HD), generator=g).to(torch.bfloat16)
    outs = []
    for fill in (0.0, float("nan"), float("inf")):
        k2, v2 = kc.clone(), vc.clone()
        for b, n in enumerate(lens):
            k2[b, :, n + 1:] = fill
            v2[b, :, n + 1:] = fill
        ws = torch.empty(moe.moe_attention_decode_workspace_bytes(s), dtype=torch.uint8, device="cuda")
        o = torch.empty((B, Hq * HD), dtype=torch.bfloat16, device="cuda")
        moe.moe_attention_decode(s, q, k2.cuda(), v2.cuda(), torch.tensor(lens, dtype=torch.int32).cuda(), o, ws)
        torch.cuda.synchronize()
        assert_status_ok()
        outs.append(o.cpu())
    assert torch.isfinite(outs[0].float()).all()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
    out = to_f64(outs[0]).reshape(B, Hq, HD)
    for b, n in enumerate(lens):
        keys = to_f64(kc[b, :, :n + 1].permute(1, 0, 2))
        vals = to_f64(vc[b, :, :n + 1].permute(1, 0, 2))
        ref = oracle.attention_one_query(to_f64(q[b].cpu()).reshape(Hq, HD), keys, vals)
        assert np.max(np.abs(out[b] - ref)) <= 1e-2 * np.max(np.abs(ref)), (b, n)


def test_attention_decode_with_a_full_cache_reports_and_keeps_the_length():
    s = moe.make_block_shape(1, 1, 256, 4, 2, 256, cache_max=64)
    q = torch.randn((1, 4 * HD), generator=_gen(6)).to(torch.bfloat16).cuda()
    kc, vc = moe.kv_cache(s)
    before = kc.clone()
    # RoPE for a token at position 64 of a 64-slot cache: reported, nothing written
    qkv = torch.randn((1, 8 * HD), generator=_gen(7)).cuda()
    pos = torch.tensor([64], dtype=torch.int32, device="cuda")
    moe.moe_rope_split(s, qkv, q, None, None, pos=pos, k_cache=kc, v_cache=vc)
    torch.cuda.synchronize()
    code, _ = moe.moe_get_device_status()
    assert code == moe.MOE_ERR_DEVICE_CHECK
    assert torch.equal(kc, before)
    ws = torch.empty(moe.moe_attention_decode_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    o = torch.empty((1, 4 * HD), dtype=torch.bfloat16, device="cuda")
    moe.moe_attention_decode(s, q, kc, vc, pos, o, ws)
    torch.cuda.synchronize()
    assert_status_ok()
    assert pos.item() == 64  # a full cache is not advanced


def _upload(p):
    return {k: v.cuda() for k, v in p.items()}


class _LazyExperts:
    """Expert weights widened to float64 one expert at a time (the Mixtral shape's would not fit at once)."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return to_f64(self.t[e])


def _oracle_params(p, lazy=True):
    """The block's tensors under the oracle's names, float64 (expert weights widened on use)."""
    q = dict(g_attn=to_f64(p["attn_norm"]), wqkv=to_f64(p["wqkv"]), wo=to_f64(p["wo"]),
             g_ffn=to_f64(p["ffn_norm"]), w_gate=to_f64(p["w_gate"]))
    for n in ("w1", "w3", "w2"):
        q[n] = _LazyExperts(p[n]) if lazy else to_f64(p[n])
    return q


def _decode_candidates(p, x_new, k_prefix, v_prefix, Hq, Hkv):
    """Oracle decode step; for a router near-tie both admissible outputs."""
    f = _oracle_params(p)
    step = oracle.decoder_block_decode(to_f64(x_new), k_prefix, v_prefix, f, Hq, Hkv)
    l = step["moe"]["logits"]
    outs = []
    for t in range(x_new.shape[0]):
        order = np.argsort(-l[t], kind="stable")
        e1, e2, e3 = order[:3]
        cands = [step["out"][t]]
        if l[t, e2] - l[t, e3] < ROUTE_GAP:
            z = l[t, [e1, e3]]
            w = np.exp(z - z.max())
            w = w / w.sum()
            y = sum(w[j] * oracle.expert_forward(step["hn"][t:t + 1], f["w1"][e], f["w3"][e], f["w2"][e])[0]
                    for j, e in enumerate((e1, e3)))
            cands.append(step["h"][t] + y)
        outs.append(cands)
    return step, outs


def test_decode_step_against_the_oracle_on_a_seeded_cache():
    c = BLOCK_CONFIGS["small"]
    p = make_block_config("small")
    d, Hq, Hkv, F = c["d"], c["n_heads"], c["n_kv_heads"], c["ffn"]
    lens = [0, 37, 200, 255]
    B, cmax = len(lens), 260
    g = _gen(11)
    k_prefix = [torch.randn((n, Hkv, HD), generator=g).to(torch.bfloat16) for n in lens]
    v_prefix = [torch.randn((n, Hkv, HD), generator=g).to(torch.bfloat16) for n in lens]
    kc = torch.zeros((B, Hkv, cmax, HD), dtype=torch.bfloat16)
    vc = torch.zeros_like(kc)
    for b, n in enumerate(lens):
        kc[b, :, :n] = k_prefix[b].permute(1, 0, 2)
        vc[b, :, :n] = v_prefix[b].permute(1, 0, 2)
    x_new = torch.randn((B, d), generator=g).to(torch.bfloat16)
    s = moe.make_block_shape(B, 1, d, Hq, Hkv, F, cache_max=cmax)
    dev = _upload(p)
    kcd, vcd = kc.cuda(), vc.cuda()
    clen = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = moe.block_decode(x_new.cuda(), dev, s, kcd, vcd, clen)
    torch.cuda.synchronize()
    assert_status_ok()
    assert clen.cpu().tolist() == [n + 1 for n in lens]
    step, outs = _decode_candidates(p, x_new, [to_f64(k) for k in k_prefix], [to_f64(v) for v in v_prefix], Hq, Hkv)
    got = to_f64(out.cpu())
    scale = max(np.max(np.abs(o[0])) for o in outs)
    _check_block(got, outs, range(B), scale)
    # the appended key and value are the oracle's (bf16 rounding of RoPE's output)
    for b, n in enumerate(lens):
        assert np.max(np.abs(to_f64(kcd[b, :, n].cpu()) - step["k_new"][b])) <= 2e-2 * np.max(np.abs(step["k_new"][b]))
        assert np.max(np.abs(to_f64(vcd[b, :, n].cpu()) - step["v_new"][b])) <= 2e-2 * np.max(np.abs(step["v_new"][b]))


def test_prefill_then_decode_steps_match_the_whole_sequence():
    c = BLOCK_CONFIGS["small"]
    d, Hq, Hkv, F = c["d"], c["n_heads"], c["n_kv_heads"], c["ffn"]
    B, S0, steps, cmax = 2, 150, 3, 160
    p = make_block(B, S0 + steps, d, Hq, Hkv, F, seed=41, weight_seed=42)
    dev = _upload(p)
    x_all = p["x"].view(B, S0 + steps, d)
    # prefill of the first S0 tokens of every sequence, filling the caches
    s_pre = moe.make_block_shape(B, S0, d, Hq, Hkv, F, cache_max=cmax)
    kc, vc = moe.kv_cache(s_pre)
    moe.block_forward(x_all[:, :S0].reshape(B * S0, d).contiguous().cuda(), dev, s_pre, k_cache=kc, v_cache=vc)
    clen = torch.full((B,), S0, dtype=torch.int32, device="cuda")
    s_dec = moe.make_block_shape(B, 1, d, Hq, Hkv, F, cache_max=cmax)
    outs = []
    for j in range(steps):
        outs.append(moe.block_decode(x_all[:, S0 + j].contiguous().cuda(), dev, s_dec, kc, vc, clen))
    torch.cuda.synchronize()
    assert_status_ok()
    assert clen.cpu().tolist() == [S0 + steps] * B
    # the oracle's block over the whole sequences: its last `steps` tokens
    full_x = to_f64(p["x"])
    f = _oracle_params(p, lazy=False)
    full = oracle.decoder_block(full_x, f, S0 + steps, Hq, Hkv)
    l = full["moe"]["logits"]
    for j in range(steps):
        got = to_f64(outs[j].cpu())
        for b in range(B):
            t = b * (S0 + steps) + S0 + j
            order = np.argsort(-l[t], kind="stable")
            cands = [full["out"][t]]
            if l[t, order[1]] - l[t, order[2]] < ROUTE_GAP:
                e1, e3 = order[0], order[2]
                z = l[t, [e1, e3]]
                w = np.exp(z - z.max())
                w = w / w.sum()
                y = sum(w[i] * oracle.expert_forward(full["hn"][t:t + 1], f["w1"][e], f["w3"][e], f["w2"][e])[0]
                        for i, e in enumerate((e1, e3)))
                cands.append(full["h"][t] + y)
            scale = np.max(np.abs(full["out"]))
            assert min(np.max(np.abs(got[b] - cnd)) for cnd in cands) <= BLOCK_TOL * scale, (j, b)


def test_decode_step_equals_its_steps():
    c = BLOCK_CONFIGS["small"]
    p = make_block_config("small")
    d, Hq, Hkv, F = c["d"], c["n_heads"], c["n_kv_heads"], c["ffn"]
    B, cmax = 3, 96
    s = moe.make_block_shape(B, 1, d, Hq, Hkv, F, cache_max=cmax)
    dev = _upload(p)
    g = _gen(12)
    kc0 = torch.randn((B, Hkv, cmax, HD), generator=g).to(torch.bfloat16).cuda()
    vc0 = torch.randn((B, Hkv, cmax, HD), generator=g).to(torch.bfloat16).cuda()
    lens = torch.tensor([3, 50, 95], dtype=torch.int32, device="cuda")
    x = dev["x"][:B].contiguous()
    kc, vc, l1 = kc0.clone(), vc0.clone(), lens.clone()
    out = moe.block_decode(x, dev, s, kc, vc, l1)
    # the same through the step calls
    kc2, vc2, l2 = kc0.clone(), vc0.clone(), lens.clone()
    bf = dict(dtype=torch.bfloat16, device="cuda")
    wq, wqkv = Hq * HD, (Hq + 2 * Hkv) * HD
    xn = torch.empty((B, d), **bf)
    qkv = torch.empty((B, wqkv), device="cuda")
    q = torch.empty((B, wq), **bf)
    attn = torch.empty((B, wq), **bf)
    o = torch.empty((B, d), device="cuda")
    h, hn = torch.empty((B, d), **bf), torch.empty((B, d), **bf)
    lw = torch.empty(max(moe.moe_linear_workspace_bytes(B, d, wqkv), moe.moe_linear_workspace_bytes(B, wq, d)),
                     dtype=torch.uint8, device="cuda")
    aw = torch.empty(moe.moe_attention_decode_workspace_bytes(s), dtype=torch.uint8, device="cuda")
    moe.moe_rmsnorm(x, dev["attn_norm"], 1e-5, xn)
    moe.moe_linear(xn, dev["wqkv"], qkv, ws=lw)
    moe.moe_rope_split(s, qkv, q, None, None, pos=l2, k_cache=kc2, v_cache=vc2)
    moe.moe_attention_decode(s, q, kc2, vc2, l2, attn, aw)
    moe.moe_linear(attn, dev["wo"], o, ws=lw)
    moe.moe_rmsnorm(x, dev["ffn_norm"], 1e-5, hn, add=o, h_out=h)
    y = moe.layer_forward(hn, dev["w_gate"], dev["w1"], dev["w3"], dev["w2"])
    steps = torch.empty_like(h)
    moe.moe_residual_add(h, y, steps)
    torch.cuda.synchronize()
    assert_status_ok()
    assert torch.equal(out, steps)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2) and torch.equal(l1, l2)


def test_decode_step_mixtral_shape():
    """Mixtral's block for 16 sequences with 500 cached tokens each (seeded cache values)."""
    d, Hq, Hkv, F = 4096, 32, 8, 14336
    B, L, cmax = 16, 500, 512
    p = make_block(B, 1, d, Hq, Hkv, F, seed=5340, weight_seed=5341)
    g = _gen(13)
    kc = torch.randn((B, Hkv, cmax, HD), generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, cmax, HD), generator=g).to(torch.bfloat16)
    s = moe.make_block_shape(B, 1, d, Hq, Hkv, F, cache_max=cmax)
    dev = _upload(p)
    clen = torch.full((B,), L, dtype=torch.int32, device="cuda")
    out = moe.block_decode(dev["x"], dev, s, kc.cuda(), vc.cuda(), clen)
    torch.cuda.synchronize()
    assert_status_ok()
    check = [0, 5, 15]
    kp = [to_f64(kc[b, :, :L].permute(1, 0, 2)) for b in check]
    vp = [to_f64(vc[b, :, :L].permute(1, 0, 2)) for b in check]
    sub = {k: (v[check] if k == "x" else v) for k, v in p.items()}
    _, outs = _decode_candidates(sub, sub["x"], kp, vp, Hq, Hkv)
    got = to_f64(out.cpu())[check]
    scale = max(np.max(np.abs(o[0])) for o in outs)
    _check_block(got, outs, range(len(check)), scale)
