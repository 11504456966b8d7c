"""The decoder block at the sizes its benchmarks time, checked on sampled outputs.

bench.py --block runs the Mixtral block on one 4096-token sequence
(`mixtral_block_prefill_B1_S4096`); bench.py --block-decode runs one decode
step for 16 sequences with 4096 cached tokens. Here the same inputs (same
seeds, same cache draw) go through the same calls, and the oracle computes the
attention side for every token and the MoE layer for sampled tokens; the
tolerances and the router near-tie acceptance are those of test_gpu_block.py.
"""
import numpy as np
import pytest
import torch

import oracle
from moe_inputs import BLOCK_CONFIGS, make_block, make_block_config, make_weights, to_f64
from sparse_mixture_experts_53_b300 import moe

from gpu_harness import assert_status_ok
from test_gpu_block import ROUTE_GAP, _check_block
from test_gpu_block_decode import _decode_candidates, _oracle_params

pytestmark = pytest.mark.gpu

HD = 128


@pytest.fixture(scope="module")
def mixtral_experts():
    return make_weights(4096, 14336, 8, "bf16", 5310)


def test_block_prefill_bench_configuration(mixtral_experts):
    c = BLOCK_CONFIGS["mixtral"]
    B, S, d, Hq, Hkv, F = c["B"], c["S"], c["d"], c["n_heads"], c["n_kv_heads"], c["ffn"]
    p = make_block_config("mixtral", moe_weights=mixtral_experts)
    dev = {k: v.cuda() for k, v in p.items()}
    s = moe.make_block_shape(B, S, d, Hq, Hkv, F)
    out = moe.block_forward(dev["x"], dev, s)
    torch.cuda.synchronize()
    assert_status_ok()
    del dev
    f = _oracle_params(p)
    a = oracle.attention_sublayer(to_f64(p["x"]), f["g_attn"], f["wqkv"], f["wo"], S, Hq, Hkv)
    hn = oracle.rms_norm(a["h"], f["g_ffn"])
    rng = np.random.default_rng(3)
    tokens = sorted(set([0, 1, 127, 128, 2047, 4095] + rng.integers(0, S, 6).tolist()))
    l = oracle.router_logits(hn[tokens], f["w_gate"])
    outs = []
    for i, t in enumerate(tokens):
        order = np.argsort(-l[i], kind="stable")
        pairs = [order[:2]]
        if l[i, order[1]] - l[i, order[2]] < ROUTE_GAP:
            pairs.append(order[[0, 2]])
        cands = []
        for pair in pairs:
            z = l[i, pair]
            w = np.exp(z - z.max())
            w = w / w.sum()
            y = sum(w[j] * oracle.expert_forward(hn[t:t + 1], f["w1"][e], f["w3"][e], f["w2"][e])[0]
                    for j, e in enumerate(pair))
            cands.append(a["h"][t] + y)
        outs.append(cands)
    got = to_f64(out.cpu())[tokens]
    scale = max(np.max(np.abs(o[0])) for o in outs)
    _check_block(got, outs, range(len(tokens)), scale)


def test_block_decode_bench_configuration(mixtral_experts):
    B, L, d, Hq, Hkv, F = 16, 4096, 4096, 32, 8, 14336
    p = make_block(B, 1, d, Hq, Hkv, F, seed=5350, weight_seed=5310, moe_weights=mixtral_experts)
    cmax = L + 5 + 2 * 200 + 8   # the capacity of the default bench run (5 warm-up, 200 timed steps)
    s = moe.make_block_shape(B, 1, d, Hq, Hkv, F, cache_max=cmax)
    g = torch.Generator(device="cuda").manual_seed(5351)
    kc = torch.randn((B, Hkv, cmax, HD), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, cmax, HD), device="cuda", generator=g).to(torch.bfloat16)
    clen = torch.full((B,), L, dtype=torch.int32, device="cuda")
    dev = {k: v.cuda() for k, v in p.items()}
    out = moe.block_decode(dev["x"], dev, s, kc, vc, clen)
    torch.cuda.synchronize()
    assert_status_ok()
    assert clen.cpu().tolist() == [L + 1] * B
    check = [0, 7, 15]
    kp = [to_f64(kc[b, :, :L].permute(1, 0, 2).cpu()) for b in check]
    vp = [to_f64(vc[b, :, :L].permute(1, 0, 2).cpu()) for b in check]
    sub = {k: (v[check] if k == "x" else v) for k, v in p.items()}
    _, outs = _decode_candidates(sub, sub["x"], kp, vp, Hq, Hkv)
    got = to_f64(out.cpu())[check]
    scale = max(np.max(np.abs(o[0])) for o in outs)
    _check_block(got, outs, range(len(check)), scale)
