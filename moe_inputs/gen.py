"""Seeded generator of synthetic MoE-layer inputs.

Recipe (the same for every consumer):

* Every tensor is drawn from its own numpy PCG64 stream, keyed by
  ``SeedSequence([seed, stream_id, chunk])`` over fixed chunks of 2**22 values.
  The result does not depend on the number of host threads.
* Draws are float32 standard normals, multiplied in float32 by the float32
  standard deviation: x ~ N(0, 1), W_g ~ N(0, 1/d), W1, W3 ~ N(0, 1/d),
  W2 ~ N(0, 1/ffn).
* bf16 layers round each float32 tensor to bf16 (round to nearest even).
* Storage follows the nn.Linear convention, ``[out][in]`` row-major:
  ``w_gate[E][d]`` (row e is the e-th column of the page's ``x . W_g``),
  ``w1[E][ffn][d]``, ``w3[E][ffn][d]``, ``w2[E][d][ffn]``.
* Skewed layers: ``x = z + c*u`` with z ~ N(0, 1) and u a fixed random unit
  vector; rows 0 and 1 of ``w_gate`` get ``u/sqrt(d)`` added (in float64, then
  rounded to float32, then to bf16).
* Token rows whose router scores have a near-tie are redrawn from a per-row
  stream ``SeedSequence([seed, 7, t, attempt])``. Which rows (and the skew
  constant c) is decided once by a calibration script under ``tests/golden``
  and stored in ``tests/golden/input_schedule.json``; this module only replays
  that list. It never evaluates the router.
"""
from __future__ import annotations

import json
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from pathlib import Path

import numpy as np
import torch

CHUNK = 1 << 22

STREAM_X = 1
STREAM_WG = 2
STREAM_W1 = 3
STREAM_W3 = 4
STREAM_W2 = 5
STREAM_U = 6
STREAM_REDRAW = 7
STREAM_ATTN_NORM = 8
STREAM_WQKV = 9
STREAM_WO = 10
STREAM_FFN_NORM = 11
STREAM_DECODE = 12

SCHEDULE_PATH = Path(__file__).resolve().parent.parent / "tests" / "golden" / "input_schedule.json"

# The five workloads. Configs 1-4 are batches through the same Mixtral-shape
# layer, so they share one weight draw (weight_seed 5310); the tokens and the
# router matrix are drawn per config.
CONFIGS = {
    0: dict(name="tiny_fp32_T64", T=64, d=128, ffn=256, E=8, dtype="f32",
            seed=5300, weight_seed=5300, aux=False, skew=False),
    1: dict(name="mixtral_decode_T16", T=16, d=4096, ffn=14336, E=8, dtype="bf16",
            seed=5301, weight_seed=5310, aux=False, skew=False),
    2: dict(name="mixtral_prefill_T4096", T=4096, d=4096, ffn=14336, E=8, dtype="bf16",
            seed=5302, weight_seed=5310, aux=False, skew=False),
    3: dict(name="mixtral_large_T16384_aux", T=16384, d=4096, ffn=14336, E=8, dtype="bf16",
            seed=5303, weight_seed=5310, aux=True, skew=False),
    4: dict(name="mixtral_skewed_T8192", T=8192, d=4096, ffn=14336, E=8, dtype="bf16",
            seed=5304, weight_seed=5310, aux=False, skew=True),
}


def _threads() -> int:
    return max(1, min(32, os.cpu_count() or 1))


def normal_f32(seed: int, stream: int, n: int, std: float) -> np.ndarray:
    """n float32 draws of N(0, std^2), chunked so the result is thread-count free."""
    out = np.empty(n, np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK
    s32 = np.float32(std)

    def fill(i: int) -> None:
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream, i])))
        a, b = i * CHUNK, min(n, (i + 1) * CHUNK)
        g.standard_normal(out=out[a:b], dtype=np.float32)
        if s32 != np.float32(1.0):
            np.multiply(out[a:b], s32, out=out[a:b])

    if nchunks <= 1:
        for i in range(nchunks):
            fill(i)
    else:
        with ThreadPoolExecutor(min(nchunks, _threads())) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


def _store(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    if dtype == "bf16":
        return t.to(torch.bfloat16)
    if dtype == "f32":
        return t
    raise ValueError(f"unknown dtype {dtype!r}")


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a stored (bf16 or f32) tensor to a float64 array."""
    return t.to(torch.float32).numpy().astype(np.float64)


def skew_direction(seed: int, d: int) -> np.ndarray:
    """The fixed random unit vector u of the skewed workload (float64)."""
    u = normal_f32(seed, STREAM_U, d, 1.0).astype(np.float64)
    return u / np.sqrt(np.dot(u, u))


def make_weights(d: int, ffn: int, E: int, dtype: str, seed: int):
    """(w1 [E][ffn][d], w3 [E][ffn][d], w2 [E][d][ffn]) as CPU tensors."""
    w1 = _store(normal_f32(seed, STREAM_W1, E * ffn * d, 1.0 / np.sqrt(d)), dtype).view(E, ffn, d)
    w3 = _store(normal_f32(seed, STREAM_W3, E * ffn * d, 1.0 / np.sqrt(d)), dtype).view(E, ffn, d)
    w2 = _store(normal_f32(seed, STREAM_W2, E * d * ffn, 1.0 / np.sqrt(ffn)), dtype).view(E, d, ffn)
    return w1, w3, w2


def _token_rows_f32(seed: int, T: int, d: int, skew_c: float | None) -> np.ndarray:
    z = normal_f32(seed, STREAM_X, T * d, 1.0).reshape(T, d)
    if skew_c is None:
        return z
    u = skew_direction(seed, d)
    return (z.astype(np.float64) + skew_c * u[None, :]).astype(np.float32)


def _gate_f32(seed: int, E: int, d: int, skew: bool) -> np.ndarray:
    wg = normal_f32(seed, STREAM_WG, E * d, 1.0 / np.sqrt(d)).reshape(E, d)
    if not skew:
        return wg
    u = skew_direction(seed, d)
    wg = wg.astype(np.float64)
    wg[0] += u / np.sqrt(d)
    wg[1] += u / np.sqrt(d)
    return wg.astype(np.float32)


def redraw_token_row(seed: int, t: int, attempt: int, d: int, skew_c: float | None = None) -> np.ndarray:
    """Replacement float32 row for token t (attempt >= 1), before storage rounding."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, STREAM_REDRAW, t, attempt])))
    z = g.standard_normal(d, dtype=np.float32)
    if skew_c is None:
        return z
    u = skew_direction(seed, d)
    return (z.astype(np.float64) + skew_c * u).astype(np.float32)


def make_tokens(T: int, d: int, E: int, dtype: str, seed: int,
                skew_c: float | None = None, redraws=None):
    """(x [T][d], w_gate [E][d]) as CPU tensors; ``redraws`` = [(t, attempt), ...]."""
    x = _token_rows_f32(seed, T, d, skew_c)
    for t, attempt in (redraws or []):
        if attempt > 0:
            x[t] = redraw_token_row(seed, t, attempt, d, skew_c)
    wg = _gate_f32(seed, E, d, skew_c is not None)
    return _store(x, dtype), _store(wg, dtype)


def make_token_stream(B: int, S: int, d: int, rho: float, seed: int, dtype: str = "bf16") -> torch.Tensor:
    """Decode-time token stream: x [S][B][d], B independent sequences of S steps whose consecutive rows
    are correlated, so that the router's choices of consecutive tokens repeat more often than chance.

    Each sequence is a first-order autoregression in float64, rounded once to the stored type:
    x_0 = z_0, x_s = rho * x_{s-1} + sqrt(1 - rho^2) * z_s with z ~ N(0, 1) i.i.d. (its own stream), so
    every row is N(0, 1) like the layer workloads' tokens and the correlation of rows s and s+1 is rho
    (rho = 0: independent tokens). The value of rho that matches the pages' locality figures is
    decided by a calibration script under tests/golden; this function only draws.
    """
    z = normal_f32(seed, STREAM_DECODE, S * B * d, 1.0).reshape(S, B, d).astype(np.float64)
    x = np.empty_like(z)
    x[0] = z[0]
    c = float(np.sqrt(max(0.0, 1.0 - rho * rho)))
    for i in range(1, S):
        x[i] = rho * x[i - 1] + c * z[i]
    return _store(x.astype(np.float32), dtype)


@dataclass
class Layer:
    T: int
    d: int
    ffn: int
    E: int
    dtype: str
    x: torch.Tensor
    w_gate: torch.Tensor
    w1: torch.Tensor
    w3: torch.Tensor
    w2: torch.Tensor
    meta: dict = field(default_factory=dict)


def make_layer(T: int, d: int, ffn: int, E: int = 8, dtype: str = "bf16", seed: int = 1,
               weight_seed: int | None = None, skew_c: float | None = None, redraws=None,
               weights=None, name: str = "custom") -> Layer:
    if weights is None:
        weights = make_weights(d, ffn, E, dtype, seed if weight_seed is None else weight_seed)
    x, wg = make_tokens(T, d, E, dtype, seed, skew_c, redraws)
    w1, w3, w2 = weights
    meta = dict(name=name, seed=seed, weight_seed=weight_seed, skew_c=skew_c,
                redraws=[list(r) for r in (redraws or [])])
    return Layer(T, d, ffn, E, dtype, x, wg, w1, w3, w2, meta)


# Decoder-block workloads (the MoE layer inside its Mixtral block): B sequences
# of S tokens. The Mixtral-shape block reuses the layer workloads' expert draw.
BLOCK_CONFIGS = {
    "small": dict(name="block_small_B2_S160", B=2, S=160, d=512, n_heads=4, n_kv_heads=2, ffn=512,
                  seed=5320, weight_seed=5321),
    "mixtral": dict(name="mixtral_block_prefill_B1_S4096", B=1, S=4096, d=4096, n_heads=32, n_kv_heads=8,
                    ffn=14336, seed=5322, weight_seed=5310),
}


def make_block(B: int, S: int, d: int, n_heads: int, n_kv_heads: int, ffn: int, E: int = 8, head_dim: int = 128,
               seed: int = 1, weight_seed: int | None = None, moe_weights=None) -> dict:
    """Inputs of one decoder block as bf16 CPU tensors.

    x [B*S][d] ~ N(0, 1) (the residual stream entering the block); RMSNorm
    gains ~ N(1, 0.1^2); wqkv [(n_heads + 2 n_kv_heads) head_dim][d] ~ N(0, 1/d);
    wo [d][n_heads head_dim] ~ N(0, 1/(n_heads head_dim)); the MoE layer's
    w_gate, w1, w3, w2 as ``make_layer`` draws them.
    """
    ws = seed if weight_seed is None else weight_seed
    T = B * S
    rows = (n_heads + 2 * n_kv_heads) * head_dim
    x = _store(normal_f32(seed, STREAM_X, T * d, 1.0), "bf16").view(T, d)
    w_gate = _store(normal_f32(seed, STREAM_WG, E * d, 1.0 / np.sqrt(d)), "bf16").view(E, d)
    g_attn = _store(1.0 + normal_f32(seed, STREAM_ATTN_NORM, d, 0.1), "bf16")
    g_ffn = _store(1.0 + normal_f32(seed, STREAM_FFN_NORM, d, 0.1), "bf16")
    wqkv = _store(normal_f32(ws, STREAM_WQKV, rows * d, 1.0 / np.sqrt(d)), "bf16").view(rows, d)
    wo = _store(normal_f32(ws, STREAM_WO, d * n_heads * head_dim, 1.0 / np.sqrt(n_heads * head_dim)),
                "bf16").view(d, n_heads * head_dim)
    w1, w3, w2 = moe_weights if moe_weights is not None else make_weights(d, ffn, E, "bf16", ws)
    return dict(x=x, attn_norm=g_attn, wqkv=wqkv, wo=wo, ffn_norm=g_ffn, w_gate=w_gate, w1=w1, w3=w3, w2=w2)


def make_block_config(name: str, moe_weights=None) -> dict:
    c = BLOCK_CONFIGS[name]
    return make_block(c["B"], c["S"], c["d"], c["n_heads"], c["n_kv_heads"], c["ffn"], seed=c["seed"],
                      weight_seed=c["weight_seed"], moe_weights=moe_weights)


def load_schedule(path: Path | None = None) -> dict:
    p = Path(path) if path is not None else SCHEDULE_PATH
    if not p.exists():
        return {}
    with open(p) as f:
        return json.load(f)


def make_config(k: int, weights=None, schedule: dict | None = None) -> Layer:
    """The named workload k (0..4), with its stored redraw list and skew constant."""
    c = dict(CONFIGS[k])
    sched = (schedule if schedule is not None else load_schedule()).get(str(k), {})
    seed = int(sched.get("seed", c["seed"]))
    skew_c = float(sched["skew_c"]) if (c["skew"] and "skew_c" in sched) else None
    if c["skew"] and skew_c is None:
        raise RuntimeError("skewed workload needs its calibrated constant in the input schedule")
    layer = make_layer(c["T"], c["d"], c["ffn"], c["E"], c["dtype"], seed=seed,
                       weight_seed=c["weight_seed"], skew_c=skew_c,
                       redraws=[tuple(r) for r in sched.get("redraws", [])],
                       weights=weights, name=c["name"])
    layer.meta.update(config=k, aux=c["aux"], skew=c["skew"])
    return layer
