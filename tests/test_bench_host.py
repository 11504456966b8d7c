"""Host logic of bench.py (CPU): the roofline arithmetic of the JSON line, the oracle sample that doubles as
the parity check, and the source digests that keep ncu traffic figures from outliving their kernel."""
import numpy as np

import bench


def test_tile_up_roofline_is_algorithmic_flops_over_launch_time():
    cfg = dict(T=16384, d=4096, ffn=14336, E=8)
    work = bench._algorithmic(cfg, [4096] * 8)
    assert work["up_flops"] == 2 * 16384 * 4 * 4096 * 14336          # 7.697 TFLOP per launch
    assert work["flops"] == 2 * 16384 * 6 * 4096 * 14336 + 2 * 16384 * 4096 * 8
    peaks = dict(hbm_gbs=6500.0, bf16_tflops=1750.0, bf16_tflops_sustained=1370.0, source="measured")
    r = bench.roofline_tile_up({"tile_up_swiglu": [20, 20 * 5.0]}, work, peaks)   # 5 ms per launch
    assert abs(r["achieved"] - work["up_flops"] / 5e-3 / 1e12) < 0.1
    assert abs(r["frac"] - r["achieved"] / 1750.0) < 1e-4
    assert abs(r["frac_of_sustained"] - r["achieved"] / 1370.0) < 1e-4
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"


def test_stream_up_roofline_counts_only_touched_experts():
    cfg = dict(T=16, d=4096, ffn=14336, E=8)
    work = bench._algorithmic(cfg, [5, 0, 7, 0, 0, 20, 0, 0])       # three experts have tokens
    assert work["touched"] == 3
    assert work["up_bytes"] == 3 * 2 * 4096 * 14336 * 2
    peaks = dict(hbm_gbs=6500.0, bf16_tflops=1750.0, bf16_tflops_sustained=1370.0, source="measured")
    r = bench.roofline_stream_up({"stream_up": [10, 1.0]}, work, peaks, read_gbs=7000.0)   # 0.1 ms per launch
    assert abs(r["achieved"] - work["up_bytes"] / 1e-4 / 1e9) < 0.1
    assert abs(r["frac_of_read_peak"] - r["achieved"] / 7000.0) < 1e-4
    assert r["bound"] == "hbm"


def test_oracle_sample_leads_with_the_rarest_experts_tokens():
    rng = np.random.default_rng(0)
    T = 1000
    idx = rng.integers(0, 6, size=(T, 2))          # experts 6 and 7 unused
    idx[17] = (6, 0)                               # expert 6 holds exactly tokens 17 and 400
    idx[400] = (2, 6)
    tokens, rare = bench._sample_tokens(idx, T, 10, seed=1)
    assert rare == 6
    assert tokens[:2] == [17, 400]
    assert len(tokens) == 10 and len(set(tokens)) == 10 and all(0 <= t < T for t in tokens)


def test_source_digests_follow_their_own_sources_only():
    src = (bench.CSRC / "libmoe.cu").read_text()
    for fn in ("run_pair_ffn", "run_ffn", "make_map", "pick_kslice"):
        text = bench._function_text(src, fn)
        assert text.split("(")[0].split()[-1] == fn and text.rstrip().endswith("}")
    assert bench._source_digest("tile_up_swiglu") == bench._source_digest("tile_down_scale")
    assert bench._source_digest("tile_up_swiglu") != bench._source_digest("stream_up")
    assert bench._profile_traffic("no_such_kernel", "mixtral_large_T16384_aux") is None


def test_tile_units_note_names_each_claiming_kernel():
    assert bench.tile_units_note(0).startswith("static")
    assert bench.tile_units_note(1) == "claimed from a counter: up"
    assert bench.tile_units_note(6) == "claimed from a counter: down, backward"
    assert bench.tile_units_note(7) == "claimed from a counter: up, down, backward"
