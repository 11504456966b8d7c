"""Throughput of the top-2 sparse MoE layer (Mixtral shape) on B300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

One step = one moe_layer_forward over one batch of synthetic tokens: router,
grouping, both expert GEMMs and the combine (plus the load-balancing statistics
f, P and L_aux for the T=16384 workload). Default workload: the large batch
(T=16384, d=4096, ffn=14336, 8 experts, top-2, bf16, with the statistics), the
largest single-GPU workload, bound by the dense bf16 tensor-core rate. The line
also carries, under "decode", the decode batch (T=16) through the same layer
weights, measured in the same process: it is bound by reading the touched
experts' weights from HBM. ``--config`` selects another of the named workloads.

Outside the timed regions the fp64 oracle runs on a bounded sample of the
workload's tokens: its rate is the line's "cpu_baseline", and its results check
the GPU's output of the timed steps ("parity": routing on every token, y on the
sampled tokens, the statistics).

Prints one JSON line (rank 0). For N > 1 every rank runs its own replica of
the workload on its own GPU (the layer has no exchange step in this data-parallel
form); value = tokens of all ranks / slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "MoE-layer tokens/s at Mixtral shape (bf16); % of BF16 TC peak / HBM BW"
UNIT = "tokens/s"
DEFAULT_CONFIG = 3
PROFILES = ROOT / "profiles"


def _peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0, source="fallback")


class _Nvml:
    """Minimal read-only NVML access through ctypes (libnvidia-ml ships with the driver)."""

    def __init__(self):
        import ctypes
        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def handle(self, cuda_index: int):
        c = self.c
        h = c.c_void_p()
        try:
            import torch
            p = torch.cuda.get_device_properties(cuda_index)
            bus = ("%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)).encode()
            if self.lib.nvmlDeviceGetHandleByPciBusId_v2(c.c_char_p(bus), c.byref(h)) == 0:
                return h
        except Exception:
            pass
        vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip().isdigit()]
        idx = int(vis[cuda_index]) if cuda_index < len(vis) else cuda_index
        if self.lib.nvmlDeviceGetHandleByIndex_v2(c.c_uint(idx), c.byref(h)) != 0:
            raise RuntimeError("no NVML handle")
        return h

    def sm_clock(self, h, max_clock=False) -> int:
        v = self.c.c_uint(0)
        f = self.lib.nvmlDeviceGetMaxClockInfo if max_clock else self.lib.nvmlDeviceGetClockInfo
        f(h, self.c.c_int(1), self.c.byref(v))  # NVML_CLOCK_SM = 1
        return int(v.value)

    def reasons(self, h) -> int:
        v = self.c.c_ulonglong(0)
        self._reasons(h, self.c.byref(v))
        return int(v.value)


class ClockSampler:
    """Samples SM clock and clock-event reasons (NVML, read-only) during the timed region."""

    REASONS = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
        0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
        0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
    }

    def __init__(self, cuda_index: int, period_s: float = 0.002):
        self.period = period_s
        self.samples, self.reasons = [], set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self.ok = False
        try:
            self.nvml = _Nvml()
            self.h = self.nvml.handle(cuda_index)
            self.max_mhz = self.nvml.sm_clock(self.h, max_clock=True)
            self.ok = True
        except Exception as exc:  # pragma: no cover - reported in the JSON line
            self.error = repr(exc)

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nvml.sm_clock(self.h))
                mask = self.nvml.reasons(self.h)
                for bit, name in self.REASONS.items():
                    if mask & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()

    def summary(self) -> dict:
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "error": getattr(self, "error", "")}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons - {"gpu_idle"}), "samples": len(self.samples)}


CSRC = ROOT / "sparse_mixture_experts_53_b300" / "csrc"


# The sources that define each profiled kernel and its launch: its own file, the shared device helpers and
# the launch functions in the ABI file (ncu figures go stale when any of them changes, not when another
# kernel or another launch does).
KERNEL_SOURCES = {
    "tile_up_swiglu": (("ffn_tc.cuh", "common.cuh"), ("run_pair_ffn", "make_map", "pair_capacity", "pair_grid")),
    "tile_down_scale": (("ffn_tc.cuh", "common.cuh"), ("run_pair_ffn", "make_map", "pair_capacity", "pair_grid")),
    "stream_up": (("ffn_tc.cuh", "common.cuh"), ("run_ffn", "make_map", "pick_kslice", "ffn_layout")),
}


def _function_text(src: str, name: str) -> str:
    """The definition of a top-level function of a C++ source: from its signature line to the closing brace
    at column 0."""
    import re
    m = re.search(r"^[^\n]*\b" + re.escape(name) + r"\(", src, re.M)
    if m is None:
        return ""
    end = src.find("\n}\n", m.start())
    return src[m.start():end + 3 if end >= 0 else len(src)]


def _source_digest(kernel: str) -> str:
    files, functions = KERNEL_SOURCES[kernel]
    h = hashlib.sha256()
    for name in files:
        h.update(name.encode())
        h.update((CSRC / name).read_bytes())
    abi = (CSRC / "libmoe.cu").read_text()
    for fn in functions:
        h.update(fn.encode())
        h.update(_function_text(abi, fn).encode())
    return h.hexdigest()[:16]


def _profile_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current source."""
    f = PROFILES / f"{kernel}__{workload}.json"
    if not f.exists():
        return None
    try:
        d = json.loads(f.read_text())
    except Exception:
        return None
    if kernel not in KERNEL_SOURCES or d.get("source_digest") != _source_digest(kernel):
        return None
    return d.get("dram_bytes_per_launch")


def _dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class Ranks:
    """The replicas of a multi-GPU run: one process per GPU, no exchange on the data path.

    Only two collectives exist, both outside the layer: a barrier around each
    timed region and the max over ranks of the measured times (the slowest
    replica sets the job's time). With one rank both are local no-ops.
    """

    def __init__(self, rank: int, world: int, local: int, backend: str = "nccl"):
        self.rank, self.world, self.backend = rank, world, backend
        self.dist = None
        if world > 1:
            import torch
            import torch.distributed as dist
            kw = {"device_id": torch.device("cuda", local)} if backend == "nccl" else {}
            dist.init_process_group(backend, rank=rank, world_size=world, **kw)
            self.dist = dist

    def _device(self):
        return "cuda" if self.backend == "nccl" else "cpu"

    def barrier(self) -> None:
        if self.dist is not None:
            self.dist.barrier()

    def max(self, values: list[float]) -> list[float]:
        if self.dist is None:
            return [float(v) for v in values]
        import torch
        t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=self._device())
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return [float(v) for v in t.cpu().tolist()]

    def close(self) -> None:
        if self.dist is not None:
            self.dist.destroy_process_group()
            self.dist = None


def throughput(tokens_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job tokens/s: the tokens of every replica over the slowest replica's step time."""
    return round(tokens_per_rank * world / (ms_max * 1e-3), 1)


def _algorithmic(cfg: dict, counts) -> dict:
    """Work of one step from the per-expert row counts (the router's decision)."""
    T, d, F = cfg["T"], cfg["d"], cfg["ffn"]
    touched = int(sum(1 for c in counts if c > 0))
    flops = 2 * T * 6 * d * F + 2 * T * d * cfg["E"]
    w_bytes = touched * 3 * d * F * 2
    return dict(touched=touched, flops=flops, weight_bytes=w_bytes,
                up_bytes=touched * 2 * d * F * 2, down_bytes=touched * d * F * 2,
                up_flops=2 * T * 4 * d * F, down_flops=2 * T * 2 * d * F,
                act_bytes=T * d * 2 * 2)


def _device_status_ok(moe, when: str) -> None:
    code, detail = moe.moe_get_device_status()
    if code != moe.MOE_OK:
        raise RuntimeError(f"device status {when}: {moe.status_string(code)} ({detail})")


def read_peak_gbs(moe, stream, nbytes: int = 4 << 30, reps: int = 10) -> float:
    """HBM read rate of this GPU: the library's read probe over a buffer 32x the L2, best of `reps` (CUDA
    events). The weight-streaming kernels only read, so this, not a copy, is their ceiling."""
    import torch
    buf = torch.ones(nbytes, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        moe.moe_read_probe(buf, sink, stream)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    best = float("inf")
    for _ in range(reps):
        a.record(stream)
        moe.moe_read_probe(buf, sink, stream)
        b.record(stream)
        b.synchronize()
        best = min(best, a.elapsed_time(b))
    del buf
    return round(nbytes / (best * 1e-3) / 1e9, 1)


def measure_layer(moe, L, cfg: dict, args, ranks, stream, x_dev=None, weights=None, e2e: bool = True) -> dict:
    """One workload through moe_layer_forward: the timed steps (device-resident inputs, clocks sampled), a
    second pass with serialised launches and CUDA events around every kernel, the end-to-end steps through
    the same call with host buffers, and the routing counts of the batch."""
    import torch

    def barrier():
        ranks.barrier()
        torch.cuda.synchronize()

    aux = bool(cfg["aux"])
    x = L.x.cuda() if x_dev is None else x_dev
    wg = L.w_gate.cuda()
    w1, w3, w2 = weights if weights is not None else (L.w1.cuda(), L.w3.cuda(), L.w2.cuda())
    shape = moe.shape_of(x, w1)
    ws = moe.workspace(shape)
    y = torch.empty_like(x)
    stats = (torch.empty(8, device="cuda"), torch.empty(8, device="cuda"), torch.empty(1, device="cuda")) if aux \
        else None

    def step():
        moe.moe_layer_forward(shape, x, wg, w1, w3, w2, y, ws, stats, stream)

    for _ in range(args.warmup):
        step()
    _device_status_ok(moe, "after warm-up")

    # ---- timed region: device-resident inputs, programmatic dependent launch as configured
    sampler = ClockSampler(torch.cuda.current_device())
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with sampler:
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        barrier()
    ms = start.elapsed_time(stop) / args.steps
    _device_status_ok(moe, "after timing")
    y_out = y.clone()
    stats_out = tuple(t.clone() for t in stats) if aux else None

    # ---- per-kernel times: the same steps with serialised launches (an early-launched kernel's events
    # would include its wait for the predecessor), CUDA events around every launch on the launching stream
    moe.moe_set_knob(moe.MOE_KNOB_PDL, 0)
    moe.moe_timing_enable(True)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    serial_ms = a.elapsed_time(b) / args.steps
    kern = moe.moe_timing_read()
    moe.moe_timing_enable(False)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, args.pdl)

    out = dict(ms=ms, serial_ms=serial_ms, kern=kern, clocks=sampler.summary(), y=y_out, stats=stats_out,
               shape=shape, x=x, wg=wg)

    if e2e:
        # ---- end to end through the public call with host buffers: every step copies its tokens in from
        # pinned host memory and reads its output back. Input and output copies run on their own streams
        # (both directions of the link at once) with two device buffers each way, so step i+1's input copy
        # and step i's output copy overlap neighbouring steps' kernels, as a serving loop would run them.
        x_host = L.x.pin_memory()
        y_host = [torch.empty_like(L.x).pin_memory() for _ in range(2)]
        xb = [torch.empty_like(x) for _ in range(2)]
        yb = [torch.empty_like(x) for _ in range(2)]
        cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
        h2d = [torch.cuda.Event() for _ in range(2)]
        comp = [torch.cuda.Event() for _ in range(2)]
        d2h = [torch.cuda.Event() for _ in range(2)]

        def e2e_steps(n):
            for i in range(n):
                bb = i & 1
                with torch.cuda.stream(cin):
                    if i >= 2:
                        cin.wait_event(comp[bb])  # xb[bb] is free once step i-2 has run
                    xb[bb].copy_(x_host, non_blocking=True)
                    h2d[bb].record(cin)
                stream.wait_event(h2d[bb])
                if i >= 2:
                    stream.wait_event(d2h[bb])  # yb[bb] has been read back
                moe.moe_layer_forward(shape, xb[bb], wg, w1, w3, w2, yb[bb], ws, stats, stream)
                comp[bb].record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(comp[bb])
                    y_host[bb].copy_(yb[bb], non_blocking=True)
                    d2h[bb].record(cout)
            stream.wait_stream(cout)

        e2e_steps(3)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        cin.wait_stream(stream)
        cout.wait_stream(stream)
        e2e_steps(args.steps)
        e1.record(stream)
        barrier()
        out["e2e_ms"] = e0.elapsed_time(e1) / args.steps
        out["io_bytes"] = int(L.x.numel() * L.x.element_size())
        out["y_host_equal"] = bool(torch.equal(y_host[(args.steps - 1) & 1], y_out.cpu()))

    # routing of this batch (read once, outside every timed region)
    idx = torch.empty((L.T, 2), dtype=torch.int32, device="cuda")
    gw = torch.empty((L.T, 2), dtype=torch.float32, device="cuda")
    moe.moe_route_top2(shape, x, wg, idx, gw)
    out["idx"] = idx.cpu()
    out["counts"] = torch.bincount(idx.flatten().long(), minlength=8).cpu().tolist()
    _device_status_ok(moe, "after the end-to-end steps")
    return out


def _kernel_ms(kern: dict, name: str) -> float:
    per = kern.get(name, [1, float("nan")])
    return per[1] / max(1, per[0])


def roofline_tile_up(kern: dict, work: dict, peaks: dict) -> dict:
    """Dominant kernel of a token-tile step: the up projection (2/3 of the FLOPs), against the dense bf16
    peak (burst; the sustained figure beside it)."""
    dom_ms = _kernel_ms(kern, "tile_up_swiglu")
    achieved = work["up_flops"] / (dom_ms * 1e-3) / 1e12
    return {"kernel": "tile_up_swiglu", "bound": "tensor", "achieved": round(achieved, 1),
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
            "peak_source": peaks["source"] + " (burst)",
            "frac_of_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4),
            "algorithmic_flops_per_launch": work["up_flops"], "launch_ms": round(dom_ms, 5)}


def roofline_stream_up(kern: dict, work: dict, peaks: dict, read_gbs: float | None) -> dict:
    """Dominant kernel of a decode step: the up projection's weight streaming, against HBM."""
    dom_ms = _kernel_ms(kern, "stream_up")
    achieved = work["up_bytes"] / (dom_ms * 1e-3) / 1e9
    r = {"kernel": "stream_up", "bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"] + " (copy)",
         "algorithmic_bytes_per_launch": work["up_bytes"], "launch_ms": round(dom_ms, 5)}
    if read_gbs:
        r.update(read_peak=read_gbs, frac_of_read_peak=round(achieved / read_gbs, 4),
                 read_peak_source="moe_read_probe over 4 GiB, best of 10")
    return r


def run_ours(args, rank, world, local) -> dict | None:
    import torch

    from moe_inputs import CONFIGS, make_config
    from sparse_mixture_experts_53_b300 import moe

    torch.cuda.set_device(local)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, args.pdl)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, args.tile_ctas)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, args.tile_sched)
    ranks = Ranks(rank, world, local, backend="nccl")
    stream = torch.cuda.current_stream()

    k = args.config
    cfg = CONFIGS[k]
    t0 = time.time()
    L = make_config(k)
    gen_s = time.time() - t0
    weights = (L.w1.cuda(), L.w3.cuda(), L.w2.cuda())
    m = measure_layer(moe, L, cfg, args, ranks, stream, weights=weights)
    ms, e2e_ms = ranks.max([m["ms"], m["e2e_ms"]])

    peaks = _peaks()
    read_gbs = read_peak_gbs(moe, stream) if rank == 0 else None
    work = _algorithmic(cfg, m["counts"])
    kern = m["kern"]
    streaming = cfg["T"] <= 64
    roof = roofline_stream_up(kern, work, peaks, read_gbs) if streaming else roofline_tile_up(kern, work, peaks)
    roof["traffic"] = _profile_traffic(roof["kernel"], cfg["name"])
    roof["timing"] = "CUDA events around each launch on its stream, launches serialised, over the timed steps"
    step_s = ms * 1e-3
    aux = bool(cfg["aux"])
    line = {
        "metric": METRIC, "value": throughput(cfg["T"], world, ms), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded Mixtral-shape tensors, random init)",
        "config": {"workload": cfg["name"], "T": cfg["T"], "d": cfg["d"], "ffn": cfg["ffn"], "E": cfg["E"], "k": 2,
                   "aux_stats": aux, "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "ffn_path": "weight-streaming (swap-AB)" if streaming else
                   ("token tiles 256x256 on CTA pairs" if args.tile_ctas == 2 or (args.tile_ctas == 0 and cfg["T"] > 384)
                    else "token tiles 128x256"),
                   "pdl": bool(args.pdl), "tile_units": tile_units_note(args.tile_sched),
                   "l2": "inputs larger than L2: each step reads %.2f GB of expert weights" % (work["weight_bytes"] / 1e9),
                   "experts_touched": work["touched"], "input_gen_s": round(gen_s, 1)},
        "step": {"tflops": round(work["flops"] / step_s / 1e12, 2),
                 "frac_bf16_burst": round(work["flops"] / step_s / 1e12 / peaks["bf16_tflops"], 4),
                 "frac_bf16_sustained": round(work["flops"] / step_s / 1e12 / peaks["bf16_tflops_sustained"], 4),
                 "weight_gbs": round(work["weight_bytes"] / step_s / 1e9, 1),
                 "frac_hbm": round(work["weight_bytes"] / step_s / 1e9 / peaks["hbm_gbs"], 4)},
        "roofline": roof,
        "kernels_ms_per_step": {n: round(v[1] / max(1, args.steps), 5) for n, v in kern.items()},
        "kernels_timing": {"ms_per_step_serialised": round(m["serial_ms"], 5),
                           "how": "second pass over the same steps with programmatic dependent launch off and "
                                  "CUDA events around every launch; the kernels' sum is within that pass's step"},
        "gpu_launches": int(sum(v[0] for v in kern.values())),
        "e2e": {"value": throughput(cfg["T"], world, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": m["io_bytes"], "d2h_bytes_per_step": m["io_bytes"],
                "ms_per_step": round(e2e_ms, 5), "output_read_back_equals_device_output": m["y_host_equal"],
                "copies": "pinned host buffers; input and output copies on two streams overlap neighbouring steps"},
        "clocks": m["clocks"],
    }
    gpu_out = {"cfg": k, "y": m["y"].cpu(), "idx": m["idx"], "stats": [t.cpu() for t in m["stats"]] if aux else None}
    del m

    if not args.no_decode and k != 1:
        # the decode batch through the same layer (configs 1-4 share one weight draw), same process
        c1 = CONFIGS[1]
        L1 = make_config(1, weights=(L.w1, L.w3, L.w2))
        d = measure_layer(moe, L1, c1, args, ranks, stream, weights=weights)
        dms, de2e = ranks.max([d["ms"], d["e2e_ms"]])
        dwork = _algorithmic(c1, d["counts"])
        droof = roofline_stream_up(d["kern"], dwork, peaks, read_gbs)
        droof["traffic"] = _profile_traffic("stream_up", c1["name"])
        line["decode"] = {
            "workload": c1["name"], "value": throughput(c1["T"], world, dms), "unit": UNIT,
            "ms_per_step": round(dms, 5),
            "weight_gbs": round(dwork["weight_bytes"] / (dms * 1e-3) / 1e9, 1),
            "frac_hbm_copy_peak": round(dwork["weight_bytes"] / (dms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "frac_hbm_read_peak": round(dwork["weight_bytes"] / (dms * 1e-3) / 1e9 / read_gbs, 4) if read_gbs else None,
            "experts_touched": dwork["touched"], "roofline": droof,
            "kernels_ms_per_step": {n: round(v[1] / max(1, args.steps), 5) for n, v in d["kern"].items()},
            "kernels_ms_per_step_serialised": round(d["serial_ms"], 5),
            "e2e": {"value": throughput(c1["T"], world, de2e), "unit": UNIT, "h2d_bytes_per_step": d["io_bytes"],
                    "d2h_bytes_per_step": d["io_bytes"], "ms_per_step": round(de2e, 5)},
            "clocks": d["clocks"]}
        line["decode"]["gpu_launches"] = int(sum(v[0] for v in d["kern"].values()))
        gpu_out["decode"] = {"cfg": 1, "y": d["y"].cpu(), "idx": d["idx"]}
        del d
    ranks.close()
    if rank != 0:
        return None
    line["_gpu_out"] = gpu_out
    return line


TRAIN_GEMM_FLOPS = {  # multiples of R*d*ffn (R = 2T slot rows) per launch
    "tile_up_swiglu": 4, "tile_down_scale": 2, "bwd_dh_swiglu": 2, "bwd_dx": 4, "bwd_dw2": 2, "bwd_dw13": 4,
}


def tile_units_note(sched: int) -> str:
    """How the CTA-pair kernels took their units (MOE_KNOB_TILE_SCHED)."""
    if sched == 0:
        return "static: pair p takes units p, p + pairs, ..."
    return "claimed from a counter: " + ", ".join(n for b, n in ((1, "up"), (2, "down"), (4, "backward")) if sched & b)


def run_training(args) -> dict:
    """One training step of the layer: forward that keeps its state, then the backward pass."""
    import torch

    from moe_inputs import CONFIGS, make_config
    from sparse_mixture_experts_53_b300 import moe

    torch.cuda.set_device(0)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, args.pdl)
    moe.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, args.tile_sched)
    k = args.config
    cfg = CONFIGS[k]
    L = make_config(k)
    x = L.x.cuda()
    wg, w1, w3, w2 = L.w_gate.cuda(), L.w1.cuda(), L.w3.cuda(), L.w2.cuda()
    dy = torch.randn(x.shape, generator=torch.Generator().manual_seed(7)).to(torch.bfloat16).cuda()
    shape = moe.shape_of(x, w1)
    state = torch.empty(moe.moe_train_state_bytes(shape), dtype=torch.uint8, device="cuda")
    ws = torch.empty(moe.moe_backward_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    dx = torch.empty_like(x)
    f32 = dict(dtype=torch.float32, device="cuda")
    dwg, dw1, dw3, dw2 = (torch.empty(t.shape, **f32) for t in (wg, w1, w3, w2))
    aux_coef = 0.01 if cfg["aux"] else 0.0
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_layer_forward_train(shape, x, wg, w1, w3, w2, y, state, None, stream)
        moe.moe_layer_backward(shape, x, wg, w1, w3, w2, dy, aux_coef, state, dx, dwg, dw1, dw3, dw2, ws, stream)

    for _ in range(args.warmup):
        step()
    code, detail = moe.moe_get_device_status()
    if code != moe.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {moe.status_string(code)} ({detail})")
    sampler = ClockSampler(0)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with sampler:
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    moe.moe_timing_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    kern = moe.moe_timing_read()
    moe.moe_timing_enable(False)
    code, detail = moe.moe_get_device_status()
    if code != moe.MOE_OK:
        raise RuntimeError(f"device status after timing: {moe.status_string(code)} ({detail})")
    T, d, F = cfg["T"], cfg["d"], cfg["ffn"]
    R = 2 * T
    peaks = _peaks()
    per = {n: (v[1] / v[0]) for n, v in kern.items()}
    gemms = {n: per[n] for n in TRAIN_GEMM_FLOPS if n in per}
    dom = max(gemms, key=gemms.get)
    achieved = TRAIN_GEMM_FLOPS[dom] * R * d * F / (per[dom] * 1e-3) / 1e12
    flops = 18 * R * d * F
    return {
        "metric": "MoE-layer training tokens/s (forward + backward) at Mixtral shape (bf16)", "pass": "forward+backward",
        "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (seeded Mixtral-shape tensors, random init)",
        "config": {"workload": cfg["name"], "T": T, "d": d, "ffn": F, "E": cfg["E"], "k": 2, "aux_coef": aux_coef},
        "step": {"tflops": round(flops / (ms * 1e-3) / 1e12, 2),
                 "frac_bf16": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)},
        "roofline": {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                     "peak_source": peaks["source"] + " (burst)", "launch_ms": round(per[dom], 5)},
        "kernels_ms_per_step": {n: round(v[1] / max(1, args.steps), 5) for n, v in kern.items()},
        "gpu_launches": int(sum(v[0] for v in kern.values())),
        "clocks": sampler.summary(),
    }


def run_block(args) -> dict:
    """The decoder block around the layer (RMSNorm, Q/K/V projection, RoPE, causal GQA attention, Wo,
    residual + RMSNorm, the MoE layer, residual) at the Mixtral shape, one 4096-token sequence."""
    import torch

    from moe_inputs import BLOCK_CONFIGS, make_block_config
    from sparse_mixture_experts_53_b300 import moe

    torch.cuda.set_device(0)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, args.pdl)
    c = BLOCK_CONFIGS["mixtral"]
    p = {k: v.cuda() for k, v in make_block_config("mixtral").items()}
    B, S, d, Hq, Hkv, F = c["B"], c["S"], c["d"], c["n_heads"], c["n_kv_heads"], c["ffn"]
    hd = 128
    shape = moe.make_block_shape(B, S, d, Hq, Hkv, F)
    ws = torch.empty(moe.moe_block_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    wts = moe.block_weights(p)
    out = torch.empty_like(p["x"])
    stream = torch.cuda.current_stream()
    T = B * S

    def step():
        moe.moe_block_forward(shape, p["x"], wts, out, ws, stream=stream)

    for _ in range(args.warmup):
        step()
    code, detail = moe.moe_get_device_status()
    if code != moe.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {moe.status_string(code)} ({detail})")
    sampler = ClockSampler(0)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with sampler:
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    # per-kernel times with serialised launches (an early-launched kernel's events would include its wait)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, 0)
    moe.moe_timing_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    kern = moe.moe_timing_read()
    moe.moe_timing_enable(False)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, args.pdl)
    # the attention kernel alone, back to back, on the shapes of the block's q, k, v
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn((T, Hq * hd), device="cuda", generator=g).to(torch.bfloat16)
    kk = torch.randn((T, Hkv * hd), device="cuda", generator=g).to(torch.bfloat16)
    vv = torch.randn((T, Hkv * hd), device="cuda", generator=g).to(torch.bfloat16)
    oo = torch.empty_like(q)
    for _ in range(3):
        moe.moe_attention(shape, q, kk, vv, oo, stream)
    n_att = 50
    a.record(stream)
    for _ in range(n_att):
        moe.moe_attention(shape, q, kk, vv, oo, stream)
    b.record(stream)
    torch.cuda.synchronize()
    att_ms = a.elapsed_time(b) / n_att
    code, detail = moe.moe_get_device_status()
    if code != moe.MOE_OK:
        raise RuntimeError(f"device status after timing: {moe.status_string(code)} ({detail})")
    per = {n: v[1] / v[0] for n, v in kern.items()}
    peaks = _peaks()
    flops = {
        "linear_qkv": 2.0 * T * d * (Hq + 2 * Hkv) * hd,
        "attention": 4.0 * hd * Hq * B * S * (S + 1) / 2,   # causal: each query against the keys up to it
        "linear_o": 2.0 * T * Hq * hd * d,
        "moe": 6.0 * 2 * T * d * F,
    }
    total = sum(flops.values())

    def tf(name):
        return round(flops[name] / (per[name] * 1e-3) / 1e12, 1) if name in per else None

    dom = max(per, key=per.get)
    up = "tile_up_swiglu"
    up_tf = 4.0 * 2 * T * d * F / (per[up] * 1e-3) / 1e12
    return {
        "metric": "Mixtral decoder-block tokens/s (attention + MoE layer, bf16)", "value": round(T / (ms * 1e-3), 1),
        "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "dtype": "bf16", "data": "synthetic (seeded Mixtral-shape block, random init)",
        "config": {"workload": c["name"], "B": B, "S": S, "d": d, "n_heads": Hq, "n_kv_heads": Hkv,
                   "head_dim": hd, "ffn": F, "E": 8, "k": 2},
        "step": {"tflops": round(total / (ms * 1e-3) / 1e12, 1),
                 "frac_bf16": round(total / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4)},
        "roofline": {"kernel": up, "bound": "tensor", "achieved": round(up_tf, 1), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(up_tf / peaks["bf16_tflops"], 4),
                     "peak_source": peaks["source"] + " (burst)", "launch_ms": round(per[up], 5)},
        "attention": {"bound": "tensor", "launch_ms": round(att_ms, 5),
                      "achieved": round(flops["attention"] / (att_ms * 1e-3) / 1e12, 1), "peak": peaks["bf16_tflops"],
                      "unit": "TFLOP/s",
                      "frac": round(flops["attention"] / (att_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                      "peak_source": peaks["source"] + " (burst)",
                      "timing": "50 launches back to back on seeded q, k, v of the block's shapes"},
        "projections_tflops": {"linear_qkv": tf("linear_qkv"), "linear_o": tf("linear_o")},
        "longest_kernel": dom,
        "kernels_ms_per_step": {n: round(v[1] / max(1, args.steps), 5) for n, v in kern.items()},
        "kernels_timing": "CUDA events around each launch, launches serialised (no programmatic dependent launch)",
        "gpu_launches": int(sum(v[0] for v in kern.values())),
        "clocks": sampler.summary(),
    }


def run_block_decode(args) -> dict:
    """One decode step of the Mixtral decoder block: 16 sequences, one new token each, against key/value
    caches holding 4096 earlier tokens (seeded values) -- the block around the decode batch of the layer."""
    import torch

    from moe_inputs import CONFIGS, make_block, make_weights
    from sparse_mixture_experts_53_b300 import moe

    torch.cuda.set_device(0)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, args.pdl)
    B, L, d, Hq, Hkv, F, hd = 16, 4096, 4096, 32, 8, 14336, 128
    cfg = CONFIGS[1]
    experts = make_weights(d, F, 8, "bf16", cfg["weight_seed"])
    p = {k: v.cuda() for k, v in make_block(B, 1, d, Hq, Hkv, F, seed=5350, weight_seed=5310,
                                            moe_weights=experts).items()}
    del experts
    cmax = L + args.warmup + 2 * args.steps + 8
    shape = moe.make_block_shape(B, 1, d, Hq, Hkv, F, cache_max=cmax)
    g = torch.Generator(device="cuda").manual_seed(5351)
    kc = torch.randn((B, Hkv, cmax, hd), device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn((B, Hkv, cmax, hd), device="cuda", generator=g).to(torch.bfloat16)
    clen = torch.full((B,), L, dtype=torch.int32, device="cuda")
    ws = torch.empty(moe.moe_block_decode_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    wts = moe.block_weights(p)
    out = torch.empty_like(p["x"])
    stream = torch.cuda.current_stream()

    def step():
        moe.moe_block_decode(shape, p["x"], wts, kc, vc, clen, out, ws, stream)

    for _ in range(args.warmup):
        step()
    code, detail = moe.moe_get_device_status()
    if code != moe.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {moe.status_string(code)} ({detail})")
    sampler = ClockSampler(0)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ctx0 = int(clen[0].item())
    torch.cuda.synchronize()
    with sampler:
        a.record(stream)
        for _ in range(args.steps):
            step()
        b.record(stream)
        torch.cuda.synchronize()
    ms = a.elapsed_time(b) / args.steps
    moe.moe_set_knob(moe.MOE_KNOB_PDL, 0)
    moe.moe_timing_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    kern = moe.moe_timing_read()
    moe.moe_timing_enable(False)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, args.pdl)
    code, detail = moe.moe_get_device_status()
    if code != moe.MOE_OK:
        raise RuntimeError(f"device status after timing: {moe.status_string(code)} ({detail})")
    per = {n: v[1] / v[0] for n, v in kern.items()}
    peaks = _peaks()
    ctx = ctx0 + args.steps // 2 + 1                   # keys per sequence, middle of the timed steps
    cache_bytes = 2.0 * B * ctx * Hkv * hd * 2         # keys and values read once
    att_ms = per.get("attention_decode", 0.0)
    return {
        "metric": "Mixtral decoder-block decode tokens/s (16 sequences, 4096-token caches, bf16)",
        "value": round(B / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic (seeded Mixtral-shape block and cache values, random init)",
        "config": {"workload": "mixtral_block_decode_B16_ctx4096", "B": B, "context": L, "d": d, "n_heads": Hq,
                   "n_kv_heads": Hkv, "head_dim": hd, "ffn": F, "E": 8, "k": 2},
        "attention_decode": {"bound": "hbm", "launch_ms": round(att_ms, 5),
                             "achieved": round(cache_bytes / (att_ms * 1e-3) / 1e9, 1) if att_ms else None,
                             "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": round(cache_bytes / (att_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)
                             if att_ms else None,
                             "bytes": cache_bytes},
        "kernels_ms_per_step": {n: round(v[1] / max(1, args.steps), 5) for n, v in kern.items()},
        "kernels_timing": "CUDA events around each launch, launches serialised (no programmatic dependent launch)",
        "gpu_launches": int(sum(v[0] for v in kern.values())),
        "clocks": sampler.summary(),
    }


def run_decode_loop(args) -> dict:
    """Decode-time expert cache (measured experiment): one decode step per sequence of a token stream
    whose consecutive tokens share experts at the lecture page's rate, through one Mixtral-shape layer or
    through 32 layers (distinct weight copies, as a model's MoE layers), with and without the weight-
    streaming path keeping part of each call's expert weights in L2 for the next call."""
    import torch

    from moe_inputs import CONFIGS, make_token_stream, make_tokens, make_weights
    from sparse_mixture_experts_53_b300 import moe

    torch.cuda.set_device(0)
    moe.moe_set_knob(moe.MOE_KNOB_PDL, args.pdl)
    sched = json.loads((ROOT / "tests" / "golden" / "locality_schedule.json").read_text())
    c = CONFIGS[1]
    d, F, E = c["d"], c["ffn"], c["E"]
    w_host = make_weights(d, F, E, c["dtype"], c["weight_seed"])
    _, wg_host = make_tokens(1, d, E, c["dtype"], c["seed"])
    wg = wg_host.cuda()
    layers_max = 32
    base = tuple(w.cuda() for w in w_host)
    del w_host
    weights = [base] + [tuple(w.clone() for w in base) for _ in range(layers_max - 1)]
    stream = torch.cuda.current_stream()
    Bmax = 4
    streams = {"locality": float(sched["rho"]), "independent": 0.0}
    n_steps = {1: 64, 32: 12}
    warm = 4
    xs = {name: make_token_stream(Bmax, n_steps[1] + warm, d, rho, sched["seed"]).cuda()
          for name, rho in streams.items()}
    ws = moe.workspace(moe.make_shape(Bmax, d, F, moe.MOE_BF16))
    y = torch.empty((Bmax, d), dtype=torch.bfloat16, device="cuda")
    keep_mb = [0, 32, 64, 96]
    results = []
    sampler = ClockSampler(0)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The evict-last priority may only take hold inside the L2 portion that the context sets aside for
    # persisting lines (0 unless the application asks for it). This experiment, as an application would,
    # runs the matrix once as found and once with that context limit raised to the device's maximum;
    # the limit belongs to this process's context and is put back before the end.
    from cuda.bindings import runtime as rt
    err, limit0 = rt.cudaDeviceGetLimit(rt.cudaLimit.cudaLimitPersistingL2CacheSize)
    err2, prop = rt.cudaGetDeviceProperties(0)
    set_asides = [int(limit0)]
    if err == rt.cudaError_t.cudaSuccess and err2 == rt.cudaError_t.cudaSuccess and prop.persistingL2CacheMaxSize > 0:
        set_asides.append(int(prop.persistingL2CacheMaxSize))
    with sampler:
        for aside in set_asides:
            rt.cudaDeviceSetLimit(rt.cudaLimit.cudaLimitPersistingL2CacheSize, aside)
            rt.cudaCtxResetPersistingL2Cache()
            for B in (1, 2, 4):
                shape = moe.make_shape(B, d, F, moe.MOE_BF16)
                for sname, x in xs.items():
                    for L in (1, 32):
                        S = n_steps[L]
                        row = {"B": B, "stream": sname, "layers": L, "steps": S,
                               "l2_set_aside_MB": round(aside / 2**20, 1)}
                        for kmb in keep_mb:
                            moe.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, kmb * 1024)

                            def run(s0, n):
                                for s in range(s0, s0 + n):
                                    for l in range(L):
                                        w1, w3, w2 = weights[l]
                                        moe.moe_layer_forward(shape, x[s, :B], wg, w1, w3, w2, y[:B], ws, None, stream)

                            run(0, warm)
                            torch.cuda.synchronize()
                            a.record(stream)
                            run(warm, S)
                            b.record(stream)
                            b.synchronize()
                            row[f"us_per_layer_step_keep{kmb}MB"] = round(a.elapsed_time(b) * 1e3 / (S * L), 2)
                        moe.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, 0)
                        t0 = row["us_per_layer_step_keep0MB"]
                        row["best_gain"] = round(t0 / min(row[f"us_per_layer_step_keep{k}MB"] for k in keep_mb) - 1, 4)
                        results.append(row)
    rt.cudaCtxResetPersistingL2Cache()
    rt.cudaDeviceSetLimit(rt.cudaLimit.cudaLimitPersistingL2CacheSize, int(limit0))
    moe.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, 0)
    _device_status_ok(moe, "after the decode loop")
    # experts touched per step on the locality stream (routing read once, outside the timed loops)
    touched = {}
    for B in (1, 2, 4):
        shape = moe.make_shape(B, d, F, moe.MOE_BF16)
        idx = torch.empty((B, 2), dtype=torch.int32, device="cuda")
        gw = torch.empty((B, 2), dtype=torch.float32, device="cuda")
        sets = []
        for s in range(warm, warm + n_steps[1]):
            moe.moe_route_top2(shape, xs["locality"][s, :B], wg, idx, gw)
            sets.append(set(idx.flatten().tolist()))
        touched[B] = {"experts_per_step": round(sum(len(t) for t in sets) / len(sets), 3),
                      "reused_from_previous_step": round(sum(len(p & q) for p, q in zip(sets, sets[1:]))
                                                         / max(1, len(sets) - 1), 3)}
    return {"metric": "decode-time expert cache: microseconds per MoE-layer decode step", "unit": "us",
            "config": {"workload": "mixtral_decode_stream", "d": d, "ffn": F, "E": E, "k": 2,
                       "stream_rho": streams, "keep_MB": keep_mb,
                       "locality_target": "62 % of consecutive tokens share an expert (lecture, layer 15)"},
            "experts": touched, "results": results, "clocks": sampler.summary(),
            "l2_set_aside_MB_tried": [round(v / 2**20, 1) for v in set_asides],
            "note": "32 layers = 32 distinct copies of the expert weights (90 GB), each step runs every layer "
                    "on the step's tokens; between two calls of one layer the other 31 stream 31 layers' weights"}


def run_ep(args) -> dict:
    """Expert parallelism emulated on one GPU: the workload's tokens split over N ranks, each rank's
    expert FFNs timed, for the contiguous, the load-balanced and the replicated expert placement
    (one more expert's weights per rank, given to copies of the hot experts)."""
    import numpy as np
    import torch

    from moe_inputs import CONFIGS, make_config
    from sparse_mixture_experts_53_b300 import ep

    torch.cuda.set_device(0)
    N = args.ep
    cfg = CONFIGS[args.config]
    L = make_config(args.config)
    T = cfg["T"]
    if T % N:
        raise SystemExit("the workload's tokens must split evenly over the ranks")
    xs = [L.x[s * T // N:(s + 1) * T // N].cuda() for s in range(N)]
    wg, w1, w3, w2 = L.w_gate.cuda(), L.w1.cuda(), L.w3.cuda(), L.w2.cuda()
    out = {}
    load = None
    for name in ("contiguous", "balanced", "replicated"):
        if name == "contiguous":
            owner = ep.contiguous_owners(8, N)
        elif name == "balanced":
            owner = ep.balanced_owners(load, N)
        else:  # room for one more expert's weights per rank: copies of the hot experts
            owner = ep.replicated_placement(load, N, 8 // N + 1)
        for _ in range(max(1, args.warmup // 3)):
            ep.emulate(xs, wg, w1, w3, w2, owner)
        runs = [ep.emulate(xs, wg, w1, w3, w2, owner, time_experts=True) for _ in range(3)]
        p = runs[-1][1]
        ms = np.median(np.array([r[2] for r in runs]), axis=0)
        load = p.counts.sum(0)
        out[name] = {"placement": p.placement, "rows_per_rank": p.rows_per_rank.tolist(),
                     "expert_ms_per_rank": [round(float(v), 4) for v in ms],
                     "max_over_mean": round(float(ms.max() / ms.mean()), 3),
                     "tokens_per_s_if_ranks_in_parallel": round(T / (ms.max() * 1e-3), 1)}
    return {"metric": "expert-parallel emulation: per-rank expert FFN time", "ep_ranks": N,
            "config": {"workload": cfg["name"], "T": T, "tokens_per_rank": T // N},
            "expert_load": [int(v) for v in load], "placements": out,
            "note": "ranks run one after another on one GPU; a rank's time is its own experts' FFN on the rows "
                    "it received, the quantity the slowest rank of a real expert-parallel step is bound by"}


def _oracle_cores() -> int:
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        return os.cpu_count() or 1


def _sample_tokens(idx_ref, T: int, n: int, seed: int):
    """n seeded token indices, led by up to 4 tokens of the least-used expert that has any."""
    import numpy as np
    counts = np.bincount(idx_ref.ravel(), minlength=8)
    used = [e for e in range(8) if counts[e] > 0]
    rare = min(used, key=lambda e: counts[e])
    lead = np.nonzero((idx_ref == rare).any(axis=1))[0][:4].tolist()
    rest = np.random.default_rng(seed).permutation(T).tolist()
    out = list(dict.fromkeys(lead + rest))
    return out[:min(n, T)], int(rare)


def cpu_baseline(gpu_out: dict, budget_s: float = 20.0, decode_budget_s: float = 6.0) -> tuple[dict, dict]:
    """The fp64 oracle, as it stands, on a bounded sample of the timed workload's tokens, one oracle call per
    token (its rate is the CPU baseline). Its results are also the parity check of the GPU's output of the
    timed steps: routing on every token, y on the sampled tokens, and the statistics when the step has them."""
    import numpy as np

    import oracle
    from moe_inputs import CONFIGS, make_config, to_f64

    cores = _oracle_cores()
    k = gpu_out["cfg"]
    cfg = CONFIGS[k]
    L = make_config(k)
    w = tuple(t.float().numpy() for t in (L.w1, L.w3, L.w2))

    def check(L, out, budget, n_max, seed):
        x64, wg64 = to_f64(L.x), to_f64(L.w_gate)
        logits = oracle.router_logits(x64, wg64)
        idx_ref, _, _ = oracle.top_k_gates(logits, 2)
        routing_exact = bool(np.array_equal(out["idx"].numpy().astype(np.int64), idx_ref))
        tokens, rare = _sample_tokens(idx_ref, L.T, n_max, seed)
        y_gpu = to_f64(out["y"])
        refs, done, t0 = [], [], time.time()
        for t in tokens:
            if done and (time.time() - t0) >= budget:
                break
            refs.append(oracle.layer_forward_tokens(x64, wg64, *w, [t])[0])
            done.append(t)
        dt = time.time() - t0
        ref = np.stack(refs)
        err = float(np.max(np.abs(y_gpu[done] - ref)) / np.max(np.abs(ref)))
        par = {"routing_exact": routing_exact, "tokens_routed": int(L.T), "y_tokens_checked": len(done),
               "y_max_rel_err": err, "tol": 2e-2, "finite": bool(np.all(np.isfinite(y_gpu))),
               "rarest_expert": rare}
        aux_ok = True
        if out.get("stats") is not None:
            # the statistics' tolerances of the GPU tests: f exact up to one fp32 rounding, P from fp32 scores
            a = oracle.aux_stats(logits, idx_ref, 8)
            f, P, l = (t.numpy().astype(np.float64) for t in out["stats"])
            par["aux"] = {"f_max_abs_err": float(np.max(np.abs(f - a["f"]))),
                          "P_max_abs_err": float(np.max(np.abs(P - a["P"]))),
                          "l_aux": float(l[0]), "l_aux_ref": float(a["l_aux"]),
                          "l_aux_rel_err": abs(float(l[0]) - float(a["l_aux"])) / float(a["l_aux"]),
                          "tol": {"f": 1e-7, "P": 2e-5, "l_aux_rel": 1e-4}}
            aux_ok = (par["aux"]["f_max_abs_err"] <= 1e-7 and par["aux"]["P_max_abs_err"] <= 2e-5
                      and par["aux"]["l_aux_rel_err"] <= 1e-4)
        par["pass"] = bool(routing_exact and par["finite"] and err <= 2e-2 and aux_ok)
        return par, len(done), dt

    par, n, dt = check(L, gpu_out, budget_s, 64, 11)
    base = {"value": round(n / dt, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of the workload's {cfg['T']} tokens, one oracle call per token (fp64 router, both "
                      f"experts incl. weight widening), {dt:.1f} s"}
    if "decode" in gpu_out:
        L1 = make_config(1, weights=(L.w1, L.w3, L.w2))
        dpar, _, _ = check(L1, gpu_out["decode"], decode_budget_s, 16, 12)
        par["decode"] = dpar
        par["pass"] = par["pass"] and dpar["pass"]
    return base, par


def run_reference(args, rank, world) -> dict | None:
    """The fp64 CPU oracle as the reference arm: each step is one token of the workload."""
    if rank != 0:
        return None
    import oracle
    from moe_inputs import CONFIGS, make_config, to_f64

    try:
        from threadpoolctl import threadpool_info
        cores = max([i.get("num_threads", 1) for i in threadpool_info()] + [1])
    except Exception:
        cores = os.cpu_count() or 1
    k = args.config
    cfg = CONFIGS[k]
    L = make_config(k)
    w = tuple(t.float().numpy() for t in (L.w1, L.w3, L.w2))
    x64, wg64 = to_f64(L.x), to_f64(L.w_gate)
    for i in range(args.warmup):
        oracle.layer_forward_tokens(x64, wg64, *w, [i % cfg["T"]])
    t0 = time.time()
    for i in range(args.steps):
        oracle.layer_forward_tokens(x64, wg64, *w, [(args.warmup + i) % cfg["T"]])
    dt = (time.time() - t0) / args.steps
    v = round(1.0 / dt, 4)
    sample = f"one token of the {cfg['T']}-token batch per step (fp64 oracle: router + both experts)"
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded Mixtral-shape tensors, random init)",
            "config": {"workload": cfg["name"], "T": cfg["T"], "d": cfg["d"], "ffn": cfg["ffn"], "E": cfg["E"],
                       "k": 2},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=[1, 2, 3, 4])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--pdl", type=int, default=1, choices=[0, 1],
                    help="programmatic dependent launch between the library's kernels")
    ap.add_argument("--ep", type=int, default=0,
                    help="emulate N expert-parallel ranks on one GPU and time each rank's experts")
    ap.add_argument("--train", action="store_true",
                    help="time a training step (forward that keeps its state + backward) instead of the forward")
    ap.add_argument("--block", action="store_true",
                    help="time the decoder block around the layer (attention + MoE) at the Mixtral shape")
    ap.add_argument("--block-decode", action="store_true",
                    help="time one decode step of the Mixtral block (16 sequences, 4096-token caches)")
    ap.add_argument("--tile-ctas", type=int, default=0, choices=[0, 1, 2],
                    help="token tiles: automatic (0), single CTAs (1), CTA pairs (2)")
    ap.add_argument("--tile-sched", type=int, default=0, choices=range(8),
                    help="CTA-pair GEMMs claiming their units from a counter: bit 0 up, bit 1 down, "
                         "bit 2 the backward's four (0, the default: static units per pair)")
    ap.add_argument("--decode-loop", action="store_true",
                    help="decode-time expert cache experiment: a locality token stream through 1 or 32 layers "
                         "with and without part of each call's expert weights kept in L2")
    ap.add_argument("--no-decode", action="store_true",
                    help="skip the decode batch that the default line carries beside the headline workload")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = _dist_env()
    if args.ep:
        print(json.dumps(run_ep(args)), flush=True)
        return
    if args.decode_loop:
        if args.impl != "ours" or world != 1:
            raise SystemExit("--decode-loop times this library's decode steps on one GPU")
        print(json.dumps(run_decode_loop(args)), flush=True)
        return
    if args.block_decode:
        if args.impl != "ours" or world != 1:
            raise SystemExit("--block-decode times this library's decode step on one GPU")
        print(json.dumps(run_block_decode(args)), flush=True)
        return
    if args.block:
        if args.impl != "ours" or world != 1:
            raise SystemExit("--block times this library's decoder block on one GPU")
        print(json.dumps(run_block(args)), flush=True)
        return
    if args.train:
        if args.impl != "ours" or world != 1:
            raise SystemExit("--train times this library's training step on one GPU")
        print(json.dumps(run_training(args)), flush=True)
        return
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    line = run_ours(args, rank, world, local)
    if line is None:
        return
    gpu_out = line.pop("_gpu_out")
    if not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = cpu_baseline(gpu_out)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
