"""Host-side checks of the C ABI: exports and argument validation (no GPU work).

Every check below returns before the library makes any CUDA call, so these run
on a machine without a GPU.
"""
import ctypes
import re
from pathlib import Path

import pytest
import torch

from sparse_mixture_experts_53_b300 import moe

HEADER = Path(__file__).resolve().parent.parent / "include" / "moe.h"


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_function_is_exported():
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(moe.lib, n), n
    assert set(names) == set(moe.EXPORTED)


def test_header_constants_match_the_binding():
    """Every MOE_* enumerator of the header has the same value in moe.py (knobs, statuses, dtypes)."""
    text = re.sub(r"/\*.*?\*/", "", HEADER.read_text(), flags=re.S)
    found = {}
    for body in re.findall(r"enum\s*\w*\s*\{(.*?)\}", text, flags=re.S):
        for name, value in re.findall(r"\b(MOE_[A-Z0-9_]+)\s*=\s*(\d+)", body):
            found[name] = int(value)
    assert len(found) >= 19
    for name, value in found.items():
        assert getattr(moe, name) == value, name


def test_version_and_status_strings():
    assert "sm_103a" in moe.version()
    assert moe.status_string(moe.MOE_OK) == "ok"
    assert moe.status_string(moe.MOE_ERR_TIMEOUT) == "device wait timed out"
    assert moe.status_string(99) == "unknown status"


def _shape(**kw):
    base = dict(T=16, d=4096, ffn=14336, dtype=moe.MOE_BF16, E=8, k=2)
    base.update(kw)
    return moe.make_shape(base["T"], base["d"], base["ffn"], base["dtype"], E=base["E"], k=base["k"])


FAKE = ctypes.c_void_p(1 << 20)        # aligned, never dereferenced
MISALIGNED = ctypes.c_void_p((1 << 20) + 4)


def _forward(shape, x=FAKE, ws_bytes=1 << 40, aux=(None, None, None)):
    return moe.lib.moe_layer_forward(ctypes.byref(shape), x, FAKE, FAKE, FAKE, FAKE, FAKE,
                                     aux[0], aux[1], aux[2], FAKE, ws_bytes, None)


def test_shape_validation_codes():
    lib = moe.lib
    assert lib.moe_route_top2(None, FAKE, FAKE, FAKE, FAKE, None, None) == moe.MOE_ERR_INVALID_ARG
    assert _forward(_shape(E=4)) == moe.MOE_ERR_UNSUPPORTED
    assert _forward(_shape(k=1)) == moe.MOE_ERR_UNSUPPORTED
    assert _forward(_shape(d=100)) == moe.MOE_ERR_UNSUPPORTED          # bf16 needs d % 256 == 0
    assert _forward(_shape(ffn=200)) == moe.MOE_ERR_UNSUPPORTED        # bf16 needs ffn % 128 == 0
    assert _forward(_shape(T=-1)) == moe.MOE_ERR_INVALID_ARG
    assert _forward(_shape(dtype=7)) == moe.MOE_ERR_INVALID_ARG
    assert _forward(_shape(d=0)) == moe.MOE_ERR_INVALID_ARG


def test_pointer_and_workspace_validation():
    s = _shape()
    assert _forward(s, x=None) == moe.MOE_ERR_INVALID_ARG
    assert _forward(s, x=MISALIGNED) == moe.MOE_ERR_INVALID_ARG
    assert _forward(s, ws_bytes=0) == moe.MOE_ERR_WORKSPACE
    assert _forward(s, ws_bytes=moe.moe_workspace_bytes(s) - 1) == moe.MOE_ERR_WORKSPACE
    # statistics pointers come all together or not at all
    assert _forward(s, aux=(FAKE, None, None)) == moe.MOE_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op():
    assert _forward(_shape(T=0), x=None, ws_bytes=0) == moe.MOE_OK


def test_workspace_sizes():
    s = _shape(T=16384)
    n = moe.moe_workspace_bytes(s)
    R = 2 * 16384
    # x_perm (bf16) + hidden (bf16) + y_slot (fp32) dominate
    assert n >= R * 4096 * 2 + R * 14336 * 2 + R * 4096 * 4
    assert n < 1.01 * (R * 4096 * 2 + R * 14336 * 2 + R * 4096 * 4) + (1 << 22)
    assert moe.moe_workspace_bytes(_shape(E=4)) == 0
    assert moe.moe_ffn_workspace_bytes(_shape(T=16)) > 0
    f = moe.make_shape(64, 128, 256, moe.MOE_F32)
    assert moe.moe_workspace_bytes(f) > 0


def test_knobs_and_timeouts():
    lib = moe.lib
    assert lib.moe_set_knob(99, 0) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 3) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_KSLICE, 100) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 3) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 4) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_TILE_CTAS, 5) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_PDL, 2) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, -1) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, 128 * 1024 + 1) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, 64 * 1024) == moe.MOE_OK
    assert lib.moe_set_knob(moe.MOE_KNOB_L2_KEEP_KB, 0) == moe.MOE_OK
    assert lib.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, -1) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, 8) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, 7) == moe.MOE_OK
    assert lib.moe_set_knob(moe.MOE_KNOB_TILE_SCHED, 0) == moe.MOE_OK
    assert lib.moe_set_knob(moe.MOE_KNOB_ROUTER_TC, 2) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_ROUTER_TC, 0) == moe.MOE_OK
    assert lib.moe_set_knob(moe.MOE_KNOB_ROUTER_TC, 1) == moe.MOE_OK
    assert lib.moe_set_knob(moe.MOE_KNOB_FUSE_COMBINE, 2) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_set_knob(moe.MOE_KNOB_FUSE_COMBINE, 0) == moe.MOE_OK
    assert lib.moe_set_knob(moe.MOE_KNOB_FUSE_COMBINE, 1) == moe.MOE_OK
    assert lib.moe_set_wait_timeout_ns(0) == moe.MOE_ERR_INVALID_ARG
    try:
        moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 2)
        # the weight-streaming path covers at most 64 tokens
        assert moe.moe_workspace_bytes(_shape(T=65)) == 0
        assert _forward(_shape(T=65)) == moe.MOE_ERR_UNSUPPORTED
    finally:
        moe.moe_set_knob(moe.MOE_KNOB_FFN_PATH, 0)
    assert moe.moe_timing_read() == {}


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device error path")
def test_device_status_without_a_device_reports_cuda_error():
    code = ctypes.c_int32(0)
    assert moe.lib.moe_get_device_status(ctypes.byref(code), None) == moe.MOE_ERR_CUDA


# ------------------------------------------------------------ decoder block

def _block(**kw):
    base = dict(B=1, S=4096, d=4096, n_heads=32, n_kv_heads=8, ffn=14336)
    base.update(kw)
    extra = {k: base.pop(k) for k in ("head_dim", "eps", "rope_base", "cache_max") if k in base}
    return moe.make_block_shape(base["B"], base["S"], base["d"], base["n_heads"], base["n_kv_heads"], base["ffn"],
                                **extra)


def _block_forward(shape, ws_bytes=1 << 40, x=FAKE, out=ctypes.c_void_p(2 << 20)):
    w = moe.moe_block_weights(*([FAKE] * 8))
    return moe.lib.moe_block_forward(ctypes.byref(shape), x, ctypes.byref(w), None, None, out, FAKE, ws_bytes, None)


def test_block_workspace_covers_its_buffers():
    s = _block()
    T, d = 4096, 4096
    n = moe.moe_block_workspace_bytes(s)
    own = T * d * 2 + T * 6144 * 4 + T * 4096 * 2 + 2 * T * 1024 * 2 + T * 4096 * 2 + 2 * T * d * 2
    layer = moe.moe_workspace_bytes(moe.make_shape(T, d, 14336, moe.MOE_BF16))
    assert own + layer <= n <= own + layer + 16 * 1024


def test_block_shape_validation_codes():
    assert _block_forward(_block(n_kv_heads=3)) == moe.MOE_ERR_INVALID_ARG      # 32 % 3
    assert _block_forward(_block(B=0)) == moe.MOE_ERR_INVALID_ARG
    assert _block_forward(_block(eps=-1.0)) == moe.MOE_ERR_INVALID_ARG
    assert _block_forward(_block(rope_base=0.0)) == moe.MOE_ERR_INVALID_ARG
    assert _block_forward(_block(head_dim=64)) == moe.MOE_ERR_UNSUPPORTED
    assert _block_forward(_block(d=4000)) == moe.MOE_ERR_UNSUPPORTED
    assert _block_forward(_block(n_heads=1, n_kv_heads=1)) == moe.MOE_ERR_UNSUPPORTED  # projection 384 wide
    assert _block_forward(_block(), x=MISALIGNED) == moe.MOE_ERR_INVALID_ARG
    assert _block_forward(_block(), out=FAKE) == moe.MOE_ERR_INVALID_ARG           # out aliases x
    s = _block()
    assert _block_forward(s, ws_bytes=moe.moe_block_workspace_bytes(s) - 1) == moe.MOE_ERR_WORKSPACE


def test_block_step_validation_codes():
    lib = moe.lib
    assert lib.moe_rmsnorm(4, 12, FAKE, None, FAKE, 1e-5, None, FAKE, None) == moe.MOE_ERR_INVALID_ARG  # d % 8
    assert lib.moe_rmsnorm(4, 16, FAKE, FAKE, FAKE, 1e-5, None, FAKE, None) == moe.MOE_ERR_INVALID_ARG  # no h_out
    assert lib.moe_rmsnorm(0, 16, None, None, None, 1e-5, None, None, None) == moe.MOE_OK
    assert lib.moe_linear(4, 96, 256, FAKE, FAKE, FAKE, None, 0, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_linear(4, 64, 200, FAKE, FAKE, FAKE, None, 0, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_linear(0, 64, 256, None, None, None, None, 0, None) == moe.MOE_OK
    # weight streaming for up to 64 rows: K-slice partials of rows x n_out fp32
    n = moe.moe_linear_workspace_bytes(16, 4096, 6144)
    assert n > 0 and n % (16 * 6144 * 4) == 0
    assert moe.moe_linear_workspace_bytes(65, 4096, 6144) == 0
    assert lib.moe_residual_add(12, FAKE, FAKE, FAKE, None) == moe.MOE_ERR_INVALID_ARG
    s = _block(head_dim=64)
    assert lib.moe_attention(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_rope_split(ctypes.byref(_block()), None, None, FAKE, FAKE, FAKE, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    # positions (decode) need one token per sequence; a cache needs room for the prefill
    assert lib.moe_rope_split(ctypes.byref(_block()), FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None) == \
        moe.MOE_ERR_INVALID_ARG
    assert lib.moe_rope_split(ctypes.byref(_block(cache_max=100)), FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, None) \
        == moe.MOE_ERR_INVALID_ARG


def test_block_decode_validation_codes():
    w = moe.moe_block_weights(*([FAKE] * 8))
    dec = _block(S=1, B=16, cache_max=4096)
    n = moe.moe_block_decode_workspace_bytes(dec)
    assert n > 0

    def call(s, cache_len=FAKE, ws_bytes=1 << 40):
        return moe.lib.moe_block_decode(ctypes.byref(s), FAKE, ctypes.byref(w), FAKE, FAKE, cache_len,
                                        ctypes.c_void_p(2 << 20), FAKE, ws_bytes, None)
    assert call(_block(S=2, B=16, cache_max=4096)) == moe.MOE_ERR_INVALID_ARG    # one token per sequence
    assert call(_block(S=1, B=16, cache_max=0)) == moe.MOE_ERR_INVALID_ARG       # no cache
    assert call(dec, cache_len=None) == moe.MOE_ERR_INVALID_ARG
    assert call(dec, ws_bytes=n - 1) == moe.MOE_ERR_WORKSPACE
    # the decode attention takes up to 16 query heads per KV head
    assert moe.moe_block_decode_workspace_bytes(_block(S=1, n_heads=32, n_kv_heads=1, cache_max=64)) == 0
    assert moe.moe_block_decode_workspace_bytes(_block(S=1, n_heads=16, n_kv_heads=1, cache_max=64)) > 0
    assert moe.moe_block_decode_workspace_bytes(_block(S=1, n_heads=24, n_kv_heads=8, cache_max=64)) > 0
    # one partial (128 channels, maximum, sum) per query head and split; splits fill the SMs once
    att = moe.moe_attention_decode_workspace_bytes(dec)
    assert 16 * 32 * (128 + 2) * 4 <= att <= 16 * 32 * 64 * (128 + 2) * 4 + 4096


def test_debug_knob_and_environment():
    assert moe.lib.moe_set_knob(moe.MOE_KNOB_DEBUG, 2) == moe.MOE_ERR_INVALID_ARG
    assert moe.lib.moe_set_knob(moe.MOE_KNOB_DEBUG, 1) == moe.MOE_OK
    assert moe.lib.moe_set_knob(moe.MOE_KNOB_DEBUG, 0) == moe.MOE_OK
    # the library loads with the debug flag and with a wait limit (valid or not) in the environment
    import os
    import subprocess
    import sys
    code = ("import sys; sys.path.insert(0, '.'); from sparse_mixture_experts_53_b300 import moe; "
            "print(moe.version())")
    for env in ({"MOE_DEBUG": "1", "MOE_WAIT_TIMEOUT_NS": "5000000"}, {"MOE_WAIT_TIMEOUT_NS": "not a number"}):
        r = subprocess.run([sys.executable, "-c", code], env=dict(os.environ, **env), capture_output=True, text=True,
                           cwd=str(HEADER.parent.parent), timeout=300)
        assert r.returncode == 0 and "sm_103a" in r.stdout, r.stderr

