"""Thin ctypes binding of libmoe.so (include/moe.h).

Argument marshalling only: each function takes torch tensors that already live
on the GPU, passes their device pointers and the current CUDA stream to the C
ABI, and raises ``MoEError`` on a non-OK status. Every step of the layer runs in
the library's CUDA kernels; there is no fallback of any kind. Importing this
module fails loudly when the shared library is missing.
"""
from __future__ import annotations

import ctypes
import json
from pathlib import Path

import torch

_LIB_PATH = Path(__file__).resolve().parent / "libmoe.so"

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6

MOE_F32 = 0
MOE_BF16 = 1

MOE_KNOB_FFN_PATH = 1
MOE_KNOB_KSLICE = 2
MOE_KNOB_GRID = 3
MOE_KNOB_PDL = 4
MOE_KNOB_TILE_CTAS = 5
MOE_KNOB_DEBUG = 6
MOE_KNOB_L2_KEEP_KB = 7
MOE_KNOB_TILE_SCHED = 8
MOE_KNOB_ROUTER_TC = 9
MOE_KNOB_FUSE_COMBINE = 10

EXPORTED = (
    "moe_version", "moe_status_string", "moe_workspace_bytes", "moe_ffn_workspace_bytes",
    "moe_permute_workspace_bytes",
    "moe_route_top2", "moe_permute", "moe_expert_ffn", "moe_combine", "moe_aux_stats",
    "moe_layer_forward", "moe_layer_forward_noalloc", "moe_get_device_status", "moe_set_wait_timeout_ns", "moe_set_knob",
    "moe_timing_enable", "moe_timing_read", "moe_train_state_bytes", "moe_backward_workspace_bytes",
    "moe_layer_forward_train", "moe_layer_backward", "moe_gather_rows", "moe_selftest_wait_timeout",
    "moe_check_device_status", "moe_block_workspace_bytes", "moe_block_forward", "moe_rmsnorm", "moe_linear",
    "moe_rope_split", "moe_attention", "moe_residual_add", "moe_block_decode_workspace_bytes", "moe_block_decode",
    "moe_linear_workspace_bytes", "moe_attention_decode_workspace_bytes", "moe_attention_decode",
    "moe_read_probe",
)


class moe_shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class moe_block_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("S", ctypes.c_int64), ("d", ctypes.c_int32), ("n_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("eps", ctypes.c_float),
                ("rope_base", ctypes.c_float), ("cache_max", ctypes.c_int64)]


class moe_block_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("attn_norm", "wqkv", "wo", "ffn_norm", "w_gate", "w1", "w3", "w2")]


class MoEError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


def _load() -> ctypes.CDLL:
    if not _LIB_PATH.exists():
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "or `python sparse_mixture_experts_53_b300/build.py`")
    lib = ctypes.CDLL(str(_LIB_PATH))
    P = ctypes.c_void_p
    S = ctypes.POINTER(moe_shape)
    BS = ctypes.POINTER(moe_block_shape)
    I = ctypes.c_int
    sig = {
        "moe_version": ([], ctypes.c_char_p),
        "moe_status_string": ([I], ctypes.c_char_p),
        "moe_workspace_bytes": ([S], ctypes.c_size_t),
        "moe_ffn_workspace_bytes": ([S], ctypes.c_size_t),
        "moe_route_top2": ([S, P, P, P, P, P, P], I),
        "moe_permute": ([S, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], I),
        "moe_permute_workspace_bytes": ([S], ctypes.c_size_t),
        "moe_expert_ffn": ([S, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], I),
        "moe_combine": ([S, P, P, P, P], I),
        "moe_aux_stats": ([S, P, P, P, P, P, P], I),
        "moe_layer_forward": ([S, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], I),
        "moe_layer_forward_noalloc": ([S, P, P, P, P, P, P, P], I),
        "moe_get_device_status": ([ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)], I),
        "moe_set_wait_timeout_ns": ([ctypes.c_uint64], I),
        "moe_set_knob": ([ctypes.c_int32, ctypes.c_int64], I),
        "moe_timing_enable": ([ctypes.c_int32], I),
        "moe_timing_read": ([ctypes.c_char_p, ctypes.c_size_t], I),
        "moe_gather_rows": ([P, ctypes.c_int64, P, ctypes.c_int64, ctypes.c_int64, P, P], I),
        "moe_selftest_wait_timeout": ([ctypes.c_uint64, P, P], I),
        "moe_read_probe": ([P, ctypes.c_size_t, P, P], I),
        "moe_check_device_status": ([P], I),
        "moe_train_state_bytes": ([S], ctypes.c_size_t),
        "moe_backward_workspace_bytes": ([S], ctypes.c_size_t),
        "moe_layer_forward_train": ([S, P, P, P, P, P, P, P, P, P, P, ctypes.c_size_t, P], I),
        "moe_layer_backward": ([S, P, P, P, P, P, P, ctypes.c_float, P, ctypes.c_size_t, P, P, P, P, P, P,
                                ctypes.c_size_t, P], I),
        "moe_block_workspace_bytes": ([BS], ctypes.c_size_t),
        "moe_block_forward": ([BS, P, ctypes.POINTER(moe_block_weights), P, P, P, P, ctypes.c_size_t, P], I),
        "moe_block_decode_workspace_bytes": ([BS], ctypes.c_size_t),
        "moe_block_decode": ([BS, P, ctypes.POINTER(moe_block_weights), P, P, P, P, P, ctypes.c_size_t, P], I),
        "moe_rmsnorm": ([ctypes.c_int64, ctypes.c_int32, P, P, P, ctypes.c_float, P, P, P], I),
        "moe_linear_workspace_bytes": ([ctypes.c_int64, ctypes.c_int32, ctypes.c_int32], ctypes.c_size_t),
        "moe_linear": ([ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, P, P, P, P, ctypes.c_size_t, P], I),
        "moe_rope_split": ([BS, P, P, P, P, P, P, P, P], I),
        "moe_attention_decode_workspace_bytes": ([BS], ctypes.c_size_t),
        "moe_attention_decode": ([BS, P, P, P, P, P, P, ctypes.c_size_t, P], I),
        "moe_attention": ([BS, P, P, P, P, P], I),
        "moe_residual_add": ([ctypes.c_int64, P, P, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


lib = _load()


def status_string(code: int) -> str:
    return lib.moe_status_string(int(code)).decode()


def _check(fn: str, code: int) -> None:
    if code != MOE_OK:
        raise MoEError(fn, code)


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.numel() and not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr()) if t.numel() else ctypes.c_void_p(0)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return MOE_BF16
    if t.dtype == torch.float32:
        return MOE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def make_shape(T: int, d: int, ffn: int, dtype: int, E: int = 8, k: int = 2) -> moe_shape:
    return moe_shape(int(T), int(d), int(ffn), int(E), int(k), int(dtype))


def shape_of(x: torch.Tensor, w1: torch.Tensor) -> moe_shape:
    E, ffn, d = w1.shape
    return make_shape(x.shape[0], d, ffn, dtype_code(x), E=E)


def version() -> str:
    return lib.moe_version().decode()


def moe_workspace_bytes(shape: moe_shape) -> int:
    return int(lib.moe_workspace_bytes(ctypes.byref(shape)))


def moe_ffn_workspace_bytes(shape: moe_shape) -> int:
    return int(lib.moe_ffn_workspace_bytes(ctypes.byref(shape)))


def moe_route_top2(shape, x, w_gate, topk_idx, topk_w, logits=None, stream=None):
    _check("moe_route_top2", lib.moe_route_top2(ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(topk_idx),
                                                _ptr(topk_w), _ptr(logits), _stream(stream)))


def moe_permute_workspace_bytes(shape: moe_shape) -> int:
    return int(lib.moe_permute_workspace_bytes(ctypes.byref(shape)))


def moe_permute(shape, topk_idx, topk_w, x, counts, offsets, perm_token, slot_row, perm_w, x_perm, ws=None,
                stream=None):
    """ws: optional byte tensor of moe_permute_workspace_bytes(shape) (many-CTA grouping)."""
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check("moe_permute", lib.moe_permute(ctypes.byref(shape), _ptr(topk_idx), _ptr(topk_w), _ptr(x),
                                          _ptr(counts), _ptr(offsets), _ptr(perm_token), _ptr(slot_row),
                                          _ptr(perm_w), _ptr(x_perm), _ptr(ws), nbytes, _stream(stream)))


def moe_expert_ffn(shape, x_perm, offsets, perm_w, w1, w3, w2, y_slot, ws, stream=None):
    _check("moe_expert_ffn", lib.moe_expert_ffn(ctypes.byref(shape), _ptr(x_perm), _ptr(offsets), _ptr(perm_w),
                                                _ptr(w1), _ptr(w3), _ptr(w2), _ptr(y_slot), _ptr(ws),
                                                ws.numel() * ws.element_size(), _stream(stream)))


def moe_combine(shape, y_slot, slot_row, y, stream=None):
    _check("moe_combine", lib.moe_combine(ctypes.byref(shape), _ptr(y_slot), _ptr(slot_row), _ptr(y),
                                          _stream(stream)))


def moe_aux_stats(shape, logits, counts, f, P, l_aux, stream=None):
    _check("moe_aux_stats", lib.moe_aux_stats(ctypes.byref(shape), _ptr(logits), _ptr(counts), _ptr(f), _ptr(P),
                                              _ptr(l_aux), _stream(stream)))


def moe_layer_forward(shape, x, w_gate, w1, w3, w2, y, ws, aux=None, stream=None):
    """aux: None or a tuple of (f [E], P [E], l_aux [1]) float32 device tensors."""
    f, P, l = aux if aux is not None else (None, None, None)
    _check("moe_layer_forward", lib.moe_layer_forward(
        ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(y), _ptr(f), _ptr(P),
        _ptr(l), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_layer_forward_noalloc(shape, x, w_gate, w1, w3, w2, y, stream=None):
    """moe_layer_forward on the library's fixed static scratch (no workspace, no allocation)."""
    _check("moe_layer_forward_noalloc", lib.moe_layer_forward_noalloc(
        ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(y), _stream(stream)))


def moe_gather_rows(src, index, dst, stream=None):
    """dst[r] = src[index[r]] (rows of src's trailing dimensions); index is int32 on the device."""
    rows = index.numel()
    row_bytes = dst[0].numel() * dst.element_size() if rows else 16
    _check("moe_gather_rows", lib.moe_gather_rows(_ptr(src), src.shape[0], _ptr(index), rows, row_bytes, _ptr(dst),
                                                  _stream(stream)))


def moe_train_state_bytes(shape: moe_shape) -> int:
    return int(lib.moe_train_state_bytes(ctypes.byref(shape)))


def moe_backward_workspace_bytes(shape: moe_shape) -> int:
    return int(lib.moe_backward_workspace_bytes(ctypes.byref(shape)))


def moe_layer_forward_train(shape, x, w_gate, w1, w3, w2, y, state, aux=None, stream=None):
    """moe_layer_forward that keeps its intermediates in `state` (moe_train_state_bytes bytes)."""
    f, P, l = aux if aux is not None else (None, None, None)
    _check("moe_layer_forward_train", lib.moe_layer_forward_train(
        ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(y), _ptr(f), _ptr(P),
        _ptr(l), _ptr(state), state.numel() * state.element_size(), _stream(stream)))


def moe_layer_backward(shape, x, w_gate, w1, w3, w2, dy, aux_coef, state, dx, dw_gate, dw1, dw3, dw2, ws,
                       stream=None):
    _check("moe_layer_backward", lib.moe_layer_backward(
        ctypes.byref(shape), _ptr(x), _ptr(w_gate), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(dy), float(aux_coef),
        _ptr(state), state.numel() * state.element_size(), _ptr(dx), _ptr(dw_gate), _ptr(dw1), _ptr(dw3),
        _ptr(dw2), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_selftest_wait_timeout(timeout_ns: int, gave_up, stream=None):
    _check("moe_selftest_wait_timeout", lib.moe_selftest_wait_timeout(int(timeout_ns), _ptr(gave_up),
                                                                      _stream(stream)))


def moe_read_probe(buf, sink, stream=None):
    """Reads every byte of the device tensor `buf` once (HBM read-rate probe); sink: a device int32 tensor."""
    _check("moe_read_probe", lib.moe_read_probe(_ptr(buf), buf.numel() * buf.element_size(), _ptr(sink),
                                                _stream(stream)))


def moe_check_device_status(stream=None) -> int:
    """Waits for the stream and returns (and clears) the latched device error code."""
    return int(lib.moe_check_device_status(_stream(stream)))


def moe_get_device_status() -> tuple[int, int]:
    code = ctypes.c_int32(0)
    detail = ctypes.c_int32(0)
    _check("moe_get_device_status", lib.moe_get_device_status(ctypes.byref(code), ctypes.byref(detail)))
    return int(code.value), int(detail.value)


def moe_set_wait_timeout_ns(ns: int) -> None:
    _check("moe_set_wait_timeout_ns", lib.moe_set_wait_timeout_ns(int(ns)))


def moe_set_knob(knob: int, value: int) -> None:
    _check("moe_set_knob", lib.moe_set_knob(int(knob), int(value)))


def moe_timing_enable(enable: bool) -> None:
    _check("moe_timing_enable", lib.moe_timing_enable(1 if enable else 0))


def moe_timing_read() -> dict:
    buf = ctypes.create_string_buffer(1 << 16)
    _check("moe_timing_read", lib.moe_timing_read(buf, len(buf)))
    return json.loads(buf.value.decode() or "{}")


# ------------------------------------------------------------------ helpers

def workspace(shape: moe_shape, device="cuda", ffn_only: bool = False) -> torch.Tensor:
    """A byte tensor of the size the ABI asks for (allocated by torch, not the library)."""
    n = moe_ffn_workspace_bytes(shape) if ffn_only else moe_workspace_bytes(shape)
    if n == 0 and shape.T > 0:
        raise MoEError("workspace sizing", MOE_ERR_UNSUPPORTED)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


def layer_forward(x, w_gate, w1, w3, w2, aux: bool = False, ws=None, out=None, stream=None):
    """Allocates y (and the statistics) with torch and calls moe_layer_forward."""
    shape = shape_of(x, w1)
    if ws is None:
        ws = workspace(shape, x.device)
    y = out if out is not None else torch.empty_like(x)
    stats = None
    if aux:
        E = w1.shape[0]
        stats = (torch.empty(E, dtype=torch.float32, device=x.device),
                 torch.empty(E, dtype=torch.float32, device=x.device),
                 torch.empty(1, dtype=torch.float32, device=x.device))
    moe_layer_forward(shape, x, w_gate, w1, w3, w2, y, ws, stats, stream)
    return (y, stats) if aux else y


def _bytes(n: int, device) -> torch.Tensor:
    return torch.empty(max(int(n), 16), dtype=torch.uint8, device=device)


def layer_forward_train(x, w_gate, w1, w3, w2, aux: bool = False, stream=None):
    """Training forward: returns (y, state[, stats]); the state feeds layer_backward."""
    shape = shape_of(x, w1)
    n = moe_train_state_bytes(shape)
    if n == 0 and shape.T > 0:
        raise MoEError("moe_train_state_bytes", MOE_ERR_UNSUPPORTED)
    state = _bytes(n, x.device)
    y = torch.empty_like(x)
    stats = None
    if aux:
        E = w1.shape[0]
        stats = tuple(torch.empty(m, dtype=torch.float32, device=x.device) for m in (E, E, 1))
    moe_layer_forward_train(shape, x, w_gate, w1, w3, w2, y, state, stats, stream)
    return (y, state, stats) if aux else (y, state)


def layer_backward(x, w_gate, w1, w3, w2, dy, state, aux_coef: float = 0.0, ws=None, stream=None):
    """Gradients (dx, dw_gate, dw1, dw3, dw2) for the upstream gradient dy; weight gradients in float32."""
    shape = shape_of(x, w1)
    if ws is None:
        n = moe_backward_workspace_bytes(shape)
        if n == 0:
            raise MoEError("moe_backward_workspace_bytes", MOE_ERR_UNSUPPORTED)
        ws = _bytes(n, x.device)
    f32 = dict(dtype=torch.float32, device=x.device)
    dx = torch.empty_like(x)
    dw_gate = torch.empty(w_gate.shape, **f32)
    dw1 = torch.empty(w1.shape, **f32)
    dw3 = torch.empty(w3.shape, **f32)
    dw2 = torch.empty(w2.shape, **f32)
    moe_layer_backward(shape, x, w_gate, w1, w3, w2, dy, aux_coef, state, dx, dw_gate, dw1, dw3, dw2, ws, stream)
    return dx, dw_gate, dw1, dw3, dw2


# ------------------------------------------------------------ decoder block

def make_block_shape(B: int, S: int, d: int, n_heads: int, n_kv_heads: int, ffn: int, head_dim: int = 128,
                     E: int = 8, k: int = 2, eps: float = 1e-5, rope_base: float = 10000.0,
                     cache_max: int = 0) -> moe_block_shape:
    return moe_block_shape(int(B), int(S), int(d), int(n_heads), int(n_kv_heads), int(head_dim), int(ffn), int(E),
                           int(k), float(eps), float(rope_base), int(cache_max))


def moe_block_workspace_bytes(shape: moe_block_shape) -> int:
    return int(lib.moe_block_workspace_bytes(ctypes.byref(shape)))


def block_weights(p: dict) -> moe_block_weights:
    """p: device tensors attn_norm, wqkv, wo, ffn_norm, w_gate, w1, w3, w2 (bf16)."""
    return moe_block_weights(*[_ptr(p[n]) for n, _ in moe_block_weights._fields_])


def moe_block_forward(shape, x, weights: moe_block_weights, out, ws, k_cache=None, v_cache=None, stream=None):
    _check("moe_block_forward", lib.moe_block_forward(ctypes.byref(shape), _ptr(x), ctypes.byref(weights),
                                                      _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(ws),
                                                      ws.numel() * ws.element_size(), _stream(stream)))


def moe_block_decode_workspace_bytes(shape: moe_block_shape) -> int:
    return int(lib.moe_block_decode_workspace_bytes(ctypes.byref(shape)))


def moe_block_decode(shape, x, weights: moe_block_weights, k_cache, v_cache, cache_len, out, ws, stream=None):
    _check("moe_block_decode", lib.moe_block_decode(ctypes.byref(shape), _ptr(x), ctypes.byref(weights),
                                                    _ptr(k_cache), _ptr(v_cache), _ptr(cache_len), _ptr(out),
                                                    _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_attention_decode_workspace_bytes(shape: moe_block_shape) -> int:
    return int(lib.moe_attention_decode_workspace_bytes(ctypes.byref(shape)))


def moe_attention_decode(shape, q, k_cache, v_cache, cache_len, o, ws, stream=None):
    _check("moe_attention_decode", lib.moe_attention_decode(ctypes.byref(shape), _ptr(q), _ptr(k_cache),
                                                            _ptr(v_cache), _ptr(cache_len), _ptr(o), _ptr(ws),
                                                            ws.numel() * ws.element_size(), _stream(stream)))


def moe_rmsnorm(x, g, eps, y, add=None, h_out=None, stream=None):
    rows, d = x.shape
    _check("moe_rmsnorm", lib.moe_rmsnorm(rows, d, _ptr(x), _ptr(add), _ptr(g), float(eps), _ptr(h_out), _ptr(y),
                                          _stream(stream)))


def moe_linear_workspace_bytes(rows: int, n_in: int, n_out: int) -> int:
    return int(lib.moe_linear_workspace_bytes(int(rows), int(n_in), int(n_out)))


def moe_linear(x, w, y, ws=None, stream=None):
    """y [rows][n_out] fp32 = x [rows][n_in] . w^T (bf16 operands); ws: weight streaming for <= 64 rows."""
    rows, n_in = x.shape
    nbytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check("moe_linear", lib.moe_linear(rows, n_in, w.shape[0], _ptr(x), _ptr(w), _ptr(y), _ptr(ws), nbytes,
                                        _stream(stream)))


def moe_rope_split(shape, qkv, q, k, v, pos=None, k_cache=None, v_cache=None, stream=None):
    _check("moe_rope_split", lib.moe_rope_split(ctypes.byref(shape), _ptr(qkv), _ptr(pos), _ptr(q), _ptr(k), _ptr(v),
                                                _ptr(k_cache), _ptr(v_cache), _stream(stream)))


def moe_attention(shape, q, k, v, o, stream=None):
    _check("moe_attention", lib.moe_attention(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
                                              _stream(stream)))


def moe_residual_add(a, b, out, stream=None):
    _check("moe_residual_add", lib.moe_residual_add(a.numel(), _ptr(a), _ptr(b), _ptr(out), _stream(stream)))


def block_forward(x, p: dict, shape: moe_block_shape, ws=None, k_cache=None, v_cache=None, stream=None):
    """Allocates out (and the workspace) with torch and calls moe_block_forward."""
    if ws is None:
        n = moe_block_workspace_bytes(shape)
        if n == 0:
            raise MoEError("moe_block_workspace_bytes", MOE_ERR_UNSUPPORTED)
        ws = _bytes(n, x.device)
    out = torch.empty_like(x)
    moe_block_forward(shape, x, block_weights(p), out, ws, k_cache, v_cache, stream)
    return out


def kv_cache(shape: moe_block_shape, device="cuda"):
    """Empty key and value caches [B][n_kv_heads][cache_max][head_dim] bf16 for the shape."""
    dims = (shape.B, shape.n_kv_heads, shape.cache_max, shape.head_dim)
    return (torch.zeros(dims, dtype=torch.bfloat16, device=device),
            torch.zeros(dims, dtype=torch.bfloat16, device=device))


def block_decode(x, p: dict, shape: moe_block_shape, k_cache, v_cache, cache_len, ws=None, stream=None):
    """One decode step (x [B][d]: each sequence's next token); appends to the caches, advances cache_len."""
    if ws is None:
        n = moe_block_decode_workspace_bytes(shape)
        if n == 0:
            raise MoEError("moe_block_decode_workspace_bytes", MOE_ERR_UNSUPPORTED)
        ws = _bytes(n, x.device)
    out = torch.empty_like(x)
    moe_block_decode(shape, x, block_weights(p), k_cache, v_cache, cache_len, out, ws, stream)
    return out

