"""Thin ctypes binding of libmla (include/mla.h).

Argument marshalling only: every function checks shapes, dtypes and devices
of the PyTorch tensors it is given, passes their device pointers and the
current CUDA stream to the C entry point of the same name, and raises
``MLAError`` on a non-zero status.  All arithmetic runs in the CUDA kernels
of libmla; if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

from . import build as _build

KV_LORA_RANK, QK_ROPE, QK_NOPE, V_HEAD, ROW = 512, 64, 128, 128, 576
Q8_BLOCKS = 18

STATUS = {0: "MLA_OK", -1: "MLA_ERR_INVALID_ARG", -2: "MLA_ERR_UNSUPPORTED", -3: "MLA_ERR_MISALIGNED",
          -4: "MLA_ERR_WORKSPACE", -5: "MLA_ERR_CUDA", -6: "MLA_ERR_TIMEOUT", -7: "MLA_ERR_RANGE"}


class MLAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)} ({status})")


class MLADims(ctypes.Structure):
    _fields_ = [("n_head", ctypes.c_int32), ("kv_lora_rank", ctypes.c_int32), ("qk_rope", ctypes.c_int32),
                ("qk_nope", ctypes.c_int32), ("v_head", ctypes.c_int32), ("scale", ctypes.c_float)]


def make_dims(n_head: int, scale: Optional[float] = None) -> MLADims:
    if scale is None:
        scale = 1.0 / math.sqrt(QK_NOPE + QK_ROPE)
    return MLADims(n_head, KV_LORA_RANK, QK_ROPE, QK_NOPE, V_HEAD, scale)


_P = ctypes.c_void_p
_I32, _I64, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_D = ctypes.POINTER(MLADims)

_SIGS = {
    "mla_absorb_q": ([_D, _P, _P, _P, _I32, _P], ctypes.c_int),
    "mla_prefill_workspace_size": ([_D, _I32], _SZ),
    "mla_attn_prefill": ([_D, _P, _P, _P, _I32, _I32, _I32, _P, _SZ, _P, _P, _P], ctypes.c_int),
    "mla_attn_prefill_q8_0": ([_D, _P, _P, _P, _P, _I32, _I32, _I32, _P, _SZ, _P, _P, _P], ctypes.c_int),
    "mla_prefill_materialized_workspace_size": ([_D, _I32, _I32, _I32], _SZ),
    "mla_attn_prefill_materialized": ([_D, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _SZ, _P, _P, _P],
                                      ctypes.c_int),
    "mla_attn_prefill_materialized_q8_0": ([_D, _P, _P, _P, _P, _P, _P, _I32, _I32, _I32, _I32, _P, _SZ, _P, _P,
                                            _P], ctypes.c_int),
    "mla_decode_workspace_size": ([_D, _I32, _I32], _SZ),
    "mla_attn_decode": ([_D, _P, _P, _P, _I64, _P, _P, _I32, _I32, _P, _SZ, _P, _P], ctypes.c_int),
    "mla_attn_decode_q8_0": ([_D, _P, _P, _P, _P, _I64, _P, _P, _I32, _I32, _P, _SZ, _P, _P], ctypes.c_int),
    "mla_attn_decode_static": ([_D, _P, _P, _P, _I64, _P, _P, _I32, _I32, _P, _P], ctypes.c_int),
    "mla_late_decompress": ([_D, _P, _P, _P, _I32, _P], ctypes.c_int),
    "mla_late_decompress_f16": ([_D, _P, _P, _P, _I32, _P], ctypes.c_int),
    "mla_convert_bf16_to_f16": ([_P, _P, _I64, _P], ctypes.c_int),
    "mla_output_project": ([_D, _P, _P, _P, _I32, _I32, _P], ctypes.c_int),
    "mla_quantize_q8_0": ([_P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "mla_rope_append": ([_P, _P, _P, _P, _I32, ctypes.c_float, ctypes.c_float, _P, _P, _P, _I64, _I64, _P],
                        ctypes.c_int),
    "mla_get_device_error": ([_P], ctypes.c_int),
    "mla_selftest_wait_timeout": ([_I32, _P], ctypes.c_int),
    "mla_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "mla_version": ([], ctypes.c_char_p),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def load_library() -> ctypes.CDLL:
    """Load libmla.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"libmla.so is not built ({_build.LIB}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(_build.LIB)
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def declared_symbols():
    return sorted(_SIGS)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(fn: str, status: int):
    if status != 0:
        raise MLAError(fn, status)


def _need(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return ctypes.c_void_p(t.data_ptr())


def mla_absorb_q(q_nope: torch.Tensor, wk_b: torch.Tensor, q_lat: torch.Tensor, scale=None, stream=None):
    T, H = q_nope.shape[0], q_nope.shape[1]
    d = make_dims(H, scale)
    args = (_need(q_nope, "q_nope", torch.bfloat16, (T, H, QK_NOPE)),
            _need(wk_b, "wk_b", torch.bfloat16, (H, QK_NOPE, KV_LORA_RANK)),
            _need(q_lat, "q_lat", torch.float16, (T, H, KV_LORA_RANK)))
    _check("mla_absorb_q", load_library().mla_absorb_q(ctypes.byref(d), *args, T, _stream(stream)))


def mla_late_decompress(o_lat: torch.Tensor, wv_b: torch.Tensor, o: torch.Tensor, scale=None, stream=None):
    T, H = o_lat.shape[0], o_lat.shape[1]
    d = make_dims(H, scale)
    args = (_need(o_lat, "o_lat", torch.float16, (T, H, KV_LORA_RANK)),
            _need(wv_b, "wv_b", torch.bfloat16, (H, KV_LORA_RANK, V_HEAD)),
            _need(o, "o", torch.float32, (T, H, V_HEAD)))
    _check("mla_late_decompress", load_library().mla_late_decompress(ctypes.byref(d), *args, T, _stream(stream)))


def mla_late_decompress_f16(o_lat: torch.Tensor, wv_b: torch.Tensor, o: torch.Tensor, scale=None, stream=None):
    T, H = o_lat.shape[0], o_lat.shape[1]
    d = make_dims(H, scale)
    args = (_need(o_lat, "o_lat", torch.float16, (T, H, KV_LORA_RANK)),
            _need(wv_b, "wv_b", torch.bfloat16, (H, KV_LORA_RANK, V_HEAD)),
            _need(o, "o", torch.float16, (T, H, V_HEAD)))
    _check("mla_late_decompress_f16",
           load_library().mla_late_decompress_f16(ctypes.byref(d), *args, T, _stream(stream)))


def mla_convert_bf16_to_f16(src: torch.Tensor, dst: torch.Tensor, stream=None):
    """dst = fp16(src), elementwise (weight preparation, e.g. w_o)."""
    if src.shape != dst.shape:
        raise ValueError("src and dst must have the same shape")
    st = load_library().mla_convert_bf16_to_f16(_need(src, "src", torch.bfloat16), _need(dst, "dst", torch.float16),
                                                src.numel(), _stream(stream))
    _check("mla_convert_bf16_to_f16", st)


def mla_output_project(o: torch.Tensor, w_o: torch.Tensor, u: torch.Tensor, scale=None, stream=None):
    """u [T, D] fp32 = o [T, H, 128] fp16 flattened, times w_o [H, 128, D] fp16."""
    T, H = o.shape[0], o.shape[1]
    D = w_o.shape[2]
    d = make_dims(H, scale)
    args = (_need(o, "o", torch.float16, (T, H, V_HEAD)), _need(w_o, "w_o", torch.float16, (H, V_HEAD, D)),
            _need(u, "u", torch.float32, (T, D)))
    _check("mla_output_project", load_library().mla_output_project(ctypes.byref(d), *args, T, D, _stream(stream)))


def mla_prefill_workspace_size(n_head: int, n_kv: int, scale=None) -> int:
    d = make_dims(n_head, scale)
    return int(load_library().mla_prefill_workspace_size(ctypes.byref(d), n_kv))


def _prefill_ws(workspace, H: int, n_kv: int, device):
    """The caller's workspace, or a fresh one from PyTorch's allocator."""
    if workspace is None:
        workspace = torch.empty(mla_prefill_workspace_size(H, n_kv), dtype=torch.uint8, device=device)
    return _need(workspace, "workspace", torch.uint8), workspace.numel()


def mla_attn_prefill(q_lat, q_pe, kv, q_pos0: int, o_lat, lse=None, scale=None, stream=None, workspace=None):
    T, H = q_lat.shape[0], q_lat.shape[1]
    n_kv = kv.shape[0]
    d = make_dims(H, scale)
    lp = _need(lse, "lse", torch.float32, (T, H)) if lse is not None else None
    wp, wn = _prefill_ws(workspace, H, n_kv, kv.device)
    st = load_library().mla_attn_prefill(
        ctypes.byref(d), _need(q_lat, "q_lat", torch.float16, (T, H, KV_LORA_RANK)),
        _need(q_pe, "q_pe", torch.bfloat16, (T, H, QK_ROPE)), _need(kv, "kv", torch.bfloat16, (n_kv, ROW)),
        n_kv, T, q_pos0, wp, wn, _need(o_lat, "o_lat", torch.float16, (T, H, KV_LORA_RANK)), lp, _stream(stream))
    _check("mla_attn_prefill", st)


def mla_attn_prefill_q8_0(q_lat, q_pe, kv_q, kv_d, q_pos0: int, o_lat, lse=None, scale=None, stream=None,
                          workspace=None):
    T, H = q_lat.shape[0], q_lat.shape[1]
    n_kv = kv_q.shape[0]
    d = make_dims(H, scale)
    lp = _need(lse, "lse", torch.float32, (T, H)) if lse is not None else None
    wp, wn = _prefill_ws(workspace, H, n_kv, kv_q.device)
    st = load_library().mla_attn_prefill_q8_0(
        ctypes.byref(d), _need(q_lat, "q_lat", torch.float16, (T, H, KV_LORA_RANK)),
        _need(q_pe, "q_pe", torch.bfloat16, (T, H, QK_ROPE)), _need(kv_q, "kv_q", torch.int8, (n_kv, ROW)),
        _need(kv_d, "kv_d", torch.float16, (Q8_BLOCKS, n_kv)), n_kv, T, q_pos0, wp, wn,
        _need(o_lat, "o_lat", torch.float16, (T, H, KV_LORA_RANK)), lp, _stream(stream))
    _check("mla_attn_prefill_q8_0", st)


def mla_prefill_materialized_workspace_size(n_head: int, T: int, q_pos0: int, head_chunk: int = 0,
                                            scale=None) -> int:
    d = make_dims(n_head, scale)
    return int(load_library().mla_prefill_materialized_workspace_size(ctypes.byref(d), T, q_pos0, head_chunk))


def mla_attn_prefill_materialized(q_nope, q_pe, kv, wk_b, wv_b, q_pos0: int, o, lse=None, head_chunk: int = 0,
                                  workspace=None, scale=None, stream=None):
    """o [T, H, 128] fp32 by decompressing the visible cache rows per head and
    running standard causal attention on them (the pp_opt prefill)."""
    T, H = q_nope.shape[0], q_nope.shape[1]
    n_kv = kv.shape[0]
    d = make_dims(H, scale)
    if workspace is None:
        workspace = torch.empty(mla_prefill_materialized_workspace_size(H, T, q_pos0, head_chunk, scale),
                                dtype=torch.uint8, device=kv.device)
    lp = _need(lse, "lse", torch.float32, (T, H)) if lse is not None else None
    st = load_library().mla_attn_prefill_materialized(
        ctypes.byref(d), _need(q_nope, "q_nope", torch.bfloat16, (T, H, QK_NOPE)),
        _need(q_pe, "q_pe", torch.bfloat16, (T, H, QK_ROPE)), _need(kv, "kv", torch.bfloat16, (n_kv, ROW)),
        _need(wk_b, "wk_b", torch.bfloat16, (H, QK_NOPE, KV_LORA_RANK)),
        _need(wv_b, "wv_b", torch.bfloat16, (H, KV_LORA_RANK, V_HEAD)), n_kv, T, q_pos0, head_chunk,
        _need(workspace, "workspace", torch.uint8), workspace.numel(), _need(o, "o", torch.float32, (T, H, V_HEAD)),
        lp, _stream(stream))
    _check("mla_attn_prefill_materialized", st)


def mla_attn_prefill_materialized_q8_0(q_nope, q_pe, kv_q, kv_d, wk_b, wv_b, q_pos0: int, o, lse=None,
                                       head_chunk: int = 0, workspace=None, scale=None, stream=None):
    """The materialised prefill over a q8_0 cache (kv_q int8 [n, 576], kv_d fp16 [18, n])."""
    T, H = q_nope.shape[0], q_nope.shape[1]
    n_kv = kv_q.shape[0]
    d = make_dims(H, scale)
    if workspace is None:
        workspace = torch.empty(mla_prefill_materialized_workspace_size(H, T, q_pos0, head_chunk, scale),
                                dtype=torch.uint8, device=kv_q.device)
    lp = _need(lse, "lse", torch.float32, (T, H)) if lse is not None else None
    st = load_library().mla_attn_prefill_materialized_q8_0(
        ctypes.byref(d), _need(q_nope, "q_nope", torch.bfloat16, (T, H, QK_NOPE)),
        _need(q_pe, "q_pe", torch.bfloat16, (T, H, QK_ROPE)), _need(kv_q, "kv_q", torch.int8, (n_kv, ROW)),
        _need(kv_d, "kv_d", torch.float16, (Q8_BLOCKS, n_kv)),
        _need(wk_b, "wk_b", torch.bfloat16, (H, QK_NOPE, KV_LORA_RANK)),
        _need(wv_b, "wv_b", torch.bfloat16, (H, KV_LORA_RANK, V_HEAD)), n_kv, T, q_pos0, head_chunk,
        _need(workspace, "workspace", torch.uint8), workspace.numel(), _need(o, "o", torch.float32, (T, H, V_HEAD)),
        lp, _stream(stream))
    _check("mla_attn_prefill_materialized_q8_0", st)


def mla_decode_workspace_size(n_head: int, B: int, max_len: int, scale=None) -> int:
    d = make_dims(n_head, scale)
    return int(load_library().mla_decode_workspace_size(ctypes.byref(d), B, max_len))


def mla_attn_decode(q_lat, q_pe, kv, seq_start, seq_len, max_len: int, workspace, o_lat, scale=None, stream=None):
    B, H = q_lat.shape[0], q_lat.shape[1]
    d = make_dims(H, scale)
    st = load_library().mla_attn_decode(
        ctypes.byref(d), _need(q_lat, "q_lat", torch.float16, (B, H, KV_LORA_RANK)),
        _need(q_pe, "q_pe", torch.bfloat16, (B, H, QK_ROPE)), _need(kv, "kv", torch.bfloat16),
        kv.shape[0], _need(seq_start, "seq_start", torch.int64, (B,)), _need(seq_len, "seq_len", torch.int32, (B,)),
        B, max_len, _need(workspace, "workspace", torch.uint8), workspace.numel(),
        _need(o_lat, "o_lat", torch.float16, (B, H, KV_LORA_RANK)), _stream(stream))
    _check("mla_attn_decode", st)


def mla_attn_decode_static(q_lat, q_pe, kv, seq_start, seq_len, max_len: int, o_lat, scale=None, stream=None):
    """Decode without a workspace argument (the library's fixed device scratch)."""
    B, H = q_lat.shape[0], q_lat.shape[1]
    d = make_dims(H, scale)
    st = load_library().mla_attn_decode_static(
        ctypes.byref(d), _need(q_lat, "q_lat", torch.float16, (B, H, KV_LORA_RANK)),
        _need(q_pe, "q_pe", torch.bfloat16, (B, H, QK_ROPE)), _need(kv, "kv", torch.bfloat16),
        kv.shape[0], _need(seq_start, "seq_start", torch.int64, (B,)), _need(seq_len, "seq_len", torch.int32, (B,)),
        B, max_len, _need(o_lat, "o_lat", torch.float16, (B, H, KV_LORA_RANK)), _stream(stream))
    _check("mla_attn_decode_static", st)


def mla_attn_decode_q8_0(q_lat, q_pe, kv_q, kv_d, seq_start, seq_len, max_len: int, workspace, o_lat,
                         scale=None, stream=None):
    B, H = q_lat.shape[0], q_lat.shape[1]
    n_rows = kv_q.shape[0]
    d = make_dims(H, scale)
    st = load_library().mla_attn_decode_q8_0(
        ctypes.byref(d), _need(q_lat, "q_lat", torch.float16, (B, H, KV_LORA_RANK)),
        _need(q_pe, "q_pe", torch.bfloat16, (B, H, QK_ROPE)), _need(kv_q, "kv_q", torch.int8, (n_rows, ROW)),
        _need(kv_d, "kv_d", torch.float16, (Q8_BLOCKS, n_rows)), n_rows,
        _need(seq_start, "seq_start", torch.int64, (B,)), _need(seq_len, "seq_len", torch.int32, (B,)),
        B, max_len, _need(workspace, "workspace", torch.uint8), workspace.numel(),
        _need(o_lat, "o_lat", torch.float16, (B, H, KV_LORA_RANK)), _stream(stream))
    _check("mla_attn_decode_q8_0", st)


def mla_quantize_q8_0(kv, kv_q, kv_d, stream=None):
    n = kv.shape[0]
    if kv_d.dim() != 2 or kv_d.shape[0] != Q8_BLOCKS:
        raise ValueError(f"kv_d must have shape ({Q8_BLOCKS}, ld_d), got {tuple(kv_d.shape)}")
    st = load_library().mla_quantize_q8_0(
        _need(kv, "kv", torch.bfloat16, (n, ROW)), _need(kv_q, "kv_q", torch.int8, (n, ROW)),
        _need(kv_d, "kv_d", torch.float16), n, kv_d.shape[1], _stream(stream))
    _check("mla_quantize_q8_0", st)


def mla_rope_append(c_kv, k_pe, pos, slot, kv=None, kv_q=None, kv_d=None, freq_base: float = 10000.0,
                    freq_scale: float = 0.025, stream=None):
    """New tokens' rows into the cache(s): row slot[j] <- [c_kv[j] | RoPE(k_pe[j], pos[j])]."""
    n = c_kv.shape[0]
    if kv is None and kv_q is None:
        raise ValueError("mla_rope_append needs a bf16 cache (kv), a q8_0 cache (kv_q, kv_d) or both")
    n_rows = kv.shape[0] if kv is not None else kv_q.shape[0]
    kvp = _need(kv, "kv", torch.bfloat16, (n_rows, ROW)) if kv is not None else None
    if kv_q is not None:
        if kv_d is None or kv_d.dim() != 2 or kv_d.shape[0] != Q8_BLOCKS:
            raise ValueError(f"kv_d must have shape ({Q8_BLOCKS}, ld_d)")
        kqp = _need(kv_q, "kv_q", torch.int8, (n_rows, ROW))
        kdp, ld_d = _need(kv_d, "kv_d", torch.float16), kv_d.shape[1]
    else:
        kqp, kdp, ld_d = None, None, 0
    st = load_library().mla_rope_append(
        _need(c_kv, "c_kv", torch.bfloat16, (n, KV_LORA_RANK)), _need(k_pe, "k_pe", torch.bfloat16, (n, QK_ROPE)),
        _need(pos, "pos", torch.int32, (n,)), _need(slot, "slot", torch.int64, (n,)), n, float(freq_base),
        float(freq_scale), kvp, kqp, kdp, ld_d, n_rows, _stream(stream))
    _check("mla_rope_append", st)


def mla_get_device_error(stream=None) -> int:
    return int(load_library().mla_get_device_error(_stream(stream)))


def mla_selftest_wait_timeout(limit_us: int, stream=None):
    _check("mla_selftest_wait_timeout", load_library().mla_selftest_wait_timeout(limit_us, _stream(stream)))


def mla_status_string(status: int) -> str:
    return load_library().mla_status_string(status).decode()


def mla_version() -> str:
    return load_library().mla_version().decode()
