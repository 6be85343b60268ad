"""Paged-KV attention step for GB300: a thin PyTorch binding of libpagedattn.so.

The binding only marshals arguments: it checks devices, dtypes and contiguity of torch tensors
and passes their device pointers and the current CUDA stream to the C ABI (include/pa.h).  Every
step of the computation runs in the library's CUDA kernels; if the library is missing the calls
raise, there is no CPU fallback.

    import paged_kv_cache_286_gb300 as pa
    ws = pa.new_workspace(pa.attention_workspace_size(...), device="cuda")
    pa.cache_append(k, v, slot_mapping, k_cache, v_cache, ws)
    out = pa.attention(q, k_cache, v_cache, block_tables, context_lens, query_start_loc, ws,
                       scale=..., max_context_len=..., max_query_len=...)
"""

from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _lib
from ._lib import (PA_BF16, PA_FP8_E4M3, PA_FP32, PA_WORKSPACE_HEADER_BYTES,  # noqa: F401
                   PagedAttnError)

__all__ = ["cache_append", "attention", "attention_workspace_size", "new_workspace",
           "check_error", "library", "version", "PagedAttnError", "set_kernel_timing_events",
           "set_prefill_timing_events", "set_kernel_span_buffer"]


def library() -> ctypes.CDLL:
    return _lib.load()


def version() -> str:
    return _lib.load().pa_version().decode()


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtypes, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


_FP8_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def cache_desc(k_cache: torch.Tensor, k_scale: float = 1.0, v_scale: float = 1.0):
    nb, hkv, bs, d = k_cache.shape
    dt = PA_FP8_E4M3 if k_cache.dtype in _FP8_DTYPES else PA_BF16
    return _lib.CacheDesc(nb, bs, hkv, d, dt, float(k_scale), float(v_scale))


def new_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A workspace tensor with its error word cleared."""
    ws = torch.empty(max(int(nbytes), PA_WORKSPACE_HEADER_BYTES), dtype=torch.uint8,
                     device=device)
    ws[:PA_WORKSPACE_HEADER_BYTES].zero_()
    return ws


def cache_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, workspace: torch.Tensor, *,
                 k_scale: float = 1.0, v_scale: float = 1.0, stream=None) -> None:
    """Write k/v [T, Hkv, D] (bf16) into the pools through slot_mapping [T] (int64)."""
    _need(k, "k", (torch.bfloat16,), 3)
    _need(v, "v", (torch.bfloat16,), 3)
    _need(slot_mapping, "slot_mapping", (torch.int64,), 1)
    _need(k_cache, "k_cache", (torch.bfloat16,) + _FP8_DTYPES, 4)
    _need(v_cache, "v_cache", (k_cache.dtype,), 4)
    if k_cache.shape != v_cache.shape:
        raise ValueError("k_cache and v_cache shapes differ")
    if k.shape != v.shape or k.shape[0] != slot_mapping.shape[0] or \
            k.shape[1:] != (k_cache.shape[1], k_cache.shape[3]):
        raise ValueError("k/v/slot_mapping shapes do not match the cache")
    desc = cache_desc(k_cache, k_scale, v_scale)
    L = _lib.load()
    _lib.check(L.pa_cache_append(_ptr(k), _ptr(v), _ptr(slot_mapping), k.shape[0],
                                 _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
                                 _ptr(workspace), _stream(stream)))


def attention_workspace_size(num_seqs: int, num_q_tokens: int, num_q_heads: int,
                             num_kv_heads: int, head_dim: int, max_context_len: int,
                             max_query_len: int, block_size: int = 16) -> int:
    return int(_lib.load().pa_attention_workspace_size(
        num_seqs, num_q_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
        max_context_len, max_query_len))


def attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor,
              query_start_loc: torch.Tensor, workspace: torch.Tensor, *, scale: float,
              max_context_len: int, max_query_len: int, out: Optional[torch.Tensor] = None,
              out_dtype: torch.dtype = torch.float32, k_scale: float = 1.0,
              v_scale: float = 1.0, stream=None) -> torch.Tensor:
    """Ragged paged attention: q [T, Hq, D] bf16 -> out [T, Hq, D] (fp32 or bf16)."""
    _need(q, "q", (torch.bfloat16,), 3)
    _need(k_cache, "k_cache", (torch.bfloat16,) + _FP8_DTYPES, 4)
    _need(v_cache, "v_cache", (k_cache.dtype,), 4)
    _need(block_tables, "block_tables", (torch.int32,), 2)
    _need(context_lens, "context_lens", (torch.int32,), 1)
    _need(query_start_loc, "query_start_loc", (torch.int32,), 1)
    _need(workspace, "workspace", (torch.uint8,), 1)
    T, Hq, D = q.shape
    S = context_lens.shape[0]
    Hkv = k_cache.shape[1]
    if query_start_loc.shape[0] != S + 1 or block_tables.shape[0] != S:
        raise ValueError("query_start_loc must have num_seqs + 1 entries and block_tables "
                         "num_seqs rows")
    if out is None:
        out = torch.empty((T, Hq, D), dtype=out_dtype, device=q.device)
    else:
        _need(out, "out", (torch.float32, torch.bfloat16), 3)
        if tuple(out.shape) != (T, Hq, D):
            raise ValueError("out has the wrong shape")
    odt = PA_FP32 if out.dtype == torch.float32 else PA_BF16
    desc = cache_desc(k_cache, k_scale, v_scale)
    L = _lib.load()
    _lib.check(L.pa_attention(
        _ptr(q), T, _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), _ptr(query_start_loc), S,
        int(max_context_len), int(max_query_len), Hq, Hkv, D, float(scale), _ptr(out), odt,
        _ptr(workspace), workspace.numel(), _stream(stream)))
    return out


def check_error(workspace: torch.Tensor, stream=None, raise_on_error: bool = True) -> int:
    """Synchronise, read and clear the device error word; returns its PA_DEVERR_* bits."""
    word = ctypes.c_uint32(0)
    st = _lib.load().pa_check_error(_ptr(workspace), _stream(stream), ctypes.byref(word))
    if raise_on_error and st != _lib.PA_OK:
        raise _lib.PagedAttnError(st, _lib.load().pa_last_error_string().decode())
    return int(word.value)


def set_kernel_timing_events(before: Optional[torch.cuda.Event],
                             after: Optional[torch.cuda.Event]) -> None:
    """Have later attention calls of this thread record `before`/`after` around their main
    kernel (benchmark hook); pass None to stop."""
    b = ctypes.c_void_p(before.cuda_event) if before is not None else ctypes.c_void_p(0)
    a = ctypes.c_void_p(after.cuda_event) if after is not None else ctypes.c_void_p(0)
    _lib.load().pa_set_kernel_timing_events(b, a)


def set_kernel_span_buffer(buf: Optional[torch.Tensor]) -> None:
    """Have later attention calls of this thread record the global-timer span (ns) of their
    split-KV kernel into buf[0:2] and of their prefill-tile kernel into buf[2:4] (int64 CUDA
    tensor preset to [-1, 0, -1, 0], read as unsigned); None stops (benchmark hook)."""
    if buf is not None:
        _need(buf, "span buffer", (torch.int64,), 1)
        if buf.numel() < 4:
            raise ValueError("the span buffer needs four entries")
    _lib.load().pa_set_kernel_span_buffer(_ptr(buf) if buf is not None else ctypes.c_void_p(0))


def set_prefill_timing_events(before: Optional[torch.cuda.Event],
                              after: Optional[torch.cuda.Event]) -> None:
    """Have later attention calls of this thread record `before`/`after` around their
    tensor-core prefill-tile kernel, when they launch one (benchmark hook); None stops."""
    b = ctypes.c_void_p(before.cuda_event) if before is not None else ctypes.c_void_p(0)
    a = ctypes.c_void_p(after.cuda_event) if after is not None else ctypes.c_void_p(0)
    _lib.load().pa_set_prefill_timing_events(b, a)
