"""ctypes binding of libpagedattn.so, with the C entry points' names.

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI. Torch tensors supply device pointers and the
current CUDA stream; torch is used for nothing else. There is no CPU or
PyTorch fallback: if the compiled library is missing, importing this module
raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

import numpy as np
import torch

from . import build as _build

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE_BOUNDS = 5
PA_ERR_DEVICE_TIMEOUT = 6
PA_ERR_NO_PAGES = 7

PA_DEVERR_PAGE_ID = 0x1
PA_DEVERR_SLOT = 0x2
PA_DEVERR_CONTEXT_LEN = 0x4
PA_DEVERR_TIMEOUT = 0x8

LIB_PATH = _build.LIB


class pa_shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("q_len", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_pages", ctypes.c_int32)]


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
    lib.pa_append_kv.argtypes = [vp, vp, vp, vp, vp, i32, pa_shape, vp]
    lib.pa_append_kv.restype = ctypes.c_int
    lib.pa_decode_workspace_bytes.argtypes = [pa_shape]
    lib.pa_decode_workspace_bytes.restype = sz
    attn = [vp, vp, vp, vp, vp, i32, f32, ctypes.c_int, vp, pa_shape]
    lib.pa_decode.argtypes = attn + [i32, vp, sz, vp]
    lib.pa_decode.restype = ctypes.c_int
    lib.pa_prefill.argtypes = attn + [vp]
    lib.pa_prefill.restype = ctypes.c_int
    lib.pa_append_kv_fp8.argtypes = [vp, vp, vp, vp, vp, i32, f32, f32, pa_shape, vp]
    lib.pa_append_kv_fp8.restype = ctypes.c_int
    lib.pa_decode_fp8.argtypes = [vp, vp, vp, vp, vp, i32, f32, f32, f32, ctypes.c_int, vp,
                                  pa_shape, i32, vp, sz, vp]
    lib.pa_decode_fp8.restype = ctypes.c_int
    lib.pa_prefill_workspace_bytes.argtypes = [pa_shape, i32]
    lib.pa_prefill_workspace_bytes.restype = sz
    lib.pa_prefill_fp8_workspace_bytes.argtypes = [pa_shape, i32]
    lib.pa_prefill_fp8_workspace_bytes.restype = sz
    lib.pa_prefill_fp8.argtypes = [vp, vp, vp, vp, vp, i32, f32, f32, f32, ctypes.c_int, vp,
                                   pa_shape, i32, vp, sz, vp]
    lib.pa_prefill_fp8.restype = ctypes.c_int
    lib.pa_attention_fp8_workspace_bytes.argtypes = [pa_shape, i32]
    lib.pa_attention_fp8_workspace_bytes.restype = sz
    lib.pa_attention_fp8.argtypes = lib.pa_prefill_fp8.argtypes
    lib.pa_attention_fp8.restype = ctypes.c_int
    lib.pa_prefill_split.argtypes = attn + [vp, sz, vp]
    lib.pa_prefill_split.restype = ctypes.c_int
    i64 = ctypes.c_int64
    lib.pa_kv_cache_create.argtypes = [i32, i32, ctypes.POINTER(vp)]
    lib.pa_kv_cache_create.restype = ctypes.c_int
    lib.pa_kv_cache_destroy.argtypes = [vp]
    lib.pa_kv_cache_destroy.restype = None
    lib.pa_kv_cache_add.argtypes = [vp, i64]
    lib.pa_kv_cache_add.restype = ctypes.c_int
    lib.pa_kv_cache_release.argtypes = [vp, i64]
    lib.pa_kv_cache_release.restype = ctypes.c_int
    lib.pa_kv_cache_free_pages.argtypes = [vp]
    lib.pa_kv_cache_free_pages.restype = i32
    lib.pa_kv_cache_context_len.argtypes = [vp, i64]
    lib.pa_kv_cache_context_len.restype = i32
    lib.pa_kv_cache_plan.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp, vp]
    lib.pa_kv_cache_plan.restype = ctypes.c_int
    lib.pa_kv_cache_step_table_bytes.argtypes = [i32, i32, i32]
    lib.pa_kv_cache_step_table_bytes.restype = sz
    lib.pa_kv_cache_step.argtypes = [vp, i32, vp, vp, i32, i32, vp, vp, sz, vp, vp, vp, vp, vp,
                                     i32, i32, i32, ctypes.c_float, vp, vp, sz, vp]
    lib.pa_kv_cache_step.restype = ctypes.c_int
    lib.pa_kv_cache_snapshot_take.argtypes = [vp, ctypes.POINTER(vp)]
    lib.pa_kv_cache_snapshot_take.restype = ctypes.c_int
    lib.pa_kv_cache_restore.argtypes = [vp, vp]
    lib.pa_kv_cache_restore.restype = ctypes.c_int
    lib.pa_kv_cache_snapshot_destroy.argtypes = [vp]
    lib.pa_kv_cache_snapshot_destroy.restype = None
    lib.pa_gather_kv.argtypes = [vp, vp, vp, vp, i32, pa_shape, i32, vp, vp, vp]
    lib.pa_gather_kv.restype = ctypes.c_int
    lib.pa_decode_dense.argtypes = [vp, vp, vp, vp, i32, ctypes.c_float, ctypes.c_int, vp,
                                    pa_shape, i32, vp, sz, vp]
    lib.pa_decode_dense.restype = ctypes.c_int
    lib.pa_attention.argtypes = attn + [i32, vp, sz, vp]
    lib.pa_attention.restype = ctypes.c_int
    lib.pa_attention_route.argtypes = [pa_shape, i32]
    lib.pa_attention_route.restype = i32
    lib.pa_get_device_error.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.pa_get_device_error.restype = ctypes.c_int
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_version.argtypes = []
    lib.pa_version.restype = ctypes.c_char_p
    lib.pa_debug_arm_wait_timeout.argtypes = []
    lib.pa_debug_arm_wait_timeout.restype = None
    lib.pa_debug_prefill_variant.argtypes = [ctypes.c_int]
    lib.pa_debug_prefill_variant.restype = ctypes.c_int
    return lib


_lib = _load()


def status_string(status: int) -> str:
    return _lib.pa_status_string(int(status)).decode()


def version() -> str:
    return _lib.pa_version().decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PagedAttentionError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev_ptr(t: torch.Tensor, dtype: torch.dtype, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def make_shape(query_shape, pages_shape, max_pages: int) -> pa_shape:
    B, H_q, L, D = (int(x) for x in query_shape)
    P, H_kv, _, D2 = (int(x) for x in pages_shape)
    if D2 != D:
        raise ValueError("query and pages disagree on head_dim")
    return pa_shape(B, H_q, H_kv, D, L, P, int(max_pages))


# ---------------------------------------------------------------------------
# Workspace cache: one buffer per device, grown on demand (its contents never
# matter to the library).

_ws_lock = threading.Lock()
_ws_cache = {}


def _cached_workspace(need: int, device: torch.device) -> torch.Tensor:
    with _ws_lock:
        buf = _ws_cache.get(device.index)
        if buf is None or buf.numel() < need:
            buf = torch.zeros(max(need, 256), dtype=torch.uint8, device=device)
            _ws_cache[device.index] = buf
    return buf


def prefill_workspace(shape: pa_shape, page_size: int,
                      device: torch.device) -> Tuple[Optional[torch.Tensor], int]:
    """(buffer, bytes) for pa_prefill_split, or (None, 0) when the shape's
    prefill kernel needs none."""
    need = pa_prefill_workspace_bytes(shape, page_size, device)
    if need == 0:
        return None, 0
    return _cached_workspace(need, device), need


def pa_prefill_workspace_bytes(shape: pa_shape, page_size: int,
                               device: Optional[torch.device] = None) -> int:
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(_lib.pa_prefill_workspace_bytes(shape, int(page_size)))


def decode_workspace(shape: pa_shape, device: torch.device) -> Tuple[torch.Tensor, int]:
    need = pa_decode_workspace_bytes(shape, device)
    with _ws_lock:
        buf = _ws_cache.get(device.index)
        if buf is None or buf.numel() < need:
            buf = torch.zeros(max(need, 256), dtype=torch.uint8, device=device)
            _ws_cache[device.index] = buf
    return buf, need


def pa_decode_workspace_bytes(shape: pa_shape, device: Optional[torch.device] = None) -> int:
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(_lib.pa_decode_workspace_bytes(shape))


# ---------------------------------------------------------------------------
# Entry points


def pa_append_kv(key: torch.Tensor, value: torch.Tensor, key_pages: torch.Tensor,
                 value_pages: torch.Tensor, slot_mapping: torch.Tensor, page_size: int,
                 stream=None) -> None:
    """key/value [B, H_kv, L_new, D] bf16 -> pages [P, H_kv, page_size, D] at
    slot_mapping [B, L_new] int32 (in place)."""
    B, H_kv, L_new, D = key.shape
    if tuple(value.shape) != tuple(key.shape):
        raise ValueError("key and value shapes differ")
    if tuple(slot_mapping.shape) != (B, L_new):
        raise ValueError("slot_mapping must be [B, L_new]")
    if key_pages.shape[1:] != (H_kv, page_size, D) or value_pages.shape != key_pages.shape:
        raise ValueError("page pool shape does not match key / page_size")
    shape = pa_shape(B, 0, H_kv, D, L_new, key_pages.shape[0], 0)
    st = _lib.pa_append_kv(_dev_ptr(key, torch.bfloat16, "key"),
                           _dev_ptr(value, torch.bfloat16, "value"),
                           _dev_ptr(key_pages, torch.bfloat16, "key_pages"),
                           _dev_ptr(value_pages, torch.bfloat16, "value_pages"),
                           _dev_ptr(slot_mapping, torch.int32, "slot_mapping"),
                           int(page_size), shape, _stream(stream))
    _check(st, "pa_append_kv")


def pa_append_kv_fp8(key: torch.Tensor, value: torch.Tensor, key_pages: torch.Tensor,
                     value_pages: torch.Tensor, slot_mapping: torch.Tensor, page_size: int,
                     k_scale: float, v_scale: float, stream=None) -> None:
    """key/value [B, H_kv, L_new, D] bf16 -> uint8 e4m3 pages [P, H_kv,
    page_size, D] at slot_mapping [B, L_new], code = e4m3(x / scale)."""
    B, H_kv, L_new, D = key.shape
    if tuple(value.shape) != tuple(key.shape):
        raise ValueError("key and value shapes differ")
    if tuple(slot_mapping.shape) != (B, L_new):
        raise ValueError("slot_mapping must be [B, L_new]")
    if key_pages.shape[1:] != (H_kv, page_size, D) or value_pages.shape != key_pages.shape:
        raise ValueError("page pool shape does not match key / page_size")
    shape = pa_shape(B, 0, H_kv, D, L_new, key_pages.shape[0], 0)
    st = _lib.pa_append_kv_fp8(_dev_ptr(key, torch.bfloat16, "key"),
                               _dev_ptr(value, torch.bfloat16, "value"),
                               _dev_ptr(key_pages, torch.uint8, "key_pages"),
                               _dev_ptr(value_pages, torch.uint8, "value_pages"),
                               _dev_ptr(slot_mapping, torch.int32, "slot_mapping"),
                               int(page_size), float(k_scale), float(v_scale), shape,
                               _stream(stream))
    _check(st, "pa_append_kv_fp8")


def pa_decode_fp8(query, key_pages, value_pages, block_table, context_lens, page_size: int,
                  k_scale: float, v_scale: float, scale: Optional[float] = None,
                  causal: bool = True, out=None, max_context_len: int = 0,
                  workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Split-KV paged attention over uint8 e4m3 pools (K = code * k_scale,
    V = code * v_scale); query and out [B, H_q, L, D] bf16."""
    B, H_q, L, D = query.shape
    if key_pages.shape[2] != page_size or value_pages.shape != key_pages.shape:
        raise ValueError("page pool shape does not match page_size")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and context_lens [B]")
    if out is None:
        out = torch.empty_like(query)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    shape = make_shape(query.shape, key_pages.shape, block_table.shape[1])
    if workspace is None:
        workspace, _ = decode_workspace(shape, query.device)
    st = _lib.pa_decode_fp8(_dev_ptr(query, torch.bfloat16, "query"),
                            _dev_ptr(key_pages, torch.uint8, "key_pages"),
                            _dev_ptr(value_pages, torch.uint8, "value_pages"),
                            _dev_ptr(block_table, torch.int32, "block_table"),
                            _dev_ptr(context_lens, torch.int32, "context_lens"),
                            int(page_size), float(scale), float(k_scale), float(v_scale),
                            int(bool(causal)), _dev_ptr(out, torch.bfloat16, "out"), shape,
                            int(max_context_len), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_decode_fp8")
    return out


def pa_prefill_fp8_workspace_bytes(shape: pa_shape, max_context_len: int,
                                   device: Optional[torch.device] = None) -> int:
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        return int(_lib.pa_prefill_fp8_workspace_bytes(shape, int(max_context_len)))


def pa_prefill_fp8(query, key_pages, value_pages, block_table, context_lens, page_size: int,
                   k_scale: float, v_scale: float, scale: Optional[float] = None,
                   causal: bool = True, out=None, max_context_len: Optional[int] = None,
                   workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Tensor-core prefill over uint8 e4m3 pools (K = code * k_scale, V =
    code * v_scale); query and out [B, H_q, L, 128] bf16. max_context_len
    bounds context_lens and sizes the bf16 copy in the workspace; None reads
    context_lens.max() (a device-to-host copy)."""
    B, H_q, L, D = query.shape
    if key_pages.shape[2] != page_size or value_pages.shape != key_pages.shape:
        raise ValueError("page pool shape does not match page_size")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and context_lens [B]")
    if out is None:
        out = torch.empty_like(query)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item())
    shape = make_shape(query.shape, key_pages.shape, block_table.shape[1])
    if workspace is None:
        need = pa_prefill_fp8_workspace_bytes(shape, max_context_len, query.device)
        if need == 0:
            raise PagedAttentionError(PA_ERR_UNSUPPORTED, "pa_prefill_fp8")
        workspace = _cached_workspace(need, query.device)
    st = _lib.pa_prefill_fp8(_dev_ptr(query, torch.bfloat16, "query"),
                             _dev_ptr(key_pages, torch.uint8, "key_pages"),
                             _dev_ptr(value_pages, torch.uint8, "value_pages"),
                             _dev_ptr(block_table, torch.int32, "block_table"),
                             _dev_ptr(context_lens, torch.int32, "context_lens"),
                             int(page_size), float(scale), float(k_scale), float(v_scale),
                             int(bool(causal)), _dev_ptr(out, torch.bfloat16, "out"), shape,
                             int(max_context_len), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_prefill_fp8")
    return out


def pa_attention_fp8(query, key_pages, value_pages, block_table, context_lens, page_size: int,
                     k_scale: float, v_scale: float, scale: Optional[float] = None,
                     causal: bool = True, out=None, max_context_len: Optional[int] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The dispatch for e4m3 pools: pa_decode_fp8 for up to 8 query rows,
    pa_prefill_fp8 beyond (pa_attention_route's rule)."""
    B, H_q, L, D = query.shape
    if key_pages.shape[2] != page_size or value_pages.shape != key_pages.shape:
        raise ValueError("page pool shape does not match page_size")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and context_lens [B]")
    if out is None:
        out = torch.empty_like(query)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if max_context_len is None:
        max_context_len = int(context_lens.max().item())
    shape = make_shape(query.shape, key_pages.shape, block_table.shape[1])
    if workspace is None:
        with torch.cuda.device(query.device):
            need = int(_lib.pa_attention_fp8_workspace_bytes(shape, int(max_context_len)))
        if need == 0:
            raise PagedAttentionError(PA_ERR_UNSUPPORTED, "pa_attention_fp8")
        workspace = _cached_workspace(need, query.device)
    st = _lib.pa_attention_fp8(_dev_ptr(query, torch.bfloat16, "query"),
                               _dev_ptr(key_pages, torch.uint8, "key_pages"),
                               _dev_ptr(value_pages, torch.uint8, "value_pages"),
                               _dev_ptr(block_table, torch.int32, "block_table"),
                               _dev_ptr(context_lens, torch.int32, "context_lens"),
                               int(page_size), float(scale), float(k_scale), float(v_scale),
                               int(bool(causal)), _dev_ptr(out, torch.bfloat16, "out"), shape,
                               int(max_context_len), workspace.data_ptr(),
                               workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_attention_fp8")
    return out


def _attn_common(query, key_pages, value_pages, block_table, context_lens, page_size,
                 scale, out):
    B, H_q, L, D = query.shape
    if key_pages.shape[2] != page_size or value_pages.shape != key_pages.shape:
        raise ValueError("page pool shape does not match page_size")
    if block_table.dim() != 2 or block_table.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_table must be [B, max_pages] and context_lens [B]")
    if out is None:
        out = torch.empty_like(query)
    elif tuple(out.shape) != tuple(query.shape):
        raise ValueError("out must have the query's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    shape = make_shape(query.shape, key_pages.shape, block_table.shape[1])
    ptrs = (_dev_ptr(query, torch.bfloat16, "query"),
            _dev_ptr(key_pages, torch.bfloat16, "key_pages"),
            _dev_ptr(value_pages, torch.bfloat16, "value_pages"),
            _dev_ptr(block_table, torch.int32, "block_table"),
            _dev_ptr(context_lens, torch.int32, "context_lens"))
    return shape, ptrs, float(scale), out


def pa_decode(query, key_pages, value_pages, block_table, context_lens, page_size: int,
              scale: Optional[float] = None, causal: bool = True, out=None,
              max_context_len: int = 0, workspace: Optional[torch.Tensor] = None,
              stream=None) -> torch.Tensor:
    """Split-KV paged attention; returns out [B, H_q, L, D] bf16."""
    shape, ptrs, scale, out = _attn_common(query, key_pages, value_pages, block_table,
                                           context_lens, page_size, scale, out)
    if workspace is None:
        workspace, _ = decode_workspace(shape, query.device)
    st = _lib.pa_decode(*ptrs, int(page_size), scale, int(bool(causal)),
                        _dev_ptr(out, torch.bfloat16, "out"), shape, int(max_context_len),
                        workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        _stream(stream))
    _check(st, "pa_decode")
    return out


def pa_prefill(query, key_pages, value_pages, block_table, context_lens, page_size: int,
               scale: Optional[float] = None, causal: bool = True, out=None,
               stream=None) -> torch.Tensor:
    """Page-walking prefill attention; returns out [B, H_q, L, D] bf16."""
    shape, ptrs, scale, out = _attn_common(query, key_pages, value_pages, block_table,
                                           context_lens, page_size, scale, out)
    st = _lib.pa_prefill(*ptrs, int(page_size), scale, int(bool(causal)),
                         _dev_ptr(out, torch.bfloat16, "out"), shape, _stream(stream))
    _check(st, "pa_prefill")
    return out


def pa_prefill_split(query, key_pages, value_pages, block_table, context_lens, page_size: int,
                     scale: Optional[float] = None, causal: bool = True, out=None,
                     workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """pa_prefill on the kernel that spreads the K/V tiles evenly over the
    SMs (needs a workspace; the library's shared one is used when none is
    given)."""
    shape, ptrs, scale, out = _attn_common(query, key_pages, value_pages, block_table,
                                           context_lens, page_size, scale, out)
    if workspace is None:
        workspace, _ = prefill_workspace(shape, page_size, query.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = _lib.pa_prefill_split(*ptrs, int(page_size), scale, int(bool(causal)),
                               _dev_ptr(out, torch.bfloat16, "out"), shape, ws_ptr, ws_bytes,
                               _stream(stream))
    _check(st, "pa_prefill_split")
    return out


def pa_attention_route(query_shape, pages_shape, max_pages: int, max_context_len: int = 0) -> int:
    return int(_lib.pa_attention_route(make_shape(query_shape, pages_shape, max_pages),
                                       int(max_context_len)))


def pa_attention(query, key_pages, value_pages, block_table, context_lens, page_size: int,
                 scale: Optional[float] = None, causal: bool = True, out=None,
                 max_context_len: int = 0, workspace: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """Dispatching entry point (decode for short queries, prefill otherwise)."""
    shape, ptrs, scale, out = _attn_common(query, key_pages, value_pages, block_table,
                                           context_lens, page_size, scale, out)
    route = int(_lib.pa_attention_route(shape, int(max_context_len)))
    ws_ptr, ws_bytes = None, 0
    if route == 0 and workspace is None:
        workspace, _ = decode_workspace(shape, query.device)
    elif route == 1 and workspace is None:
        workspace, _ = prefill_workspace(shape, page_size, query.device)
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    st = _lib.pa_attention(*ptrs, int(page_size), scale, int(bool(causal)),
                           _dev_ptr(out, torch.bfloat16, "out"), shape, int(max_context_len),
                           ws_ptr, ws_bytes, _stream(stream))
    _check(st, "pa_attention")
    return out


def pa_debug_arm_wait_timeout() -> None:
    """Test support: the next attention call on this thread runs one bounded
    wait on a barrier nothing arrives at (records PA_DEVERR_TIMEOUT)."""
    _lib.pa_debug_arm_wait_timeout()


def pa_get_device_error(stream=None) -> Tuple[int, int]:
    """Synchronises the stream; returns (status, PA_DEVERR_* flags) and clears them."""
    flags = ctypes.c_uint32(0)
    st = _lib.pa_get_device_error(_stream(stream), ctypes.byref(flags))
    return int(st), int(flags.value)


# ---------------------------------------------------------------------------
# Decode without a caller-provided workspace (for callers that cannot
# allocate device memory; the scratch is a fixed array inside the library).

_noalloc_ready = False


def pa_decode_noalloc(query, key_pages, value_pages, block_table, context_lens,
                      page_size: int, scale: Optional[float] = None, causal: bool = True,
                      out=None, max_context_len: int = 0, stream=None) -> torch.Tensor:
    """pa_decode with the library's built-in 32 MiB scratch instead of a
    workspace; `out` must be given by callers that allocate nothing."""
    global _noalloc_ready
    if not _noalloc_ready:
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        _lib.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, ctypes.c_float,
                                           ctypes.c_int, vp, pa_shape, i32, vp]
        _lib.pa_decode_noalloc.restype = ctypes.c_int
        _noalloc_ready = True
    shape, ptrs, scale, out = _attn_common(query, key_pages, value_pages, block_table,
                                           context_lens, page_size, scale, out)
    st = _lib.pa_decode_noalloc(*ptrs, int(page_size), scale, int(bool(causal)),
                                _dev_ptr(out, torch.bfloat16, "out"), shape,
                                int(max_context_len), _stream(stream))
    _check(st, "pa_decode_noalloc")
    return out


def pa_debug_prefill_variant(variant: int) -> int:
    """Select the tensor-core prefill kernel for this thread's calls: 0 auto,
    1 one query head per block, 2 two heads of a KV group per block (even
    group size). Returns the previous setting."""
    return int(_lib.pa_debug_prefill_variant(int(variant)))


def pa_gather_kv(key_pages, value_pages, block_table, context_lens, page_size: int,
                 dense_len: int, key_dense=None, value_dense=None, stream=None):
    """Dense copies [B, H_kv, dense_len, D] of every request's visible K and V
    rows (the dense baseline's gather); returns (key_dense, value_dense)."""
    P, H_kv, ps, D = key_pages.shape
    if ps != page_size or value_pages.shape != key_pages.shape:
        raise ValueError("page pool shape does not match page_size")
    B = block_table.shape[0]
    if key_dense is None:
        key_dense = torch.empty((B, H_kv, dense_len, D), dtype=torch.bfloat16,
                                device=key_pages.device)
    if value_dense is None:
        value_dense = torch.empty_like(key_dense)
    for t in (key_dense, value_dense):
        if tuple(t.shape) != (B, H_kv, dense_len, D):
            raise ValueError("dense buffers must be [B, H_kv, dense_len, D]")
    shape = pa_shape(B, H_kv, H_kv, D, 1, P, block_table.shape[1])
    st = _lib.pa_gather_kv(_dev_ptr(key_pages, torch.bfloat16, "key_pages"),
                           _dev_ptr(value_pages, torch.bfloat16, "value_pages"),
                           _dev_ptr(block_table, torch.int32, "block_table"),
                           _dev_ptr(context_lens, torch.int32, "context_lens"), int(page_size),
                           shape, int(dense_len), _dev_ptr(key_dense, torch.bfloat16, "key_dense"),
                           _dev_ptr(value_dense, torch.bfloat16, "value_dense"), _stream(stream))
    _check(st, "pa_gather_kv")
    return key_dense, value_dense


def pa_decode_dense(query, key_dense, value_dense, context_lens, scale: Optional[float] = None,
                    causal: bool = True, out=None, max_context_len: int = 0,
                    workspace: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Split-KV decode over dense K/V [B, H_kv, dense_len, D] (the dense
    baseline's attention); returns out [B, H_q, L, D] bf16."""
    B, H_q, L, D = query.shape
    Bk, H_kv, dense_len, Dk = key_dense.shape
    if (Bk, Dk) != (B, D) or value_dense.shape != key_dense.shape:
        raise ValueError("dense K/V must be [B, H_kv, dense_len, D]")
    if out is None:
        out = torch.empty_like(query)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    shape = pa_shape(B, H_q, H_kv, D, L, B, 1)
    if workspace is None:
        workspace, _ = decode_workspace(shape, query.device)
    st = _lib.pa_decode_dense(_dev_ptr(query, torch.bfloat16, "query"),
                              _dev_ptr(key_dense, torch.bfloat16, "key_dense"),
                              _dev_ptr(value_dense, torch.bfloat16, "value_dense"),
                              _dev_ptr(context_lens, torch.int32, "context_lens"), int(dense_len),
                              float(scale), int(bool(causal)), _dev_ptr(out, torch.bfloat16, "out"),
                              shape, int(max_context_len), workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "pa_decode_dense")
    return out


class KVCache:
    """Host-side page allocator and per-step metadata of one layer pool (the
    C++ pa_kv_cache): freed pages first, tail-fill placement, all-or-nothing
    steps, release exactly once."""

    def __init__(self, num_pages: int, page_size: int):
        h = ctypes.c_void_p()
        _check(_lib.pa_kv_cache_create(int(num_pages), int(page_size), ctypes.byref(h)),
               "pa_kv_cache_create")
        self._h = h
        self.num_pages = int(num_pages)
        self.page_size = int(page_size)

    def close(self) -> None:
        if self._h:
            _lib.pa_kv_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def add(self, seq_id: int) -> None:
        _check(_lib.pa_kv_cache_add(self._h, int(seq_id)), "pa_kv_cache_add")

    def release(self, seq_id: int) -> None:
        _check(_lib.pa_kv_cache_release(self._h, int(seq_id)), "pa_kv_cache_release")

    @property
    def free_pages(self) -> int:
        return int(_lib.pa_kv_cache_free_pages(self._h))

    def context_len(self, seq_id: int) -> int:
        return int(_lib.pa_kv_cache_context_len(self._h, int(seq_id)))

    def snapshot(self) -> "KVCacheSnapshot":
        """Copy of the bookkeeping, for restore() after a failed step."""
        h = ctypes.c_void_p()
        _check(_lib.pa_kv_cache_snapshot_take(self._h, ctypes.byref(h)),
               "pa_kv_cache_snapshot_take")
        return KVCacheSnapshot(h)

    def restore(self, snapshot: "KVCacheSnapshot") -> None:
        _check(_lib.pa_kv_cache_restore(self._h, snapshot._h), "pa_kv_cache_restore")

    def plan(self, seq_ids, new_tokens, max_pages: int, l_new: int):
        """One step: returns (block_table [n, max_pages], context_lens [n],
        slot_mapping [n, l_new]) as int32 numpy arrays; raises
        PagedAttentionError (PA_ERR_NO_PAGES) with nothing changed when the
        step does not fit."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        toks = np.ascontiguousarray(new_tokens, dtype=np.int32)
        n = int(ids.shape[0])
        bt = np.empty((n, int(max_pages)), dtype=np.int32)
        cl = np.empty((n,), dtype=np.int32)
        sm = np.empty((n, max(int(l_new), 1)), dtype=np.int32)
        st = _lib.pa_kv_cache_plan(self._h, n, ids.ctypes.data, toks.ctypes.data, int(max_pages),
                                   int(l_new), bt.ctypes.data, cl.ctypes.data, sm.ctypes.data)
        _check(st, "pa_kv_cache_plan")
        return bt, cl, sm[:, :int(l_new)]

    @staticmethod
    def step_table_bytes(n: int, max_pages: int, l_new: int) -> int:
        """Bytes of the packed tables of one pa_kv_cache_step."""
        return int(_lib.pa_kv_cache_step_table_bytes(int(n), int(max_pages), int(l_new)))

    def step(self, seq_ids, new_tokens, l_new: int, max_pages: int, host_tables, device_tables,
             key_new, value_new, query, key_pages, value_pages, out=None,
             scale: Optional[float] = None, workspace: Optional[torch.Tensor] = None,
             stream=None) -> torch.Tensor:
        """One whole step in one native call (pa_kv_cache_step): plan into the
        pinned `host_tables`, one copy to `device_tables`, append, attention.
        Returns out [n, H_q, l_new, D]. `host_tables` must not be rewritten
        (by a later step) before this step's copy has run."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        toks = np.ascontiguousarray(new_tokens, dtype=np.int32)
        n = int(ids.shape[0])
        if n != query.shape[0] or n != key_new.shape[0] or int(l_new) != query.shape[2]:
            raise ValueError("query / key_new must be [n, heads, l_new, D] for the n requests")
        if not host_tables.is_pinned() or not device_tables.is_cuda:
            raise ValueError("host_tables must be pinned host memory, device_tables on the GPU")
        nbytes = min(host_tables.numel() * host_tables.element_size(),
                     device_tables.numel() * device_tables.element_size())
        _, H_q, _, D = (int(x) for x in query.shape)
        H_kv = int(key_new.shape[1])
        if out is None:
            out = torch.empty_like(query)
        if scale is None:
            scale = 1.0 / math.sqrt(D)
        if workspace is None:
            shape = pa_shape(n, H_q, H_kv, D, int(l_new), int(key_pages.shape[0]), int(max_pages))
            workspace, _ = decode_workspace(shape, query.device)
            pws, _ = prefill_workspace(shape, self.page_size, query.device)
            if pws is not None and pws.numel() > workspace.numel():
                workspace = pws
        st = _lib.pa_kv_cache_step(
            self._h, n, ids.ctypes.data, toks.ctypes.data, int(l_new), int(max_pages),
            host_tables.data_ptr(), device_tables.data_ptr(), nbytes,
            _dev_ptr(key_new, torch.bfloat16, "key_new"), _dev_ptr(value_new, torch.bfloat16, "value_new"),
            _dev_ptr(query, torch.bfloat16, "query"), _dev_ptr(key_pages, torch.bfloat16, "key_pages"),
            _dev_ptr(value_pages, torch.bfloat16, "value_pages"), H_q, H_kv, D, float(scale),
            _dev_ptr(out, torch.bfloat16, "out"), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), _stream(stream))
        _check(st, "pa_kv_cache_step")
        return out


class KVCacheSnapshot:
    """A pa_kv_cache_snapshot handle (freed with the object)."""

    def __init__(self, handle):
        self._h = handle

    def close(self) -> None:
        if self._h:
            _lib.pa_kv_cache_snapshot_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
