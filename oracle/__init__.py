"""fp64 CPU oracle for paged attention.

TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package. The product path (the
CUDA library and its binding) never imports, links or calls it, and the two
share no code: the arithmetic lives in ``pa_oracle.c`` (plain C, fp64), this
module only compiles it with gcc and marshals numpy arrays.

Definitions followed (page titles and sections, see the C file's header):
  * translation: Week 3 Day 4: Direct Paged Attention, "Why block_table
    Matters";
  * append: Reading vLLM's PagedAttention Kernel, 3.2 "Writing into the cache";
  * attention: Reading vLLM's PagedAttention Kernel, section 4 (dense
    reference), over the gathered valid page prefixes of Tutorial 13,
    section 5 "Reading Pages for Attention";
  * FP8 pages: Reading vLLM's PagedAttention Kernel, section 3.2 (the write
    path's cache dtype and per-tensor k_scale / v_scale), with e4m3 codes
    from the format's own definition.

Every function here is pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

BF16 = 0
F64 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc (OpenMP on). Returns the library path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        p = ctypes.c_void_p
        i32 = ctypes.c_int32
        lib.pa_oracle_translate.argtypes = [p, i32, i32, ctypes.c_int64, p, p]
        lib.pa_oracle_translate.restype = ctypes.c_int
        lib.pa_oracle_append_kv.argtypes = [p, p, p, p, p] + [i32] * 6
        lib.pa_oracle_append_kv.restype = ctypes.c_int64
        lib.pa_oracle_gather.argtypes = [p, p, p] + [i32] * 7 + [p]
        lib.pa_oracle_gather.restype = ctypes.c_int
        lib.pa_oracle_attention_rows.argtypes = (
            [p] * 5 + [i32] * 8 + [ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                   p, ctypes.c_int64, p, ctypes.c_int])
        lib.pa_oracle_attention_rows.restype = ctypes.c_int
        lib.pa_oracle_e4m3_encode.argtypes = [p, p, ctypes.c_int64]
        lib.pa_oracle_e4m3_encode.restype = None
        lib.pa_oracle_e4m3_decode.argtypes = [p, p, ctypes.c_int64]
        lib.pa_oracle_e4m3_decode.restype = None
        lib.pa_oracle_append_kv_fp8.argtypes = ([p, p, p, p, p] + [i32] * 6 +
                                                [ctypes.c_float, ctypes.c_float])
        lib.pa_oracle_append_kv_fp8.restype = ctypes.c_int64
        _lib = lib
        return lib


class OracleError(RuntimeError):
    pass


_STATUS = {1: "page id outside the pool", 2: "context length out of range",
           3: "inconsistent shape arguments", 4: "out of memory"}


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _elem_kind(*arrays: np.ndarray) -> int:
    kinds = {a.dtype for a in arrays}
    if kinds == {np.dtype(np.uint16)}:
        return BF16
    if kinds == {np.dtype(np.float64)}:
        return F64
    raise TypeError("query and pages must all be uint16 (bf16 bits) or all float64")


def translate(block_table_row, page_size: int, num_pages: int, pos: int):
    """Logical key position -> (physical page id, slot in page)."""
    lib = _load()
    row = np.ascontiguousarray(block_table_row, dtype=np.int32)
    page = ctypes.c_int32()
    slot = ctypes.c_int32()
    status = lib.pa_oracle_translate(_ptr(row), page_size, num_pages, pos,
                                     ctypes.byref(page), ctypes.byref(slot))
    if status:
        raise OracleError(_STATUS.get(status, str(status)))
    return page.value, slot.value


def append_kv(key, value, key_pages, value_pages, slot_mapping, page_size: int) -> int:
    """Scatter key/value [B, H_kv, L_new, D] (uint16 bf16 bits) into the pages
    [P, H_kv, page_size, D] in place, by slot_mapping [B, L_new].
    Returns the number of slots that pointed beyond the pool (skipped)."""
    lib = _load()
    for a in (key, value, key_pages, value_pages):
        if a.dtype != np.uint16 or not a.flags.c_contiguous:
            raise TypeError("append_kv works on contiguous uint16 (bf16 bit) arrays")
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    B, H_kv, L_new, D = key.shape
    P = key_pages.shape[0]
    assert value.shape == key.shape and value_pages.shape == key_pages.shape
    assert key_pages.shape[1:] == (H_kv, page_size, D)
    assert slots.shape == (B, L_new)
    return int(lib.pa_oracle_append_kv(_ptr(key), _ptr(value), _ptr(key_pages),
                                       _ptr(value_pages), _ptr(slots), B, L_new,
                                       H_kv, D, page_size, P))


def gather(pages, block_table, context_lens, page_size: int, dense_len: int,
           fill: int = 0) -> np.ndarray:
    """Dense copy of every request's visible K (or V) rows: pages
    [P, H_kv, page_size, D] uint16 (bf16 bits) -> [B, H_kv, dense_len, D];
    rows past a request's context hold `fill`."""
    lib = _load()
    if pages.dtype != np.uint16 or not pages.flags.c_contiguous:
        raise TypeError("gather works on contiguous uint16 (bf16 bit) pages")
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    P, H_kv, ps, D = pages.shape
    assert ps == page_size
    B, max_pages = bt.shape
    out = np.full((B, H_kv, dense_len, D), fill, dtype=np.uint16)
    status = lib.pa_oracle_gather(_ptr(pages), _ptr(bt), _ptr(cl), B, H_kv, D, page_size, P,
                                  max_pages, dense_len, _ptr(out))
    if status:
        raise OracleError(_STATUS.get(status, str(status)))
    return out


def attention(query, key_pages, value_pages, block_table, context_lens,
              page_size: int, scale: float | None = None, causal: bool = True,
              rows=None, n_threads: int = 1) -> np.ndarray:
    """Paged attention in fp64.

    query [B, H_q, L, D]; pages [P, H_kv, page_size, D]; all uint16 (bf16
    bits) or all float64. block_table [B, max_pages] and context_lens [B]
    int32. ``scale=None`` means 1/sqrt(D). ``rows`` (optional) is an
    [n, 3] array of (b, h_q, i); the result is then [n, D], else
    [B, H_q, L, D]."""
    lib = _load()
    kind = _elem_kind(query, key_pages, value_pages)
    q = np.ascontiguousarray(query)
    kp = np.ascontiguousarray(key_pages)
    vp = np.ascontiguousarray(value_pages)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, H_q, L, D = q.shape
    P, H_kv, ps, D2 = kp.shape
    if ps != page_size or D2 != D or vp.shape != kp.shape:
        raise ValueError("page pool shape does not match query / page_size")
    if bt.ndim != 2 or bt.shape[0] != B or cl.shape != (B,):
        raise ValueError("block_table must be [B, max_pages], context_lens [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if rows is None:
        bb, hh, ii = np.meshgrid(np.arange(B), np.arange(H_q), np.arange(L), indexing="ij")
        row_arr = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1).astype(np.int32)
    else:
        row_arr = np.ascontiguousarray(rows, dtype=np.int32).reshape(-1, 3)
    out = np.zeros((row_arr.shape[0], D), dtype=np.float64)
    status = lib.pa_oracle_attention_rows(
        _ptr(q), _ptr(kp), _ptr(vp), _ptr(bt), _ptr(cl), B, H_q, H_kv, L, D,
        page_size, P, bt.shape[1], kind, float(scale), int(bool(causal)),
        _ptr(row_arr), row_arr.shape[0], _ptr(out), int(n_threads))
    if status:
        raise OracleError(_STATUS.get(status, str(status)))
    if rows is None:
        return out.reshape(B, H_q, L, D)
    return out


# ---------------------------------------------------------------------------
# FP8 (e4m3) pages with per-tensor scales (Reading vLLM's PagedAttention
# Kernel, section 3.2: the write path takes the cache dtype, k_scale and
# v_scale). See the C file for the encoding and the reading of the pages.


def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> e4m3 codes (nearest, ties to even, saturated to +-448)."""
    lib = _load()
    xs = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(xs.shape, dtype=np.uint8)
    lib.pa_oracle_e4m3_encode(_ptr(xs), _ptr(out), xs.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 codes -> their exact values (fp64; NaN for S.1111.111)."""
    lib = _load()
    cs = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(cs.shape, dtype=np.float64)
    lib.pa_oracle_e4m3_decode(_ptr(cs), _ptr(out), cs.size)
    return out


def append_kv_fp8(key, value, key_pages, value_pages, slot_mapping, page_size: int,
                  k_scale: float, v_scale: float) -> int:
    """Scatter key/value [B, H_kv, L_new, D] (uint16 bf16 bits) into uint8
    e4m3 pages [P, H_kv, page_size, D] in place: each element stored as the
    code of fp32(x) / fp32(scale). Returns the count of slots past the pool."""
    lib = _load()
    for a in (key, value):
        if a.dtype != np.uint16 or not a.flags.c_contiguous:
            raise TypeError("key/value must be contiguous uint16 (bf16 bit) arrays")
    for a in (key_pages, value_pages):
        if a.dtype != np.uint8 or not a.flags.c_contiguous:
            raise TypeError("FP8 pages must be contiguous uint8 arrays")
    slots = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    B, H_kv, L_new, D = key.shape
    P = key_pages.shape[0]
    assert value.shape == key.shape and value_pages.shape == key_pages.shape
    assert key_pages.shape[1:] == (H_kv, page_size, D)
    assert slots.shape == (B, L_new)
    return int(lib.pa_oracle_append_kv_fp8(_ptr(key), _ptr(value), _ptr(key_pages),
                                           _ptr(value_pages), _ptr(slots), B, L_new, H_kv,
                                           D, page_size, P, float(np.float32(k_scale)),
                                           float(np.float32(v_scale))))


def attention_fp8(query, key_pages, value_pages, k_scale: float, v_scale: float,
                  block_table, context_lens, page_size: int, scale: float | None = None,
                  causal: bool = True, rows=None, n_threads: int = 1) -> np.ndarray:
    """Paged attention in fp64 over e4m3 pages: every K (V) element is the
    exact value of its code times k_scale (v_scale); query uint16 bf16 bits.
    Otherwise as attention()."""
    q = bf16_bits_to_f64(query)
    kp = e4m3_decode(key_pages) * float(np.float32(k_scale))
    vp = e4m3_decode(value_pages) * float(np.float32(v_scale))
    return attention(q, kp, vp, block_table, context_lens, page_size, scale=scale,
                     causal=causal, rows=rows, n_threads=n_threads)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """uint16 bf16 bit patterns -> their exact values in fp64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
