"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers of this library only ever hold pointers handed to them by
another runtime (which owns all device memory), or run where cudaMalloc and
cudaFree are not allowed because they can stall the device mid-flight.
pa_decode_noalloc serves them with a fixed scratch array inside the library.
These tests call it through the C ABI and check it against pa_decode (the
entry point with a caller-provided workspace) on two calls in a row: the same
kernels over the same split, so the outputs must be bit-identical; both are
also compared with the oracle. Shapes beyond its scratch must be refused
without touching the output.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import (DeviceBatch, assert_close, check_no_device_error, host_bits, host_f64,
                      oracle_out, oracle_pages)

pytestmark = pytest.mark.gpu


def _lib():
    from paged_kv_attention_06_gb300 import binding
    lib = binding._lib
    vp, i32 = ctypes.c_void_p, ctypes.c_int32
    lib.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, ctypes.c_float, ctypes.c_int,
                                      vp, binding.pa_shape, i32, vp]
    lib.pa_decode_noalloc.restype = ctypes.c_int
    return binding, lib


@pytest.mark.parametrize("name", ["decode_b32_gqa7_ps16", "tiny_decode"])
def test_noalloc_matches_workspace_decode_on_two_calls(name):
    binding, lib = _lib()
    b = wl.make_workload(name)
    db = DeviceBatch(b)
    binding.pa_append_kv(db.key_new, db.value_new, db.key_pages, db.value_pages,
                         db.slot_mapping, b.page_size)
    max_ctx = int(b.context_lens.max())
    ref = binding.pa_decode(db.query, db.key_pages, db.value_pages, db.block_table,
                            db.context_lens, b.page_size, scale=b.scale, causal=b.causal,
                            max_context_len=max_ctx)
    shape = binding.make_shape(db.query.shape, db.key_pages.shape, db.block_table.shape[1])
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    ref_bits = host_bits(ref)
    kp, vp = oracle_pages(b)
    assert_close(host_f64(ref), oracle_out(b, kp, vp), f"{name} pa_decode")
    for call in range(2):
        out = torch.full_like(db.query, float("nan"))
        st = lib.pa_decode_noalloc(db.query.data_ptr(), db.key_pages.data_ptr(),
                                   db.value_pages.data_ptr(), db.block_table.data_ptr(),
                                   db.context_lens.data_ptr(), b.page_size, b.scale,
                                   int(b.causal), out.data_ptr(), shape, max_ctx, stream)
        assert st == 0, binding.status_string(st)
        torch.cuda.synchronize()
        check_no_device_error()
        assert np.array_equal(host_bits(out), ref_bits), f"call {call}: not bit-identical"
        assert_close(host_f64(out), oracle_out(b, kp, vp), f"{name} noalloc call {call}")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    binding, lib = _lib()
    b = wl.make_workload("tiny_decode")
    db = DeviceBatch(b)
    # 2048 requests x 8 KV heads: the partial-state slots alone exceed 32 MiB.
    shape = binding.pa_shape(2048, 64, 8, 128, 1, b.num_pages, db.block_table.shape[1])
    out = torch.full((8, 8), 3.0, dtype=torch.bfloat16, device="cuda")
    st = lib.pa_decode_noalloc(db.query.data_ptr(), db.key_pages.data_ptr(),
                               db.value_pages.data_ptr(), db.block_table.data_ptr(),
                               db.context_lens.data_ptr(), b.page_size, b.scale, 1,
                               out.data_ptr(), shape, 0, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == binding.PA_ERR_WORKSPACE
    assert torch.all(out == 3.0)
