"""Error behaviour of the C ABI on a GPU. Nothing here faults, traps or hangs
a GPU: bad host arguments are rejected before any launch; bad device-side
values are clamped by the kernels and recorded in the device error word; the
timeout path is exercised by a bounded wait on a barrier nothing arrives at."""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import DeviceBatch, assert_close, gpu_step, host_bits, host_f64, oracle_out, oracle_pages

pytestmark = pytest.mark.gpu


def _pa():
    import paged_kv_attention_06_gb300 as pa
    return pa


def _call_decode(db, **over):
    pa = _pa()
    b = db.b
    shape = pa.make_shape(db.query.shape, db.key_pages.shape, db.block_table.shape[1])
    for k, v in over.pop("shape", {}).items():
        setattr(shape, k, v)
    out = over.pop("out")
    ws, need = pa.decode_workspace(shape if shape.head_dim in (64, 128) and shape.q_len > 0
                                   and shape.num_kv_heads > 0
                                   and shape.num_q_heads % shape.num_kv_heads == 0
                                   else pa.make_shape(db.query.shape, db.key_pages.shape,
                                                      db.block_table.shape[1]),
                                   db.query.device)
    args = dict(q=db.query.data_ptr(), k=db.key_pages.data_ptr(), v=db.value_pages.data_ptr(),
                bt=db.block_table.data_ptr(), cl=db.context_lens.data_ptr(), ps=b.page_size,
                scale=b.scale, causal=1, out=out.data_ptr(), shape=shape,
                mcl=int(b.context_lens.max()), ws=ws.data_ptr(), wsb=need,
                stream=torch.cuda.current_stream().cuda_stream)
    args.update(over)
    return pa.binding._lib.pa_decode(args["q"], args["k"], args["v"], args["bt"], args["cl"],
                                     args["ps"], args["scale"], args["causal"], args["out"],
                                     args["shape"], args["mcl"], args["ws"], args["wsb"],
                                     args["stream"])


@pytest.mark.parametrize("bad,expect", [
    (dict(scale=0.0), 1), (dict(scale=float("nan")), 1), (dict(scale=-1.0), 1),
    (dict(q=None), 1), (dict(bt=None), 1), (dict(ws=None), 3), (dict(wsb=16), 3),
    (dict(ps=3), 2), (dict(ps=512), 2), (dict(shape=dict(head_dim=96)), 2),
    (dict(shape=dict(num_q_heads=6, num_kv_heads=4)), 2), (dict(shape=dict(batch=0)), 1),
])
def test_host_rejects_bad_arguments_and_touches_nothing(bad, expect):
    b = wl.make_workload("tiny_decode")
    db = DeviceBatch(b)
    out = torch.full_like(db.query, 7.0)
    torch.cuda.synchronize()
    st = _call_decode(db, out=out, **bad)
    torch.cuda.synchronize()
    assert st == expect
    assert torch.all(out == 7.0)
    assert _pa().pa_get_device_error() == (0, 0)


def test_misaligned_pointer_rejected():
    b = wl.make_workload("tiny_decode")
    db = DeviceBatch(b)
    out = torch.full_like(db.query, 7.0)
    st = _call_decode(db, out=out, q=db.query.data_ptr() + 2)
    assert st == 1 and torch.all(out == 7.0)


def test_bad_page_id_is_flagged_not_faulted():
    pa = _pa()
    b = wl.make_workload("tiny_decode")
    bt = b.block_table.copy()
    bt[0, 1] = b.num_pages + 5               # inside the context: will be read
    import dataclasses
    db = DeviceBatch(dataclasses.replace(b, block_table=bt))
    gpu_step(db, route="decode", append=False)
    st, flags = pa.pa_get_device_error()
    assert st == pa.PA_ERR_DEVICE_BOUNDS and flags & pa.PA_DEVERR_PAGE_ID
    gpu_step(db, route="prefill", append=False)
    st, flags = pa.pa_get_device_error()
    assert st == pa.PA_ERR_DEVICE_BOUNDS and flags & pa.PA_DEVERR_PAGE_ID
    assert pa.pa_get_device_error() == (0, 0)        # read-and-clear
    torch.cuda.synchronize()


def test_bad_context_len_is_flagged():
    pa = _pa()
    b = wl.make_workload("tiny_decode")
    import dataclasses
    cl = b.context_lens.copy()
    cl[1] = b.max_pages * b.page_size + 3
    db = DeviceBatch(dataclasses.replace(b, context_lens=cl))
    gpu_step(db, route="decode", append=False)
    st, flags = pa.pa_get_device_error()
    assert st == pa.PA_ERR_DEVICE_BOUNDS and flags & pa.PA_DEVERR_CONTEXT_LEN


def test_bad_slot_is_flagged_and_skipped():
    pa = _pa()
    b = wl.build_batch("slots", B=3, H_q=4, H_kv=2, D=64, page_size=4, L=2,
                       context_lens=[5, 9, 2], seed=1, L_new=2)
    sm = b.slot_mapping.copy()
    sm[1, 0] = b.num_pages * b.page_size + 1   # beyond the pool
    sm[2, 1] = -1                              # padding token
    import dataclasses
    b2 = dataclasses.replace(b, slot_mapping=sm)
    db = DeviceBatch(b2)
    pa.pa_append_kv(db.key_new, db.value_new, db.key_pages, db.value_pages, db.slot_mapping,
                    b.page_size)
    st, flags = pa.pa_get_device_error()
    assert st == pa.PA_ERR_DEVICE_BOUNDS and flags == pa.PA_DEVERR_SLOT
    kp, vp = oracle_pages(b2)                  # the oracle skips the same two tokens
    assert np.array_equal(host_bits(db.key_pages), kp)
    assert np.array_equal(host_bits(db.value_pages), vp)


def test_wait_timeout_is_reported_and_context_survives():
    pa = _pa()
    b = wl.make_workload("tiny_decode")
    db = DeviceBatch(b)
    pa.pa_debug_arm_wait_timeout()
    out = gpu_step(db, route="decode")
    st, flags = pa.pa_get_device_error()
    assert st == pa.PA_ERR_DEVICE_TIMEOUT and flags == pa.PA_DEVERR_TIMEOUT
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), "after timeout")
    out2 = gpu_step(db, route="decode", append=False)
    assert pa.pa_get_device_error() == (0, 0)
    assert_close(host_f64(out2), oracle_out(b, kp, vp), "next call")
