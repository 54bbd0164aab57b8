"""The dense baseline on the GPU: pa_gather_kv (pages -> dense K/V) against
the oracle's gather, bit for bit, and pa_decode_dense over the gathered rows
against pa_decode over the pages (same kernel, same keys: bit-identical) and
against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import (DeviceBatch, assert_close, check_no_device_error, dev, host_bits, host_f64)

pytestmark = pytest.mark.gpu


def _dense_len(b):
    return max(64, -(-int(b.context_lens.max()) // 64) * 64)


@pytest.mark.parametrize("name", ["tiny_decode", "decode_b32_gqa7_ps16", "decode_b64_ps128"])
def test_gather_bit_exact_vs_oracle(name):
    import paged_kv_attention_06_gb300 as pa
    b = wl.make_workload(name)
    db = DeviceBatch(b)
    N = _dense_len(b)
    fill = 0x7FC1          # a NaN pattern: rows past a context must stay as they were
    kd = torch.full((b.B, b.H_kv, N, b.D), fill, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    vd = kd.clone()
    pa.pa_gather_kv(db.key_pages, db.value_pages, db.block_table, db.context_lens, b.page_size, N,
                    key_dense=kd, value_dense=vd)
    check_no_device_error()
    want_k = oracle.gather(b.key_pages, b.block_table, b.context_lens, b.page_size, N, fill=fill)
    want_v = oracle.gather(b.value_pages, b.block_table, b.context_lens, b.page_size, N, fill=fill)
    assert np.array_equal(host_bits(kd), want_k)
    assert np.array_equal(host_bits(vd), want_v)


@pytest.mark.parametrize("ps", [1, 4, 16, 128, 256])
def test_gather_page_sizes(ps):
    import paged_kv_attention_06_gb300 as pa
    lens = [300, 1, 0, 257, 64]
    b = wl.build_batch("gather", B=5, H_q=8, H_kv=2, D=64, page_size=ps, L=1, context_lens=lens,
                       seed=ps, L_new=0, placement="churn")
    db = DeviceBatch(b)
    N = 320
    kd, vd = pa.pa_gather_kv(db.key_pages, db.value_pages, db.block_table, db.context_lens, ps, N,
                             key_dense=torch.zeros((5, 2, N, 64), dtype=torch.bfloat16, device="cuda"),
                             value_dense=torch.zeros((5, 2, N, 64), dtype=torch.bfloat16, device="cuda"))
    check_no_device_error()
    assert np.array_equal(host_bits(kd), oracle.gather(b.key_pages, b.block_table, b.context_lens, ps, N))
    assert np.array_equal(host_bits(vd), oracle.gather(b.value_pages, b.block_table, b.context_lens, ps, N))


@pytest.mark.parametrize("name", ["tiny_decode", "decode_b32_gqa7_ps16", "decode_b64_ps128"])
def test_dense_decode_bit_identical_to_paged_decode(name):
    import paged_kv_attention_06_gb300 as pa
    b = wl.make_workload(name)
    db = DeviceBatch(b)
    N = _dense_len(b)
    kd, vd = pa.pa_gather_kv(db.key_pages, db.value_pages, db.block_table, db.context_lens,
                             b.page_size, N)
    maxc = int(b.context_lens.max())
    paged = pa.pa_decode(db.query, db.key_pages, db.value_pages, db.block_table, db.context_lens,
                         b.page_size, scale=b.scale, causal=b.causal, max_context_len=maxc)
    dense = pa.pa_decode_dense(db.query, kd, vd, db.context_lens, scale=b.scale, causal=b.causal,
                               max_context_len=maxc)
    check_no_device_error()
    assert np.array_equal(host_bits(paged), host_bits(dense))


def test_dense_decode_vs_oracle_multi_row_causal():
    import paged_kv_attention_06_gb300 as pa
    b = wl.build_batch("dense_l4", B=3, H_q=8, H_kv=2, D=128, page_size=16, L=4,
                       context_lens=[70, 4, 129], seed=21, L_new=0)
    db = DeviceBatch(b)
    N = 192
    kd, vd = pa.pa_gather_kv(db.key_pages, db.value_pages, db.block_table, db.context_lens, 16, N)
    out = pa.pa_decode_dense(db.query, kd, vd, db.context_lens, scale=b.scale, causal=True)
    check_no_device_error()
    ref = oracle.attention(b.query, b.key_pages, b.value_pages, b.block_table, b.context_lens, 16,
                           scale=b.scale, causal=True)
    assert_close(host_f64(out), ref, "dense decode")


def test_gather_flags_bad_page_and_long_context():
    import paged_kv_attention_06_gb300 as pa
    b = wl.make_workload("tiny_decode")
    db = DeviceBatch(b)
    bt = db.block_table.clone()
    bt[0, 1] = b.num_pages + 3
    pa.pa_gather_kv(db.key_pages, db.value_pages, bt, db.context_lens, b.page_size, 64)
    st, flags = pa.pa_get_device_error()
    assert st == pa.PA_ERR_DEVICE_BOUNDS and flags & pa.PA_DEVERR_PAGE_ID
    pa.pa_gather_kv(db.key_pages, db.value_pages, db.block_table, db.context_lens, b.page_size, 8)
    st, flags = pa.pa_get_device_error()
    assert st != 0 and flags & pa.PA_DEVERR_CONTEXT_LEN


def test_dense_decode_rejects_bad_dense_len():
    import paged_kv_attention_06_gb300 as pa
    b = wl.make_workload("tiny_decode")
    db = DeviceBatch(b)
    kd = torch.zeros((b.B, b.H_kv, 96, b.D), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pa.PagedAttentionError):
        pa.pa_decode_dense(db.query, kd, kd.clone(), db.context_lens, scale=b.scale)
