"""Decode with several query rows per request (short chunks, speculative
tokens): the G * L rows of a (request, KV head) span several 16-row tiles,
and one segment carries up to four of them so that every K/V granule loaded
serves all of them (Week 3 Day 4, "Choose a Schedule for Each Query Shape":
expose parallelism across the cached context rather than reserving work for
rows that do not exist; "Task 2", the L <= 8 branch).

Compared with the oracle on every row, at shapes that take one, two and four
row tiles per segment (with an empty fourth tile, and two segments per KV
group), page sizes with and without the swizzled layout, head_dim 64 and
128, causal and not, and contexts long enough that segments straddle blocks
(so the merge pass combines multi-tile partial states)."""
import numpy as np
import pytest

import workloads as wl
from gpu_util import (DeviceBatch, assert_close, check_no_device_error, gpu_step, host_bits,
                      host_f64, oracle_out, oracle_pages)

pytestmark = pytest.mark.gpu

# (page_size, H_q, H_kv, D, L, causal): row tiles MT = ceil(G L / 16), tiles per
# segment 1 / 2 / 4 (3 tiles -> a group of 4 with one empty), segments per group
CASES = [
    (16, 28, 4, 128, 8, True),     # G 7: 56 rows, 4 tiles, one segment
    (16, 32, 8, 128, 8, True),     # G 4: 32 rows, 2 tiles
    (32, 28, 4, 128, 5, True),     # 35 rows: 3 tiles in a group of 4
    (128, 32, 2, 128, 6, True),    # G 16: 96 rows, 6 tiles, two segments (4 + 2)
    (4, 16, 2, 64, 8, True),       # head_dim 64, linear stage layout, 4 tiles
    (16, 8, 8, 128, 40, False),    # G 1, 40 rows, 3 tiles, all keys visible
    (1, 12, 4, 64, 7, True),       # pages of one token, 21 rows, 2 tiles
    (16, 28, 4, 128, 3, True),     # 21 rows, 2 tiles
]


def _lens(L, B, seed, max_len):
    rng = np.random.default_rng(seed)
    base = [L, L + 1, 63 + L, 64 + L, 1000, max_len]
    while len(base) < B:
        base.append(int(rng.integers(L, max_len)))
    return base[:B]


def _batch(ps, H_q, H_kv, D, L, causal, max_len=3000, B=8, seed=0):
    lens = _lens(L, B, seed + ps * 7 + H_q + L, max_len)
    return wl.build_batch("multirow", B=B, H_q=H_q, H_kv=H_kv, D=D, page_size=ps, L=L,
                          context_lens=lens, seed=seed + 101 * L + ps + D, L_new=min(L, 2),
                          causal=causal, placement="churn")


@pytest.mark.parametrize("ps,H_q,H_kv,D,L,causal", CASES)
def test_multirow_decode_matches_oracle(ps, H_q, H_kv, D, L, causal):
    b = _batch(ps, H_q, H_kv, D, L, causal)
    db = DeviceBatch(b)
    out = gpu_step(db, route="decode")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp),
                 f"multirow decode ps={ps} G={H_q // H_kv} D={D} L={L} causal={causal}")


def test_multirow_decode_one_long_request_many_blocks():
    """One request, one KV group of four row tiles, 30k keys: the segment is
    cut into one piece per block and the merge pass combines four tiles'
    partial states; repeated calls are bit-identical."""
    b = wl.build_batch("multirow_long", B=1, H_q=8, H_kv=1, D=128, page_size=16, L=8,
                       context_lens=[30000], seed=77, L_new=0)
    db = DeviceBatch(b)
    outs = [host_bits(gpu_step(db, route="decode", append=False)) for _ in range(3)]
    check_no_device_error()
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)
    assert_close(host_f64(gpu_step(db, route="decode", append=False)),
                 oracle_out(b, b.key_pages, b.value_pages), "multirow one long request")


def test_multirow_workspace_contents_and_relabelling():
    """Multi-tile segments: the result does not depend on what the workspace
    held, and relabelling physical pages gives the same bits."""
    import dataclasses

    import torch

    import paged_kv_attention_06_gb300 as pa
    b = _batch(16, 28, 4, 128, 8, True, B=6, seed=5)
    db = DeviceBatch(b)
    first = host_bits(gpu_step(db, route="decode"))
    shape = pa.make_shape(db.query.shape, db.key_pages.shape, db.block_table.shape[1])
    ws, _ = pa.decode_workspace(shape, db.query.device)
    ws.fill_(0xFF)
    again = host_bits(gpu_step(db, route="decode", append=False))
    assert np.array_equal(first, again)
    perm = np.random.default_rng(9).permutation(b.num_pages).astype(np.int32)
    kp, vp = np.empty_like(b.key_pages), np.empty_like(b.value_pages)
    kp[perm] = b.key_pages
    vp[perm] = b.value_pages
    bt = b.block_table.copy()
    bt[bt >= 0] = perm[bt[bt >= 0]]
    sm = b.slot_mapping.copy()
    ok = sm >= 0
    sm[ok] = perm[sm[ok] // b.page_size] * b.page_size + sm[ok] % b.page_size
    b2 = dataclasses.replace(b, key_pages=kp, value_pages=vp, block_table=bt, slot_mapping=sm)
    relab = host_bits(gpu_step(DeviceBatch(b2), route="decode"))
    check_no_device_error()
    assert np.array_equal(first, relab)
    del torch


@pytest.mark.parametrize("L,causal", [(40, True), (100, False), (257, True)])
def test_prefill_route_head_dim64(L, causal):
    """head_dim 64 prefill through pa_prefill at several lengths, causal and
    not (the pairs kernel's 64-column form at G = 4)."""
    b = wl.build_batch("prefill64", B=3, H_q=8, H_kv=2, D=64, page_size=16, L=L,
                       context_lens=[L, L + 100, L + 700], seed=L, causal=causal)
    db = DeviceBatch(b)
    out = gpu_step(db, route="prefill")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"prefill D=64 L={L}")


@pytest.mark.parametrize("L", [40, 257])
def test_prefill_head_dim64_one_head_per_group_whole_segments(L):
    """head_dim 64 with one query head per KV group has no pairs: the split-KV
    kernel with whole segments per block (four row tiles per segment)."""
    b = wl.build_batch("prefill64g1", B=3, H_q=4, H_kv=4, D=64, page_size=16, L=L,
                       context_lens=[L, L + 100, L + 700], seed=L + 1, causal=True)
    db = DeviceBatch(b)
    out = gpu_step(db, route="prefill")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"prefill D=64 G=1 L={L}")


@pytest.mark.parametrize("L,H_q,H_kv,max_len", [(12, 28, 4, 3000), (24, 28, 4, 3000),
                                                 (24, 8, 8, 3000), (32, 32, 8, 5000)])
def test_attention_routes_short_chunks_to_decode(L, H_q, H_kv, max_len):
    """pa_attention sends these chunk lengths to the decode schedule (the
    GB300 thresholds: L <= 24, or L <= 32 with contexts of 3072 tokens or
    more) and the result matches the oracle on every row."""
    import paged_kv_attention_06_gb300 as pa
    b = _batch(16, H_q, H_kv, 128, L, True, max_len=max_len, B=6, seed=L)
    db = DeviceBatch(b)
    shape = pa.make_shape(db.query.shape, db.key_pages.shape, db.block_table.shape[1])
    assert int(pa.binding._lib.pa_attention_route(shape, int(b.context_lens.max()))) == 0
    out = gpu_step(db, route="attention")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"pa_attention L={L} G={H_q // H_kv}")
