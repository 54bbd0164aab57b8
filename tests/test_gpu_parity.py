"""GPU path vs the fp64 oracle, element by element, through the C ABI.

Append and indexing must be bit-exact; attention outputs must satisfy
max |err| <= 2e-2 and mean |err| <= 2e-3 against the oracle on the same
seeded inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import (DeviceBatch, assert_close, check_no_device_error, gpu_step, host_bits,
                      host_f64, oracle_out, oracle_pages)

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------------------
# Named workloads, end to end (append, then the dispatching entry point)


def test_tiny_decode_full():
    b = wl.make_workload("tiny_decode")
    db = DeviceBatch(b)
    out = gpu_step(db)
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert np.array_equal(host_bits(db.key_pages), kp)
    assert np.array_equal(host_bits(db.value_pages), vp)
    assert_close(host_f64(out), oracle_out(b, kp, vp), "tiny_decode")


@pytest.mark.parametrize("name", ["decode_b32_gqa7_ps16", "decode_b64_ps128", "decode_long_b8"])
def test_decode_workloads_every_row(name):
    b = wl.make_workload(name)
    db = DeviceBatch(b)
    out = gpu_step(db)
    check_no_device_error()
    kp, vp = oracle_pages(b)
    # the append touches B rows per KV head: compare the whole pools bit for bit
    assert np.array_equal(host_bits(db.key_pages), kp)
    assert np.array_equal(host_bits(db.value_pages), vp)
    assert_close(host_f64(out), oracle_out(b, kp, vp), name)


def test_prefill_chunk_sampled_rows():
    b = wl.make_workload("prefill_chunk512")
    db = DeviceBatch(b)
    out = gpu_step(db)
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert np.array_equal(host_bits(db.key_pages), kp)
    assert np.array_equal(host_bits(db.value_pages), vp)
    rng = np.random.default_rng(0)
    rows = []
    for r in range(b.B):
        for i in sorted(set([0, 1, 63, 64, 127, 128, 255, 256, 383, 510, 511] +
                            list(rng.integers(0, b.L, 6)))):
            for h in range(b.H_q):
                rows.append((r, h, i))
    rows = np.asarray(rows, dtype=np.int32)
    ref = oracle_out(b, kp, vp, rows=rows)
    got = host_f64(out)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, ref, "prefill_chunk512 sampled")
    assert torch.isfinite(out.float()).all()


# ----------------------------------------------------------------------------
# Sweeps over page sizes, GQA ratios, head dims, query lengths and ragged
# context lengths at page boundaries


def _boundary_lens(ps, L, B, seed, max_len=700):
    rng = np.random.default_rng(seed)
    cands = [L, ps - 1, ps, ps + 1, 2 * ps, 2 * ps + 1, 63, 64, 65, 127, 129, 300]
    lens = [max(L, int(c)) for c in cands if c >= 1]
    while len(lens) < B:
        lens.append(int(rng.integers(L, max_len)))
    return [min(x, max_len) for x in lens[:B]]


SWEEP = [
    # (page_size, H_q, H_kv, D, L)
    (1, 8, 8, 64, 1), (2, 8, 4, 128, 1), (4, 4, 2, 64, 1), (16, 28, 4, 128, 1),
    (16, 32, 8, 128, 2), (64, 16, 4, 64, 1), (128, 32, 8, 128, 1), (256, 14, 2, 128, 1),
    (16, 16, 1, 128, 1), (16, 32, 1, 64, 1), (8, 12, 4, 128, 8), (32, 28, 4, 128, 5),
    (4, 8, 1, 128, 3), (128, 7, 7, 64, 2),
]


@pytest.mark.parametrize("ps,H_q,H_kv,D,L", SWEEP)
@pytest.mark.parametrize("route", ["decode", "prefill"])
def test_sweep_against_oracle(ps, H_q, H_kv, D, L, route):
    B = 12
    lens = _boundary_lens(ps, L, B, seed=ps * 131 + H_q * 7 + D + L)
    b = wl.build_batch("sweep", B=B, H_q=H_q, H_kv=H_kv, D=D, page_size=ps, L=L,
                       context_lens=lens, seed=ps + 17 * L + D, L_new=min(L, 1))
    db = DeviceBatch(b)
    out = gpu_step(db, route=route)
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"{route} ps={ps} G={H_q // H_kv} L={L}")


@pytest.mark.parametrize("L,causal", [(9, True), (16, True), (33, False), (64, True), (130, True)])
@pytest.mark.parametrize("ps", [16, 128])
def test_prefill_lengths(L, causal, ps):
    B = 5
    rng = np.random.default_rng(L + ps)
    lens = [L, L + 1, L + ps, L + 200, L + int(rng.integers(0, 600))]
    b = wl.build_batch("prefill", B=B, H_q=8, H_kv=2, D=128, page_size=ps, L=L,
                       context_lens=lens, seed=3 * L + ps, causal=causal, placement="churn")
    db = DeviceBatch(b)
    out = gpu_step(db, route="prefill")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"prefill L={L} ps={ps}")


# ----------------------------------------------------------------------------
# Invariants of Week 3 Day 4, "What Must Hold"


def _relabelled(b: wl.PagedBatch, seed: int) -> wl.PagedBatch:
    perm = np.random.default_rng(seed).permutation(b.num_pages).astype(np.int32)
    kp, vp = np.empty_like(b.key_pages), np.empty_like(b.value_pages)
    kp[perm] = b.key_pages
    vp[perm] = b.value_pages
    bt = b.block_table.copy()
    m = bt >= 0
    bt[m] = perm[bt[m]]
    sm = b.slot_mapping.copy()
    ok = sm >= 0
    sm[ok] = perm[sm[ok] // b.page_size] * b.page_size + sm[ok] % b.page_size
    import dataclasses
    return dataclasses.replace(b, key_pages=kp, value_pages=vp, block_table=bt, slot_mapping=sm)


@pytest.mark.parametrize("name", ["tiny_decode", "decode_b32_gqa7_ps16"])
def test_physical_relabelling_bit_identical(name):
    b = wl.make_workload(name)
    out1 = host_bits(gpu_step(DeviceBatch(b)))
    out2 = host_bits(gpu_step(DeviceBatch(_relabelled(b, 5))))
    check_no_device_error()
    assert np.array_equal(out1, out2)


@pytest.mark.parametrize("pattern", [0x7FC0, 0x7F80, 0xFF80, 0x0000])
@pytest.mark.parametrize("route", ["decode", "prefill"])
def test_stale_slots_never_affect_output(pattern, route):
    b = wl.build_batch("stale", B=6, H_q=16, H_kv=4, D=128, page_size=16, L=3,
                       context_lens=[3, 17, 31, 64, 100, 250], seed=77, L_new=0)
    out1 = host_bits(gpu_step(DeviceBatch(b), route=route))
    used = np.zeros((b.num_pages, b.page_size), dtype=bool)
    for r in range(b.B):
        for j in range(int(b.context_lens[r])):
            used[b.block_table[r, j // b.page_size], j % b.page_size] = True
    pages, slots = np.nonzero(~used)
    kp, vp = b.key_pages.copy(), b.value_pages.copy()
    kp[pages, :, slots, :] = pattern
    vp[pages, :, slots, :] = pattern
    import dataclasses
    b2 = dataclasses.replace(b, key_pages=kp, value_pages=vp)
    out2 = host_bits(gpu_step(DeviceBatch(b2), route=route))
    check_no_device_error()
    assert np.array_equal(out1, out2)


def test_padding_entries_never_read():
    b = wl.make_workload("tiny_decode", pad_value=-1)
    out1 = host_bits(gpu_step(DeviceBatch(b)))
    import dataclasses
    bt = b.block_table.copy()
    bt[bt < 0] = 2**30                        # far outside the pool
    out2 = host_bits(gpu_step(DeviceBatch(dataclasses.replace(b, block_table=bt))))
    check_no_device_error()                   # never dereferenced, so never flagged
    assert np.array_equal(out1, out2)


def test_shared_pages_between_requests():
    """Two requests point at the same physical prefix pages (explicit
    sharing, as in prefix caching); reads of aliased pages are legal."""
    ps, n_shared = 16, 48
    b = wl.build_batch("alias", B=3, H_q=8, H_kv=2, D=128, page_size=ps, L=1,
                       context_lens=[100, 70, 48], seed=5, L_new=0)
    bt = b.block_table.copy()
    bt[1, :n_shared // ps] = bt[0, :n_shared // ps]
    bt[2, :n_shared // ps] = bt[0, :n_shared // ps]
    import dataclasses
    b2 = dataclasses.replace(b, block_table=bt)
    out = gpu_step(DeviceBatch(b2))
    check_no_device_error()
    assert_close(host_f64(out), oracle_out(b2, b2.key_pages, b2.value_pages), "aliased")


def test_empty_contexts_and_rows_without_keys():
    b = wl.build_batch("empty", B=4, H_q=8, H_kv=4, D=64, page_size=4, L=4,
                       context_lens=[0, 2, 4, 9], seed=9, L_new=0)
    for route in ("decode", "prefill"):
        out = host_f64(gpu_step(DeviceBatch(b), route=route))
        check_no_device_error()
        ref = oracle_out(b, b.key_pages, b.value_pages)
        assert np.all(out[0] == 0)             # n = 0
        assert np.all(out[1, :, :2] == 0)      # rows at positions -2, -1
        assert_close(out, ref, route)


@pytest.mark.parametrize("ps,L,route", [(16, 1, "decode"), (16, 200, "prefill"), (128, 1, "decode"),
                                        (128, 130, "prefill"), (16, 130, "prefill_split")])
def test_full_tables_in_a_full_pool(ps, L, route):
    """Every block-table row full (each context a whole number of pages, the
    longest filling max_pages), every page of the pool in use (no slack, so
    the pool's last page is read too): the edge where a page walk ends exactly
    at the table's and the pool's last entries."""
    n_full = 12 * ps
    lens = [n_full, n_full, 6 * ps, n_full]
    b = wl.build_batch(f"full_{ps}_{L}", B=4, H_q=16, H_kv=4, D=128, page_size=ps, L=L,
                       context_lens=lens, seed=ps + L, L_new=min(L, 2), pool_slack=0.0)
    assert b.num_pages == sum(n // ps for n in lens)
    assert int((b.block_table >= 0).sum()) == b.num_pages
    db = DeviceBatch(b)
    out = gpu_step(db, route=route)
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert np.array_equal(host_bits(db.key_pages), kp)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"full tables ps={ps} L={L} {route}")


def test_decode_and_prefill_routes_agree():
    b = wl.build_batch("routes", B=8, H_q=32, H_kv=8, D=128, page_size=16, L=4,
                       context_lens=[5, 77, 300, 1000, 2047, 16, 17, 4096], seed=21, L_new=0)
    db = DeviceBatch(b)
    dec = host_f64(gpu_step(db, route="decode"))
    pre = host_f64(gpu_step(db, route="prefill"))
    ref = oracle_out(b, b.key_pages, b.value_pages)
    assert_close(dec, ref, "decode")
    assert_close(pre, ref, "prefill")


def test_workspace_contents_do_not_matter():
    """Repeated calls are bit-identical, whatever the workspace held before
    (the decode reads only partial states it wrote in the same call)."""
    import paged_kv_attention_06_gb300 as pa
    b = wl.make_workload("decode_b32_gqa7_ps16")
    db = DeviceBatch(b)
    outs = [host_bits(gpu_step(db, route="decode", append=False)) for _ in range(2)]
    shape = pa.make_shape(db.query.shape, db.key_pages.shape, db.block_table.shape[1])
    ws, need = pa.decode_workspace(shape, db.query.device)
    ws.fill_(0xFF)                              # NaN patterns everywhere
    outs.append(host_bits(gpu_step(db, route="decode", append=False)))
    ws.random_(0, 256)
    outs.append(host_bits(gpu_step(db, route="decode", append=False)))
    check_no_device_error()
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


@pytest.mark.parametrize("n_ctx,H_q", [(40000, 8), (9000, 4), (200, 2)])
def test_one_segment_split_over_blocks(n_ctx, H_q):
    """A single (request, KV head) segment cut into one piece per block: the
    pieces publish their partial states and whichever block sees them all
    merges. Repeated calls are bit-identical whichever block merged."""
    b = wl.build_batch("one_segment", B=1, H_q=H_q, H_kv=1, D=128, page_size=16, L=1,
                       context_lens=[n_ctx], seed=31, L_new=0)
    db = DeviceBatch(b)
    outs = [host_bits(gpu_step(db, route="decode", append=False)) for _ in range(6)]
    check_no_device_error()
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)
    ref = oracle_out(b, b.key_pages, b.value_pages)
    got = host_f64(gpu_step(db, route="decode", append=False))
    assert_close(got, ref, f"one segment, {n_ctx} keys")


def test_non_default_stream():
    b = wl.make_workload("tiny_decode")
    db = DeviceBatch(b)
    s = torch.cuda.Stream()
    import paged_kv_attention_06_gb300 as pa
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        pa.pa_append_kv(db.key_new, db.value_new, db.key_pages, db.value_pages,
                        db.slot_mapping, b.page_size)
        out = pa.pa_attention(db.query, db.key_pages, db.value_pages, db.block_table,
                              db.context_lens, b.page_size, scale=b.scale, max_context_len=10)
    s.synchronize()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), "stream")


# ----------------------------------------------------------------------------
# The tensor-core prefill path (head_dim 128, page_size >= 8) at its edges


@pytest.fixture(params=[1, 2, 0, 4], ids=["one_head", "head_pairs", "split", "tail_pieces"])
def prefill_variant(request):
    """Runs the test under each tensor-core prefill kernel (pairs need an even
    group size; odd groups take the one-head kernel under either setting; the
    split kernel runs through pa_prefill_split with a workspace, and odd
    groups there also fall back to the one-head kernel; the pairs kernel with
    tail pieces runs through pa_attention with its workspace on a grid of two
    thirds of the items). Yields the route for gpu_step."""
    import paged_kv_attention_06_gb300 as pa
    prev = pa.pa_debug_prefill_variant(request.param)
    yield {0: "prefill_split", 4: "attention"}.get(request.param, "prefill")
    pa.pa_debug_prefill_variant(prev)


@pytest.mark.parametrize("ps", [1, 2, 4, 8, 16, 64, 128, 256])   # below 8: rows copied one by one
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (6, 2)])   # group of 4 / 3
def test_tc_prefill_page_sizes(ps, causal, H_q, H_kv, prefill_variant):
    lens = [200, 129, 513, 300]
    b = wl.build_batch("tcprefill", B=4, H_q=H_q, H_kv=H_kv, D=128, page_size=ps, L=129,
                       context_lens=lens, seed=ps + int(causal), causal=causal,
                       placement="churn")
    out = gpu_step(DeviceBatch(b), route=prefill_variant)
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"tc prefill ps={ps} causal={causal}")


@pytest.mark.parametrize("ps", [1, 4, 8, 16, 128, 256])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (6, 2), (4, 1), (4, 4)])   # groups of 4 / 3 / 4 / 1
def test_tc_prefill_head_dim64(ps, causal, H_q, H_kv):
    """head_dim 64 on the pairs kernel (one 64-column half per row, four
    k-steps for the scores, N = 64 for P V): several query tiles, a ragged
    last tile, contexts across page boundaries, odd and even groups, and one
    query head per KV group (that head in both halves of a block)."""
    lens = [200, 129, 700, 300]
    b = wl.build_batch("tcprefill64", B=4, H_q=H_q, H_kv=H_kv, D=64, page_size=ps, L=129,
                       context_lens=lens, seed=ps + 3 * int(causal) + H_q, causal=causal,
                       placement="churn")
    out = gpu_step(DeviceBatch(b), route="prefill")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"tc prefill D=64 ps={ps} causal={causal}")


@pytest.mark.parametrize("H_q,H_kv", [(4, 2), (6, 2), (16, 2)])   # 1600 / 3200 / 6400 items
def test_tc_prefill_many_query_tiles_unranked(H_q, H_kv):
    """More (request, query tile) pairs than the pairs kernel ranks (384):
    400 requests of two query tiles take the tiles last to first without the
    ranking, and more items than 32 per SM grow the grid; every request's
    first, boundary and last rows against the oracle."""
    rng = np.random.default_rng(31)
    lens = [int(x) for x in rng.integers(130, 420, 400)]
    b = wl.build_batch("manytiles", B=400, H_q=H_q, H_kv=H_kv, D=128, page_size=16, L=130,
                       context_lens=lens, seed=32, L_new=0, placement="churn")
    out = host_f64(gpu_step(DeviceBatch(b), route="prefill"))
    check_no_device_error()
    rows = np.asarray([(r, h, i) for r in range(b.B) for h in range(b.H_q)
                       for i in (0, 127, 128, 129)], dtype=np.int32)
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, oracle_out(b, b.key_pages, b.value_pages, rows=rows), "tc prefill 800 tiles")


def test_tc_prefill_head_dim64_rows_without_keys():
    """head_dim 64 on the pairs kernel: contexts of 0, 50 and 199 tokens under
    200 query rows (rows at negative positions see no key: zeros), page size 8."""
    b = wl.build_batch("tcempty64", B=3, H_q=8, H_kv=2, D=64, page_size=8, L=200,
                       context_lens=[0, 50, 199], seed=41, L_new=0)
    out = host_f64(gpu_step(DeviceBatch(b), route="prefill"))
    check_no_device_error()
    assert np.all(out[0] == 0)
    assert np.all(out[1, :, :150] == 0) and np.all(out[2, :, :1] == 0)
    assert_close(out, oracle_out(b, b.key_pages, b.value_pages), "tc prefill D=64 empty rows")


@pytest.mark.parametrize("H_q,H_kv", [(28, 4), (10, 2)])   # groups of 7 / 5
def test_tc_prefill_odd_groups(H_q, H_kv, prefill_variant):
    """Odd group sizes: the head-pairs kernel runs each group's last head in a
    pair of its own (computed twice, written once); every head of every group
    against the oracle, over several query tiles."""
    lens = [300, 1000, 260]
    b = wl.build_batch("tcodd", B=3, H_q=H_q, H_kv=H_kv, D=128, page_size=16, L=260,
                       context_lens=lens, seed=H_q, causal=True, placement="churn")
    out = gpu_step(DeviceBatch(b), route=prefill_variant)
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"tc prefill G={H_q // H_kv}")


@pytest.mark.parametrize("H_q,H_kv", [(4, 4), (4, 2)])   # group of 1 / 2
def test_tc_prefill_rows_without_keys_and_empty_context(H_q, H_kv, prefill_variant):
    # L = 200 rows after contexts of 0, 50 and 199 tokens: rows at negative
    # positions see no key and must return zeros.
    b = wl.build_batch("tcempty", B=3, H_q=H_q, H_kv=H_kv, D=128, page_size=16, L=200,
                       context_lens=[0, 50, 199], seed=4, L_new=0)
    out = host_f64(gpu_step(DeviceBatch(b), route=prefill_variant))
    check_no_device_error()
    assert np.all(out[0] == 0)
    assert np.all(out[1, :, :150] == 0) and np.all(out[2, :, :1] == 0)
    assert_close(out, oracle_out(b, b.key_pages, b.value_pages), "tc prefill empty rows")


def test_tc_prefill_bad_page_id_is_flagged(prefill_variant):
    import dataclasses
    import paged_kv_attention_06_gb300 as pa
    b = wl.build_batch("tcbad", B=2, H_q=4, H_kv=2, D=128, page_size=16, L=32,
                       context_lens=[100, 40], seed=8, L_new=0)
    bt = b.block_table.copy()
    bt[0, 2] = b.num_pages + 7
    gpu_step(DeviceBatch(dataclasses.replace(b, block_table=bt)), route=prefill_variant)
    st, flags = pa.pa_get_device_error()
    assert st == pa.PA_ERR_DEVICE_BOUNDS and flags & pa.PA_DEVERR_PAGE_ID


def test_tc_prefill_long_context_gqa(prefill_variant):
    b = wl.build_batch("tclong", B=2, H_q=16, H_kv=2, D=128, page_size=16, L=384,
                       context_lens=[3000, 1500], seed=12, placement="permutation")
    db = DeviceBatch(b)
    out = gpu_step(db, route=prefill_variant)
    check_no_device_error()
    kp, vp = oracle_pages(b)
    rows = np.asarray([(r, h, i) for r in range(2) for h in range(16)
                       for i in (0, 1, 127, 128, 255, 256, 383)], dtype=np.int32)
    got = host_f64(out)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, oracle_out(b, kp, vp, rows=rows), "tc prefill long")


# ----------------------------------------------------------------------------
# The split prefill kernel (K/V tiles of all query tiles spread evenly over
# one block per SM; items cut by a block boundary are merged from their
# pieces' states)


def _sampled_rows(b, rng, extra=6):
    rows = []
    for r in range(b.B):
        for i in sorted(set([0, 1, 63, 64, 127, 128, b.L // 2, b.L - 2, b.L - 1] +
                            list(rng.integers(0, b.L, extra)))):
            if 0 <= i < b.L:
                for h in range(b.H_q):
                    rows.append((r, h, i))
    return np.asarray(rows, dtype=np.int32)


def test_split_prefill_chunk512_sampled_rows():
    b = wl.make_workload("prefill_chunk512")
    db = DeviceBatch(b)
    out = gpu_step(db, route="prefill_split")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    rows = _sampled_rows(b, np.random.default_rng(1))
    got = host_f64(out)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, oracle_out(b, kp, vp, rows=rows), "split prefill_chunk512")


@pytest.mark.parametrize("causal", [True, False])
def test_split_prefill_items_cut_into_many_pieces(causal):
    # One request, 2 query tiles x 4 head pairs = 8 items of ~64 K/V tiles
    # over ~150 blocks: every item is cut into ~19 pieces.
    b = wl.build_batch("splitlong", B=1, H_q=8, H_kv=2, D=128, page_size=16, L=256,
                       context_lens=[8000], seed=21, causal=causal, placement="permutation")
    out = gpu_step(DeviceBatch(b), route="prefill_split")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    rows = _sampled_rows(b, np.random.default_rng(2), extra=10)
    got = host_f64(out)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, oracle_out(b, kp, vp, rows=rows), f"split many pieces causal={causal}")


@pytest.mark.parametrize("H_q,H_kv", [(14, 2), (6, 2)])   # groups of 7 / 3
def test_split_prefill_odd_groups_cut_into_pieces(H_q, H_kv):
    """Odd group sizes on the split kernel: each group's last pair repeats its
    last head, the items are cut into many pieces, and every query head (the
    repeated last ones included) matches the oracle."""
    b = wl.build_batch("splitodd", B=1, H_q=H_q, H_kv=H_kv, D=128, page_size=16, L=256,
                       context_lens=[6000], seed=H_q, causal=True, placement="permutation")
    out = gpu_step(DeviceBatch(b), route="prefill_split")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    rng = np.random.default_rng(3)
    rows = np.asarray([(0, h, int(i)) for h in range(b.H_q)
                       for i in [0, 127, 128, 255] + list(rng.integers(0, b.L, 4))], dtype=np.int32)
    got = host_f64(out)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, oracle_out(b, kp, vp, rows=rows), f"split odd group G={H_q // H_kv}")


def test_split_prefill_fewer_units_than_blocks():
    # 3 short requests: far fewer K/V tiles than blocks (most blocks get an
    # empty range and leave at once); every row compared.
    b = wl.build_batch("splitsmall", B=3, H_q=4, H_kv=2, D=128, page_size=16, L=20,
                       context_lens=[20, 150, 300], seed=22, placement="churn")
    out = gpu_step(DeviceBatch(b), route="prefill_split")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), "split few units")


def test_split_prefill_workspace_contents_and_repeat():
    """Any workspace contents give the same output, and two runs are bit
    identical (the merge order is fixed)."""
    import paged_kv_attention_06_gb300 as pa
    b = wl.build_batch("splitws", B=2, H_q=8, H_kv=2, D=128, page_size=16, L=300,
                       context_lens=[2500, 900], seed=23, placement="churn")
    db = DeviceBatch(b)
    gpu_step(db, route="prefill_split")            # the append, once
    shape = pa.make_shape(db.query.shape, db.key_pages.shape, db.block_table.shape[1])
    need = pa.pa_prefill_workspace_bytes(shape, b.page_size)
    assert need > 0
    outs = []
    for fill in (0x00, 0xFF, 0x5A):
        ws = torch.full((need,), fill, dtype=torch.uint8, device="cuda")
        outs.append(pa.pa_prefill_split(db.query, db.key_pages, db.value_pages, db.block_table,
                                        db.context_lens, b.page_size, scale=b.scale,
                                        causal=b.causal, workspace=ws))
        check_no_device_error()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    kp, vp = b.key_pages.copy(), b.value_pages.copy()
    oracle.append_kv(b.key_new, b.value_new, kp, vp, b.slot_mapping, b.page_size)
    assert_close(host_f64(outs[0]), oracle_out(b, kp, vp), "split workspace contents")


@pytest.fixture(params=[4, 5], ids=["receiver_first", "donor_first"])
def tail_pieces(request):
    """pa_attention's pairs kernel on a grid of two thirds of the items, so
    that the blocks with two items hand the last tiles of their second one to
    blocks with one (test setting 4; setting 5 runs the pieces last, so that
    the donors usually arrive first and the receiving blocks merge)."""
    import paged_kv_attention_06_gb300 as pa
    prev = pa.pa_debug_prefill_variant(request.param)
    yield
    pa.pa_debug_prefill_variant(prev)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("H_q,H_kv", [(8, 2), (6, 2)])     # groups of 4 / 3
def test_tail_pieces_every_row(causal, H_q, H_kv, tail_pieces):
    """Ragged prefixes (items of 1 to 21 K/V tiles): the donors' second items
    are cut, their last tiles run first on the receiving blocks, and the
    donors merge the states at their ends. Every row against the oracle."""
    b = wl.build_batch("pieces", B=4, H_q=H_q, H_kv=H_kv, D=128, page_size=16, L=512,
                       context_lens=[1866, 2285, 710, 2052], seed=31 + H_q + int(causal),
                       causal=causal, placement="churn", L_new=4)
    db = DeviceBatch(b)
    out = gpu_step(db, route="attention")
    check_no_device_error()
    kp, vp = oracle_pages(b)
    assert_close(host_f64(out), oracle_out(b, kp, vp), f"tail pieces G={H_q // H_kv} causal={causal}")


def test_tail_pieces_workspace_contents_and_repeat(tail_pieces):
    """Any workspace contents (stale flags included) give the same bits."""
    import paged_kv_attention_06_gb300 as pa
    b = wl.build_batch("piecesws", B=4, H_q=8, H_kv=2, D=128, page_size=16, L=512,
                       context_lens=[1866, 2285, 710, 2052], seed=37, placement="churn", L_new=0)
    db = DeviceBatch(b)
    shape = pa.make_shape(db.query.shape, db.key_pages.shape, db.block_table.shape[1])
    need = pa.pa_prefill_workspace_bytes(shape, b.page_size)
    assert need > 0
    outs = []
    for fill in (0x00, 0xFF, 0x5A, None):
        ws = torch.full((need,), fill if fill is not None else 0, dtype=torch.uint8, device="cuda")
        if fill is None:      # the same buffer twice: the first launch's flags are stale
            pa.pa_attention(db.query, db.key_pages, db.value_pages, db.block_table,
                            db.context_lens, b.page_size, scale=b.scale, causal=b.causal,
                            max_context_len=int(b.context_lens.max()), workspace=ws)
        outs.append(pa.pa_attention(db.query, db.key_pages, db.value_pages, db.block_table,
                                    db.context_lens, b.page_size, scale=b.scale,
                                    causal=b.causal, max_context_len=int(b.context_lens.max()),
                                    workspace=ws))
        check_no_device_error()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert_close(host_f64(outs[0]), oracle_out(b, b.key_pages, b.value_pages), "pieces workspace")


def test_split_prefill_ragged_items_with_empty_rows():
    """Ragged contexts from 0 to 5000 tokens (the longest items cut over many
    blocks, the shortest with no visible key at all) in one split launch:
    sampled rows of every request against the oracle, and the rows at
    negative positions exactly zero."""
    lens = [0, 5000, 130, 2100, 7, 900, 3333, 256, 1]
    b = wl.build_batch("splitragged", B=len(lens), H_q=16, H_kv=4, D=128, page_size=16, L=256,
                       context_lens=lens, seed=25, L_new=0, placement="churn")
    out = host_f64(gpu_step(DeviceBatch(b), route="prefill_split"))
    check_no_device_error()
    assert np.all(out[0] == 0) and np.all(out[4, :, :249] == 0) and np.all(out[8, :, :255] == 0)
    rows = _sampled_rows(b, np.random.default_rng(5))
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, oracle_out(b, b.key_pages, b.value_pages, rows=rows), "split ragged")


def test_split_prefill_rejects_small_workspace():
    import paged_kv_attention_06_gb300 as pa
    b = wl.build_batch("splitsmallws", B=1, H_q=4, H_kv=2, D=128, page_size=16, L=64,
                       context_lens=[200], seed=24, L_new=0)
    db = DeviceBatch(b)
    shape = pa.make_shape(db.query.shape, db.key_pages.shape, db.block_table.shape[1])
    need = pa.pa_prefill_workspace_bytes(shape, b.page_size)
    ws = torch.empty((need - 256,), dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_prefill_split(db.query, db.key_pages, db.value_pages, db.block_table,
                            db.context_lens, b.page_size, workspace=ws)
    assert e.value.status == pa.PA_ERR_WORKSPACE
