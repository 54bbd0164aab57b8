"""Pins of the fp64 oracle against facts fixed by the pages and by mathematics.

Each test checks the oracle against something other than itself: a value the
pages print (tests/golden/*.json, each with its citation), a closed form, an
invariance the pages state, or an independent library computation (torch fp64
scaled-dot-product attention on dense tensors that were never paged).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# Worked example printed on "Reading vLLM's PagedAttention Kernel", section 4


def _p3_problem(block_table, num_pages=4):
    g = _golden("p3_worked_example.json")
    d, bs, n = g["head_dim"], g["block_size"], g["seq_len"]
    rng = np.random.default_rng(3)
    kp = rng.normal(0, 50, size=(num_pages, 1, bs, d))   # garbage everywhere
    vp = rng.normal(0, 50, size=(num_pages, 1, bs, d))
    for i in range(n):
        phys, slot = block_table[i // bs], i % bs
        kp[phys, 0, slot] = g["K"][i]
        vp[phys, 0, slot] = g["V"][i]
    q = np.asarray(g["q"], dtype=np.float64).reshape(1, 1, 1, d)
    bt = np.asarray([block_table], dtype=np.int32)
    cl = np.asarray([n], dtype=np.int32)
    return g, q, kp, vp, bt, cl


def test_p3_worked_example_printed_output():
    table = _golden("p3_worked_example.json")["block_table"]
    g, q, kp, vp, bt, cl = _p3_problem(table)
    out = oracle.attention(q, kp, vp, bt, cl, g["block_size"], scale=None, causal=True)
    expected = np.asarray(g["expected_output"])
    # The page prints 6 decimals: the exact value lies within 5e-7 of it.
    assert np.max(np.abs(out[0, 0, 0] - expected)) <= 5e-7 + 1e-12


def test_p3_worked_example_explicit_scale_matches_default():
    g, q, kp, vp, bt, cl = _p3_problem([3, 1])
    a = oracle.attention(q, kp, vp, bt, cl, 4, scale=None)
    b = oracle.attention(q, kp, vp, bt, cl, 4, scale=0.5)      # 1/sqrt(4)
    assert np.array_equal(a, b)
    c = oracle.attention(q, kp, vp, bt, cl, 4, scale=1.0)
    assert np.max(np.abs(c - a)) > 1e-3                          # scale matters


def test_p3_worked_example_relabelled_blocks():
    # The same six tokens placed at blocks [0, 2] of a 5-block pool: physical
    # placement is arbitrary, the block table restores the order.
    g, q, kp, vp, bt, cl = _p3_problem([0, 2], num_pages=5)
    out = oracle.attention(q, kp, vp, bt, cl, 4)
    assert np.max(np.abs(out[0, 0, 0] - np.asarray(g["expected_output"]))) <= 5e-7 + 1e-12


# ----------------------------------------------------------------------------
# Mapping table printed on "Week 3 Day 4", "Why block_table Matters"


def test_p1_translation_table():
    g = _golden("p1_block_table_mapping.json")
    for pos in range(g["context_len"]):
        page, slot = oracle.translate(g["page_ids"], g["page_size"], 16, pos)
        assert page == g["expected_pages_by_position"][pos]
        assert slot == g["expected_slots_by_position"][pos]


def test_p1_translation_rejects_page_outside_pool():
    with pytest.raises(oracle.OracleError):
        oracle.translate([12, 5, 3], 4, 12, 0)      # page 12 in a 12-page pool


def test_p1_mapping_recovered_through_attention():
    """K = 0 makes every visible key equally weighted, so causal row i returns
    the mean of V over positions 0..i; V stores (page, slot) of its own
    storage location, so consecutive rows give back each position's page and
    slot. This pins translation and the causal query offset together."""
    g = _golden("p1_block_table_mapping.json")
    ps, n, P, D = g["page_size"], g["context_len"], 16, 2
    kp = np.zeros((P, 1, ps, D))
    vp = np.full((P, 1, ps, D), 1e6)          # unreferenced slots: far-off values
    for pid in g["page_ids"]:
        for s in range(ps):
            vp[pid, 0, s] = (pid, s)
    q = np.ones((1, 1, n, D))
    bt = np.asarray([g["page_ids"]], dtype=np.int32)
    cl = np.asarray([n], dtype=np.int32)
    out = oracle.attention(q, kp, vp, bt, cl, ps, causal=True)[0, 0]   # [n, D]
    sums = out * np.arange(1, n + 1)[:, None]
    codes = np.diff(np.vstack([np.zeros((1, D)), sums]), axis=0)
    assert np.allclose(codes[:, 0], g["expected_pages_by_position"], atol=1e-9)
    assert np.allclose(codes[:, 1], g["expected_slots_by_position"], atol=1e-9)


# ----------------------------------------------------------------------------
# Append walkthrough of "Tutorial 13", section 4


@pytest.mark.parametrize("which", ["printed_walkthrough", "append_code"])
def test_p2_append_walkthrough(which):
    g = _golden("p2_append_walkthrough.json")
    exp = g[which]
    ps = g["page_size"]
    pool = wl.PageFreeList(ps)
    cache = wl.RequestPages(pool, policy=exp["policy"])
    P, D = 3, 8
    key_pages = np.zeros((P, 1, ps, D), dtype=np.uint16)
    value_pages = np.zeros((P, 1, ps, D), dtype=np.uint16)
    token = 0
    for c, n_tok in enumerate(g["chunks"]):
        slots = cache.append(n_tok)
        assert cache.pages == exp["page_ids_after_each_chunk"][c]
        assert cache.fill == exp["page_lens_after_each_chunk"][c]
        assert cache.length == exp["offset_after_each_chunk"][c]
        # token t's K row is the bf16 bits of (t + 1) in every lane, V of -(t+1)
        ids = np.arange(token, token + n_tok)
        key = np.repeat(wl.bf16_bits((ids + 1).astype(np.float32))[:, None], D, 1)
        val = np.repeat(wl.bf16_bits(-(ids + 1).astype(np.float32))[:, None], D, 1)
        bad = oracle.append_kv(key.reshape(1, 1, n_tok, D).copy(),
                               val.reshape(1, 1, n_tok, D).copy(),
                               key_pages, value_pages,
                               np.asarray([slots], dtype=np.int32), ps)
        assert bad == 0
        token += n_tok
    for pid, content in exp["page_contents"].items():
        for s, t in enumerate(content):
            row_k = wl.bf16_to_f32(key_pages[int(pid), 0, s])
            row_v = wl.bf16_to_f32(value_pages[int(pid), 0, s])
            if t is None:
                assert np.all(row_k == 0) and np.all(row_v == 0)
            else:
                assert np.all(row_k == t + 1) and np.all(row_v == -(t + 1))


def test_append_bit_exact_and_skips():
    rng = np.random.default_rng(5)
    P, H, ps, D, B, Ln = 6, 2, 4, 16, 2, 3
    kp = rng.integers(0, 65536, size=(P, H, ps, D), dtype=np.uint16)
    vp = rng.integers(0, 65536, size=(P, H, ps, D), dtype=np.uint16)
    k0, v0 = kp.copy(), vp.copy()
    key = rng.integers(0, 65536, size=(B, H, Ln, D), dtype=np.uint16)   # any bits, NaNs too
    val = rng.integers(0, 65536, size=(B, H, Ln, D), dtype=np.uint16)
    slots = np.asarray([[5, -1, 23], [0, 9, P * ps + 2]], dtype=np.int32)
    bad = oracle.append_kv(key, val, kp, vp, slots, ps)
    assert bad == 1                          # the slot beyond the pool
    touched = set()
    for b in range(B):
        for i in range(Ln):
            s = int(slots[b, i])
            if 0 <= s < P * ps:
                touched.add((s // ps, s % ps))
                assert np.array_equal(kp[s // ps, :, s % ps], key[b, :, i])
                assert np.array_equal(vp[s // ps, :, s % ps], val[b, :, i])
    for p in range(P):
        for s in range(ps):
            if (p, s) not in touched:
                assert np.array_equal(kp[p, :, s], k0[p, :, s])
                assert np.array_equal(vp[p, :, s], v0[p, :, s])


# ----------------------------------------------------------------------------
# Closed forms


def test_uniform_weights_give_mean_position_causal_offset():
    """K = 0: every visible key has the same score, so the output is the mean
    of the visible V. With V_j = j (position), causal row i of a chunk of L
    rows ending at position n-1 sits at p = n - L + i and returns p / 2."""
    ps, n, L, D = 4, 13, 5, 4
    P = 8
    bt = np.asarray([[6, 1, 4, 0]], dtype=np.int32)
    kp = np.zeros((P, 1, ps, D))
    vp = np.full((P, 1, ps, D), np.nan)         # never-visible slots are NaN
    for j in range(n):
        vp[bt[0, j // ps], 0, j % ps] = j
    q = np.ones((1, 1, L, D))
    out = oracle.attention(q, kp, vp, bt, np.asarray([n], np.int32), ps, causal=True)
    for i in range(L):
        p = n - L + i
        assert np.allclose(out[0, 0, i], p / 2.0, atol=1e-12)
    nc = oracle.attention(q, kp, vp, bt, np.asarray([n], np.int32), ps, causal=False)
    assert np.allclose(nc[0, 0], (n - 1) / 2.0, atol=1e-12)


def test_gqa_head_mapping_contiguous_groups():
    """V constant c_g per KV head: query head h_q must return c_{h_q // G}."""
    H_q, H_kv, ps, D, n = 12, 4, 2, 8, 5
    G = H_q // H_kv
    rng = np.random.default_rng(9)
    P = 4
    bt = np.asarray([[3, 0, 2]], dtype=np.int32)
    kp = rng.normal(size=(P, H_kv, ps, D))
    vp = np.zeros((P, H_kv, ps, D))
    for g in range(H_kv):
        vp[:, g] = 10.0 * g + 1.0
    q = rng.normal(size=(1, H_q, 1, D))
    out = oracle.attention(q, kp, vp, bt, np.asarray([n], np.int32), ps)
    for hq in range(H_q):
        assert np.allclose(out[0, hq, 0], 10.0 * (hq // G) + 1.0, atol=1e-12)


def test_single_visible_key_returns_its_value():
    rng = np.random.default_rng(2)
    D, ps = 16, 4
    kp = rng.normal(size=(3, 1, ps, D)) * 40
    vp = rng.normal(size=(3, 1, ps, D))
    q = rng.normal(size=(1, 1, 1, D))
    bt = np.asarray([[2]], dtype=np.int32)
    out = oracle.attention(q, kp, vp, bt, np.asarray([1], np.int32), ps)
    assert np.array_equal(out[0, 0, 0], vp[2, 0, 0])


def test_empty_context_and_rows_without_keys_are_zero():
    D, ps = 8, 4
    kp = np.ones((2, 1, ps, D))
    vp = np.ones((2, 1, ps, D))
    q = np.ones((2, 1, 3, D))
    bt = np.asarray([[0], [1]], dtype=np.int32)
    cl = np.asarray([0, 2], dtype=np.int32)
    out = oracle.attention(q, kp, vp, bt, cl, ps, causal=True)
    assert np.all(out[0] == 0)                 # n = 0
    assert np.all(out[1, 0, 0] == 0)           # row 0 at position -1
    assert np.allclose(out[1, 0, 1:], 1.0)


def test_oracle_rejects_bad_page_and_length():
    D, ps = 8, 4
    kp = np.ones((2, 1, ps, D))
    q = np.ones((1, 1, 1, D))
    with pytest.raises(oracle.OracleError):
        oracle.attention(q, kp, kp, np.asarray([[5]], np.int32), np.asarray([3], np.int32), ps)
    with pytest.raises(oracle.OracleError):
        oracle.attention(q, kp, kp, np.asarray([[0]], np.int32), np.asarray([5], np.int32), ps)


# ----------------------------------------------------------------------------
# Invariances stated on Week 3 Day 4, "What Must Hold"


def _random_problem(seed, B=3, H_q=6, H_kv=2, L=1, D=16, ps=4, lens=(9, 4, 12),
                    P=16, bf16=False):
    rng = np.random.default_rng(seed)
    maxp = max(math.ceil(n / ps) for n in lens)
    perm = rng.permutation(P)
    bt = np.full((B, maxp), -1, dtype=np.int32)
    k = 0
    for b, n in enumerate(lens):
        c = math.ceil(n / ps)
        bt[b, :c] = perm[k:k + c]
        k += c
    shape = (P, H_kv, ps, D)
    if bf16:
        kp, vp = wl.normal_bf16(rng, shape), wl.normal_bf16(rng, shape)
        q = wl.normal_bf16(rng, (B, H_q, L, D))
    else:
        kp, vp = rng.normal(size=shape), rng.normal(size=shape)
        q = rng.normal(size=(B, H_q, L, D))
    return q, kp, vp, bt, np.asarray(lens, dtype=np.int32)


def _relabel(kp, vp, bt, perm):
    """Move page p to id perm[p] and rewrite the table accordingly."""
    kp2, vp2 = np.empty_like(kp), np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    bt2 = bt.copy()
    m = bt >= 0
    bt2[m] = perm[bt[m]]
    return kp2, vp2, bt2


@pytest.mark.parametrize("causal,L", [(True, 1), (True, 3), (False, 2)])
def test_physical_relabelling_is_bit_identical(causal, L):
    q, kp, vp, bt, cl = _random_problem(11, L=L, bf16=True)
    ref = oracle.attention(q, kp, vp, bt, cl, 4, causal=causal)
    perm = np.random.default_rng(4).permutation(kp.shape[0])
    kp2, vp2, bt2 = _relabel(kp, vp, bt, perm)
    out = oracle.attention(q, kp2, vp2, bt2, cl, 4, causal=causal)
    assert np.array_equal(ref.view(np.uint64), out.view(np.uint64))


def test_stale_data_never_read():
    q, kp, vp, bt, cl = _random_problem(12, L=2, bf16=True)
    ref = oracle.attention(q, kp, vp, bt, cl, 4)
    used = np.zeros(kp.shape[:1] + kp.shape[2:3], dtype=bool)
    for b in range(bt.shape[0]):
        for j in range(cl[b]):
            used[bt[b, j // 4], j % 4] = True
    pages, slots = np.nonzero(~used)
    for pattern in (0x7FC0, 0x7F80, 0xFF80):          # NaN, +Inf, -Inf bits
        kp2, vp2 = kp.copy(), vp.copy()
        kp2[pages, :, slots, :] = pattern
        vp2[pages, :, slots, :] = pattern
        out = oracle.attention(q, kp2, vp2, bt, cl, 4)
        assert np.array_equal(ref.view(np.uint64), out.view(np.uint64))


def test_decode_invariant_to_complete_page_order_but_causal_prefix_is_not():
    ps, D = 4, 8
    rng = np.random.default_rng(21)
    n = 12                                       # three complete pages
    P = 5
    kp, vp = rng.normal(size=(P, 1, ps, D)), rng.normal(size=(P, 1, ps, D))
    bt = np.asarray([[4, 0, 2]], dtype=np.int32)
    bt_re = np.asarray([[2, 4, 0]], dtype=np.int32)   # same pages, other order
    cl = np.asarray([n], dtype=np.int32)
    q1 = rng.normal(size=(1, 1, 1, D))
    a = oracle.attention(q1, kp, vp, bt, cl, ps)
    b = oracle.attention(q1, kp, vp, bt_re, cl, ps)
    assert np.max(np.abs(a - b)) < 1e-12
    q5 = rng.normal(size=(1, 1, 5, D))
    a = oracle.attention(q5, kp, vp, bt, cl, ps, causal=True)
    b = oracle.attention(q5, kp, vp, bt_re, cl, ps, causal=True)
    assert np.max(np.abs(a[0, 0, :-1] - b[0, 0, :-1])) > 1e-3   # prefix rows change
    assert np.max(np.abs(a[0, 0, -1] - b[0, 0, -1])) < 1e-12    # last row sees all


# ----------------------------------------------------------------------------
# Independent library computation on dense tensors that were never paged


def _dense_to_pages(rng, Kd, Vd, lens, ps, P):
    """Scatter dense [B, H_kv, n_max, D] K/V into a garbage-filled pool."""
    B, H_kv, _, D = Kd.shape
    kp = rng.normal(0, 30, size=(P, H_kv, ps, D))
    vp = rng.normal(0, 30, size=(P, H_kv, ps, D))
    perm = list(rng.permutation(P))
    maxp = max(1, max(math.ceil(n / ps) for n in lens))
    bt = np.full((B, maxp), -1, dtype=np.int32)
    for b, n in enumerate(lens):
        for lp in range(math.ceil(n / ps)):
            bt[b, lp] = perm.pop()
        for j in range(n):
            kp[bt[b, j // ps], :, j % ps] = Kd[b, :, j]
            vp[bt[b, j // ps], :, j % ps] = Vd[b, :, j]
    return kp, vp, bt


@pytest.mark.parametrize("ps", [1, 2, 4, 16])
@pytest.mark.parametrize("H_q,H_kv", [(4, 4), (6, 2), (7, 1)])
@pytest.mark.parametrize("L,causal", [(1, True), (4, True), (3, False)])
def test_against_torch_sdpa_fp64(ps, H_q, H_kv, L, causal):
    rng = np.random.default_rng(1000 + 7 * ps + H_q + 3 * L)
    B, D = 3, 16
    lens = [int(x) for x in rng.integers(L, 23, size=B)]
    nmax = max(lens)
    Kd = rng.normal(size=(B, H_kv, nmax, D))
    Vd = rng.normal(size=(B, H_kv, nmax, D))
    q = rng.normal(size=(B, H_q, L, D))
    P = sum(math.ceil(n / ps) for n in lens) + 3
    kp, vp, bt = _dense_to_pages(rng, Kd, Vd, lens, ps, P)
    scale = 0.37
    out = oracle.attention(q, kp, vp, bt, np.asarray(lens, np.int32), ps,
                           scale=scale, causal=causal)
    G = H_q // H_kv
    for b, n in enumerate(lens):
        k = torch.from_numpy(Kd[b, :, :n]).repeat_interleave(G, dim=0)   # [H_q, n, D]
        v = torch.from_numpy(Vd[b, :, :n]).repeat_interleave(G, dim=0)
        qq = torch.from_numpy(q[b])                                       # [H_q, L, D]
        if causal:
            mask = torch.arange(n)[None, :] <= (n - L + torch.arange(L))[:, None]
        else:
            mask = torch.ones(L, n, dtype=torch.bool)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qq, k, v, attn_mask=mask, scale=scale).numpy()
        assert np.max(np.abs(out[b] - ref)) < 1e-12


def test_rows_subset_matches_full():
    q, kp, vp, bt, cl = _random_problem(31, L=3, bf16=True)
    full = oracle.attention(q, kp, vp, bt, cl, 4)
    rows = np.asarray([[2, 5, 1], [0, 0, 0], [1, 3, 2]], dtype=np.int32)
    sub = oracle.attention(q, kp, vp, bt, cl, 4, rows=rows, n_threads=2)
    for r, (b, h, i) in enumerate(rows):
        assert np.array_equal(sub[r], full[b, h, i])


# ----------------------------------------------------------------------------
# Gather (the dense baseline's first step)


def test_p1_gather_follows_printed_mapping():
    """Every page row carries its own (page, slot) marker; the gathered dense
    rows must come out in the order of the printed position -> page table."""
    g = _golden("p1_block_table_mapping.json")
    ps, n = g["page_size"], g["context_len"]
    P, H_kv, D = 16, 2, 8
    pages = np.zeros((P, H_kv, ps, D), dtype=np.uint16)
    for p in range(P):
        for h in range(H_kv):
            for s in range(ps):
                pages[p, h, s, :] = 1000 * h + 16 * p + s
    bt = np.array([g["page_ids"]], dtype=np.int32)
    dense = oracle.gather(pages, bt, np.array([n], dtype=np.int32), ps, n + 3, fill=7)
    for h in range(H_kv):
        want = [1000 * h + 16 * p + s for p, s in zip(g["expected_pages_by_position"],
                                                       g["expected_slots_by_position"])]
        assert dense[0, h, :n, 0].tolist() == want
        assert np.all(dense[0, h, n:] == 7)          # rows past the context untouched


def test_gather_invariant_to_physical_relabelling():
    b = wl.make_workload("tiny_decode")
    d0 = oracle.gather(b.key_pages, b.block_table, b.context_lens, b.page_size, 16)
    rng = np.random.default_rng(3)
    perm = rng.permutation(b.num_pages)            # page p moves to perm[p]
    pages = np.empty_like(b.key_pages)
    pages[perm] = b.key_pages
    bt = np.where(b.block_table >= 0, perm[np.clip(b.block_table, 0, None)], -1).astype(np.int32)
    d1 = oracle.gather(pages, bt, b.context_lens, b.page_size, 16)
    assert np.array_equal(d0, d1)


def test_dense_attention_over_gathered_rows_equals_paged_attention():
    """The gathered buffer is a pool with one page of dense_len tokens per
    request; attention over it with the identity table is the same fp64
    computation over the same keys in the same order: bit-identical."""
    b = wl.make_workload("tiny_decode")
    N = 12
    kd = oracle.gather(b.key_pages, b.block_table, b.context_lens, b.page_size, N)
    vd = oracle.gather(b.value_pages, b.block_table, b.context_lens, b.page_size, N)
    ident = np.arange(b.B, dtype=np.int32).reshape(b.B, 1)
    dense = oracle.attention(b.query, kd.reshape(b.B, b.H_kv, N, b.D), vd.reshape(b.B, b.H_kv, N, b.D),
                             ident, b.context_lens, N, scale=b.scale, causal=b.causal)
    paged = oracle.attention(b.query, b.key_pages, b.value_pages, b.block_table, b.context_lens,
                             b.page_size, scale=b.scale, causal=b.causal)
    assert np.array_equal(dense, paged)


def test_gather_rejects_bad_page_and_long_context():
    b = wl.make_workload("tiny_decode")
    bt = b.block_table.copy()
    bt[0, 0] = b.num_pages
    with pytest.raises(oracle.OracleError):
        oracle.gather(b.key_pages, bt, b.context_lens, b.page_size, 16)
    with pytest.raises(oracle.OracleError):
        oracle.gather(b.key_pages, b.block_table, b.context_lens, b.page_size, 8)  # 10 > 8


# ----------------------------------------------------------------------------
# FP8 (e4m3) pages with per-tensor scales (Reading vLLM's PagedAttention
# Kernel, 3.2: the write path takes kv_cache_dtype, k_scale and v_scale).


def test_e4m3_values_of_the_format():
    """Codes whose values the format fixes: bias 7, 3 mantissa bits,
    subnormals m * 2^-9, S.1111.111 = NaN, largest finite 448."""
    table = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x30: 0.5, 0x38: 1.0, 0x39: 1.125, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0,
             0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    codes = np.array(list(table), dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    assert np.array_equal(got, np.array(list(table.values())))
    assert np.signbit(got[list(table).index(0x80)])
    assert np.isnan(oracle.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


def test_e4m3_encode_matches_torch_rounding():
    """Nearest value, ties to even: the same codes as torch's float8_e4m3fn
    conversion wherever that conversion stays finite (|x| < 464)."""
    rng = np.random.default_rng(17)
    finite = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (finite[1:] + finite[:-1]) / 2                   # every tie point
    x = np.concatenate([
        rng.normal(0, 1, 4000), rng.normal(0, 60, 4000), rng.uniform(-460, 460, 4000),
        rng.uniform(-0.02, 0.02, 4000), mids, -mids, finite, -finite,
        np.nextafter(mids, 0), np.nextafter(mids, 1000)]).astype(np.float32)
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)


def test_e4m3_encode_saturates_round_trips_and_is_monotone():
    x = np.float32([448.0, 464.0, 500.0, 1e9, np.inf, -464.0, -1e9, -np.inf])
    assert oracle.e4m3_encode(x).tolist() == [0x7E] * 5 + [0xFE] * 3
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    vals = oracle.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3_encode(vals), codes)         # every finite code
    sweep = np.linspace(-470, 470, 200001, dtype=np.float32)
    dec = oracle.e4m3_decode(oracle.e4m3_encode(sweep))
    assert np.all(np.diff(dec) >= 0)
    # within half a step of the format at every magnitude below 448
    inside = np.abs(sweep) <= 448
    a = np.abs(sweep[inside]).astype(np.float64)
    step = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3))
    assert np.all(np.abs(dec[inside] - sweep[inside]) <= step / 2 + 1e-12)


def test_append_fp8_stores_codes_of_x_over_scale():
    """Values that are scale times an e4m3 value come back exactly; slots
    are the same as the bf16 append's."""
    rng = np.random.default_rng(23)
    B, H_kv, L_new, D, ps, P = 2, 2, 5, 16, 4, 8
    k_scale, v_scale = 0.0625, 0.5            # powers of two: x / scale exact in fp32
    kc = rng.integers(0, 0x7F, size=(B, H_kv, L_new, D)).astype(np.uint8)
    vc = (rng.integers(0, 0x7F, size=(B, H_kv, L_new, D)) | 0x80 * rng.integers(0, 2, size=(B, H_kv, L_new, D))).astype(np.uint8)
    vc[vc == 0xFF] = 0xFE
    kx = (oracle.e4m3_decode(kc) * k_scale).astype(np.float32)
    vx = (oracle.e4m3_decode(vc) * v_scale).astype(np.float32)
    to_bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(to_bits(kx).astype(np.uint32) << 16, kx.view(np.uint32))   # bf16 exact
    slots = rng.permutation(P * ps)[:B * L_new].reshape(B, L_new).astype(np.int32)
    slots[1, 3] = -1
    kp = np.zeros((P, H_kv, ps, D), np.uint8)
    vp = np.zeros_like(kp)
    assert oracle.append_kv_fp8(to_bits(kx), to_bits(vx), kp, vp, slots, ps, k_scale, v_scale) == 0
    for b in range(B):
        for i in range(L_new):
            s = slots[b, i]
            if s < 0:
                continue
            assert np.array_equal(kp[s // ps, :, s % ps], kc[b, :, i])
            assert np.array_equal(vp[s // ps, :, s % ps], vc[b, :, i])
    assert kp.sum() == sum(int(kc[b, :, i].astype(np.int64).sum()) for b in range(B)
                           for i in range(L_new) if slots[b, i] >= 0)


def test_attention_fp8_equals_bf16_attention_on_shared_values():
    """With unit scales and K/V values that are both bf16 and e4m3 values,
    attention over the FP8 pages equals attention over the bf16 pages."""
    rng = np.random.default_rng(29)
    b = wl.build_batch("fp8pin", B=2, H_q=4, H_kv=2, D=16, page_size=4, L=3,
                       context_lens=[9, 6], seed=31, L_new=0)
    codes_k = rng.integers(0, 0x7F, size=b.key_pages.shape).astype(np.uint8) | \
        (0x80 * rng.integers(0, 2, size=b.key_pages.shape)).astype(np.uint8)
    codes_v = rng.integers(0, 0x7F, size=b.value_pages.shape).astype(np.uint8)
    codes_k[codes_k == 0xFF] = 0x7E
    fk = oracle.e4m3_decode(codes_k).astype(np.float32)
    fv = oracle.e4m3_decode(codes_v).astype(np.float32)
    bits = lambda a: (a.view(np.uint32) >> 16).astype(np.uint16)   # e4m3 values are bf16 values
    ref = oracle.attention(b.query, bits(fk), bits(fv), b.block_table, b.context_lens,
                           b.page_size, scale=b.scale)
    got = oracle.attention_fp8(b.query, codes_k, codes_v, 1.0, 1.0, b.block_table,
                               b.context_lens, b.page_size, scale=b.scale)
    assert np.array_equal(got, ref)
