"""Host-side fixtures: the page allocator and the seeded workloads.

The allocator follows Tutorial 13: Paged Attention and Memory Management,
sections 3-4, and the invariants of Week 3 Day 4: Direct Paged Attention,
"What Must Hold, and What Breaks If It Doesn't" (items 3-5).
"""
import math

import numpy as np
import pytest

import workloads as wl


def test_lifo_reuse_and_growth():
    pool = wl.PageFreeList(4)
    a, b, c = pool.take(), pool.take(), pool.take()
    assert (a, b, c) == (0, 1, 2)
    pool.give_back(b)
    pool.give_back(a)
    assert pool.take() == a          # last freed, first reused
    assert pool.take() == b
    assert pool.take() == 3          # free list empty: grow
    assert pool.fresh == 4


def test_double_free_raises():
    pool = wl.PageFreeList(4)
    p = pool.take()
    pool.give_back(p)
    with pytest.raises(wl.DoubleFree):
        pool.give_back(p)


def test_release_returns_every_page_once():
    pool = wl.PageFreeList(4)
    caches = [wl.RequestPages(pool) for _ in range(3)]
    for c, n in zip(caches, (5, 9, 1)):
        c.append(n)
    owned = [list(c.pages) for c in caches]
    assert len({p for o in owned for p in o}) == sum(len(o) for o in owned)   # no aliasing
    caches[1].release()
    assert sorted(pool.returned) == sorted(owned[1])
    with pytest.raises(wl.DoubleFree):
        for p in owned[1]:
            pool.give_back(p)


def test_decode_allocates_only_on_tail_overflow():
    pool = wl.PageFreeList(4)
    c = wl.RequestPages(pool)
    c.append(3)
    for step in range(9):
        before = len(c.pages)
        full = c.fill[-1] == 4
        c.append(1)
        assert len(c.pages) == before + (1 if full else 0)
    assert c.length == 12 and c.fill == [4, 4, 4]


def test_slots_follow_page_and_offset():
    pool = wl.PageFreeList(16)
    for _ in range(5):
        pool.take()
    c = wl.RequestPages(pool)
    slots = c.append(20)
    assert slots[:16] == [5 * 16 + t for t in range(16)]
    assert slots[16:] == [6 * 16 + t for t in range(4)]


def test_bf16_round_trip_and_rounding():
    x = np.asarray([1.0, -2.5, 1.00390625, 1.005859375, 3.0e38, 0.0], dtype=np.float32)
    bits = wl.bf16_bits(x)
    back = wl.bf16_to_f32(bits)
    assert back[0] == 1.0 and back[1] == -2.5
    assert back[2] == 1.0                   # tie 1 + 2^-8 rounds to even (1.0)
    assert back[3] == 1.0078125             # above the tie rounds up
    assert np.isnan(wl.bf16_to_f32(wl.bf16_bits(np.asarray([np.nan], np.float32))))[0]


@pytest.mark.parametrize("name", ["tiny_decode", "prefill_chunk512"])
def test_workload_structure(name):
    b = wl.make_workload(name)
    assert b.query.shape == (b.B, b.H_q, b.L, b.D)
    assert b.key_pages.shape == (b.num_pages, b.H_kv, b.page_size, b.D)
    for r in range(b.B):
        n = int(b.context_lens[r])
        need = math.ceil(n / b.page_size)
        assert np.all(b.block_table[r, :need] >= 0)
        assert np.all(b.block_table[r, :need] < b.num_pages)
        assert np.all(b.block_table[r, need:] == -1)
        # the new tokens land on the last L_new positions of the context
        for i in range(b.L_new):
            pos = n - b.L_new + i
            s = int(b.slot_mapping[r, i])
            assert s // b.page_size == b.block_table[r, pos // b.page_size]
            assert s % b.page_size == pos % b.page_size
    used = b.block_table[b.block_table >= 0]
    assert len(np.unique(used)) == used.size       # no aliasing between requests


def test_tiny_decode_uses_the_printed_table():
    b = wl.make_workload("tiny_decode")
    assert list(b.block_table[0]) == [12, 5, 3]
    assert list(b.context_lens) == [10, 7]
    assert b.num_pages == 16 and b.D == 64 and b.page_size == 4


def test_churn_placement_reuses_freed_ids():
    rng = np.random.default_rng(0)
    lens = [300, 1000, 77]
    tables, ghosts = wl._page_tables_churn(rng, lens, 128, 20, 0.2, 128)
    flat = [p for t in tables for p in t]
    assert len(set(flat)) == len(flat) == 12
    assert set(ghosts) & set(flat)                  # freed ids were handed out again
    assert flat != sorted(flat)                     # shuffled placement


def test_seeded_inputs_are_reproducible():
    a = wl.make_workload("tiny_decode")
    b = wl.make_workload("tiny_decode")
    assert np.array_equal(a.key_pages, b.key_pages) and np.array_equal(a.query, b.query)
