"""The C++ page allocator and per-step metadata builder (pa_kv_cache, host
code): against the pinned Python allocator fixture (same page ids, slots and
tables on random histories), the printed append walkthrough of Tutorial 13
(tail-fill code), all-or-nothing steps, and release exactly once. No GPU."""
import numpy as np
import pytest

import workloads as wl


def _pa():
    import paged_kv_attention_06_gb300 as pa
    return pa


def test_append_walkthrough_tail_fill():
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "p2_append_walkthrough.json")))
    exp = g["append_code"]
    ps = g["page_size"]
    c = _pa().KVCache(8, ps)
    c.add(7)
    token = 0
    contents = {}
    for k, n_tok in enumerate(g["chunks"]):
        bt, cl, sm = c.plan([7], [n_tok], max_pages=4, l_new=4)
        pages = [int(p) for p in bt[0] if p >= 0]
        assert pages == exp["page_ids_after_each_chunk"][k]
        assert int(cl[0]) == exp["offset_after_each_chunk"][k]
        lens = [min(ps, int(cl[0]) - ps * i) for i in range(len(pages))]
        assert lens == exp["page_lens_after_each_chunk"][k]
        for t, slot in enumerate(sm[0, :n_tok]):
            contents[(int(slot) // ps, int(slot) % ps)] = token + t
        assert np.all(sm[0, n_tok:] == -1)
        token += n_tok
    for pid, row in exp["page_contents"].items():
        for s, t in enumerate(row):
            assert contents.get((int(pid), s)) == t


def test_matches_python_fixture_on_random_histories():
    """Random admissions, chunked appends and releases: the C++ cache and the
    fixture (PageFreeList last-returned-first reuse + RequestPages tail fill) give the same
    page ids, slots, tables and context lengths at every step."""
    pa = _pa()
    rng = np.random.default_rng(5)
    for trial in range(20):
        ps = int(rng.choice([1, 4, 16]))
        num_pages = 4096
        c = pa.KVCache(num_pages, ps)
        pool = wl.PageFreeList(ps)
        live = {}
        next_id = 0
        for step in range(60):
            if len(live) < 4 and rng.random() < 0.5:
                c.add(next_id)
                live[next_id] = wl.RequestPages(pool)
                next_id += 1
            if live and rng.random() < 0.15:
                sid = int(rng.choice(list(live)))
                c.release(sid)
                live.pop(sid).release()
            if not live:
                continue
            ids = list(live)
            toks = [int(rng.integers(0, 9)) for _ in ids]
            bt, cl, sm = c.plan(ids, toks, max_pages=256, l_new=8)
            for i, sid in enumerate(ids):
                slots = live[sid].append(toks[i])
                assert sm[i, :toks[i]].tolist() == slots
                assert [int(p) for p in bt[i] if p >= 0] == live[sid].pages
                assert int(cl[i]) == live[sid].length == c.context_len(sid)
        assert c.free_pages == num_pages - len(pool.in_use)


def test_step_is_all_or_nothing():
    pa = _pa()
    c = pa.KVCache(4, 4)
    c.add(1)
    c.add(2)
    c.plan([1], [5], max_pages=4, l_new=8)           # request 1: 2 pages
    free = c.free_pages
    with pytest.raises(pa.PagedAttentionError) as e:  # needs 3 + 1 pages, 2 left
        c.plan([2, 1], [9, 3], max_pages=4, l_new=9)
    assert e.value.status == pa.PA_ERR_NO_PAGES
    assert c.free_pages == free and c.context_len(1) == 5 and c.context_len(2) == 0
    # the same history without the failed step gives the same next allocation
    d = pa.KVCache(4, 4)
    d.add(1)
    d.add(2)
    d.plan([1], [5], max_pages=4, l_new=8)
    assert np.array_equal(c.plan([2], [4], 4, 4)[0], d.plan([2], [4], 4, 4)[0])
    with pytest.raises(pa.PagedAttentionError):       # block-table row too short
        c.plan([1], [8], max_pages=2, l_new=8)
    assert c.context_len(1) == 5


def test_release_exactly_once_and_bad_arguments():
    pa = _pa()
    c = pa.KVCache(8, 2)
    c.add(3)
    bt, _, _ = c.plan([3], [5], max_pages=8, l_new=5)
    assert c.free_pages == 5
    c.release(3)
    assert c.free_pages == 8
    with pytest.raises(pa.PagedAttentionError):
        c.release(3)                                  # second release
    with pytest.raises(pa.PagedAttentionError):
        c.plan([3], [1], 8, 1)                        # unknown request
    c.add(4)
    with pytest.raises(pa.PagedAttentionError):
        c.add(4)                                      # exists
    with pytest.raises(pa.PagedAttentionError):
        c.plan([4, 4], [1, 1], 8, 1)                  # listed twice
    with pytest.raises(pa.PagedAttentionError):
        c.plan([4], [2], 8, 1)                        # more tokens than l_new
    # freed pages come back last-freed first: request 3 held pages 0, 1, 2
    bt, _, _ = c.plan([4], [2], 8, 2)
    assert int(bt[0, 0]) == int(np.asarray(bt)[0, 0]) == 2


def test_snapshot_restore_rolls_back_a_step():
    """Tutorial 13 section 7: a step that failed after its pages were planned
    (its K/V write or launch failed) is undone by restoring the snapshot taken
    before it; the cache then behaves exactly like one that never ran it."""
    pa = _pa()
    c, twin = pa.KVCache(16, 4), pa.KVCache(16, 4)
    for x in (c, twin):
        x.add(1)
        x.add(2)
        x.plan([1, 2], [6, 3], max_pages=8, l_new=6)
        x.release(2)                                  # pages on the free list
    snap = c.snapshot()
    c.plan([1], [7], max_pages=8, l_new=7)            # the step that "failed"
    c.release(1)
    c.add(9)
    c.plan([9], [5], max_pages=8, l_new=5)
    c.restore(snap)
    assert c.context_len(1) == twin.context_len(1) == 6
    assert c.context_len(9) == -1 and c.free_pages == twin.free_pages
    a, b = c.plan([1], [7], 8, 7), twin.plan([1], [7], 8, 7)
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
    c.restore(snap)                                   # a snapshot can be restored again
    assert c.context_len(1) == 6
    other = pa.KVCache(16, 4)
    with pytest.raises(pa.PagedAttentionError):       # snapshot of another cache
        other.restore(snap)
    snap.close()


def test_native_step_checks_before_any_device_work():
    """pa_kv_cache_step: the packed table size, and the argument checks and
    plan failures that return before anything reaches the GPU (the cache is
    left unchanged)."""
    import ctypes
    pa = _pa()
    lib = pa.binding._lib
    assert lib.pa_kv_cache_step_table_bytes(3, 10, 4) == 3 * (10 + 1 + 4) * 4
    assert lib.pa_kv_cache_step_table_bytes(0, 10, 4) == 0
    assert lib.pa_kv_cache_step_table_bytes(3, 10, 0) == 0
    c = pa.KVCache(8, 4)
    c.add(1)
    ids = np.array([1], dtype=np.int64)
    toks = np.array([3], dtype=np.int32)
    host = (ctypes.c_int32 * 64)()
    need = lib.pa_kv_cache_step_table_bytes(1, 4, 3)

    def step(ids_, toks_, host_ptr, nbytes, max_pages=4):
        return lib.pa_kv_cache_step(c._h, len(ids_), ids_.ctypes.data, toks_.ctypes.data, 3,
                                    max_pages, host_ptr, ctypes.addressof(host), nbytes,
                                    None, None, None, None, None, 4, 2, 128, 0.1, None, None, 0,
                                    None)

    assert step(ids, toks, None, need) == pa.PA_ERR_INVALID_ARG           # no host tables
    assert step(ids, toks, ctypes.addressof(host), need - 4) == pa.PA_ERR_INVALID_ARG
    bad = np.array([2], dtype=np.int64)                                   # unknown request
    assert step(bad, toks, ctypes.addressof(host), need) == pa.PA_ERR_INVALID_ARG
    c2 = pa.KVCache(1, 4)                                                 # one page: 3 + 3 tokens do not fit
    c2.add(1)
    c2.plan([1], [3], 4, 3)
    assert lib.pa_kv_cache_step(c2._h, 1, ids.ctypes.data, toks.ctypes.data, 3, 4,
                                ctypes.addressof(host), ctypes.addressof(host), need,
                                None, None, None, None, None, 4, 2, 128, 0.1, None, None, 0,
                                None) == pa.PA_ERR_NO_PAGES
    assert c.context_len(1) == 0 and c.free_pages == 8
    assert c2.context_len(1) == 3 and c2.free_pages == 0
    c.close()
    c2.close()
