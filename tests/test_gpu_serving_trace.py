"""A small serving trace end to end: the C++ page allocator plans every step,
the tables go to the device, the new K/V rows are appended and attention runs
on the GPU (decode group and per-request prefill chunks, as the serving-trace
driver issues them). At every step the allocator's tables must equal the
Python allocator fixture's bit for bit, the device pools must equal the
oracle's pools bit for bit, and every attention output must match the oracle
run on the fixture's tables."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import N_THREADS, assert_close, check_no_device_error, dev, host_bits, host_f64

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("native", [False, True], ids=["plan_then_calls", "native_step"])
@pytest.mark.parametrize("page_size", [16, 1])
def test_serving_trace_small(page_size, native):
    """native_step: each step is one pa_kv_cache_step call (plan into pinned
    memory, one table copy, append, attention); the tables it copied to the
    device are compared with the fixture's."""
    import paged_kv_attention_06_gb300 as pa
    rng = np.random.default_rng(11 + page_size)
    n_req, batch, chunk = 6, 3, 64
    H_q, H_kv, D = 8, 2, 128
    prompts = rng.integers(20, 300, size=n_req, endpoint=True)
    outputs = rng.integers(3, 10, size=n_req, endpoint=True)
    max_pages = -(-int(prompts.max() + outputs.max()) // page_size)
    num_pages = batch * max_pages + 8
    cache = pa.KVCache(num_pages, page_size)
    pool = wl.PageFreeList(page_size)
    kp_h = wl.normal_bf16(rng, (num_pages, H_kv, page_size, D))
    vp_h = wl.normal_bf16(rng, (num_pages, H_kv, page_size, D))
    kp, vp = dev(kp_h), dev(vp_h)
    scale = D ** -0.5

    tables_h = torch.empty((1 << 16,), dtype=torch.uint8).pin_memory()
    tables_d = torch.empty((1 << 16,), dtype=torch.uint8, device="cuda")

    def call(ids, toks, l_new):
        # the fixture's tables, built independently, feed the oracle
        f_sm = np.full((len(ids), l_new), -1, dtype=np.int32)
        f_bt = np.full((len(ids), max_pages), -1, dtype=np.int32)
        f_cl = np.zeros((len(ids),), dtype=np.int32)
        for i, sid in enumerate(ids):
            f_sm[i, :toks[i]] = fixture[sid].append(toks[i])
            f_bt[i, :len(fixture[sid].pages)] = fixture[sid].pages
            f_cl[i] = fixture[sid].length
        n = len(ids)
        k_new = wl.normal_bf16(rng, (n, H_kv, l_new, D))
        v_new = wl.normal_bf16(rng, (n, H_kv, l_new, D))
        q = wl.normal_bf16(rng, (n, H_q, l_new, D))
        if native:
            out = cache.step(ids, toks, l_new, max_pages, tables_h, tables_d, dev(k_new),
                             dev(v_new), dev(q), kp, vp, scale=scale)
            check_no_device_error()
            nb = n * max_pages
            t = tables_d[:cache.step_table_bytes(n, max_pages, l_new)].view(torch.int32).cpu().numpy()
            assert np.array_equal(t[:nb].reshape(n, max_pages), f_bt)
            assert np.array_equal(t[nb:nb + n], f_cl)
            assert np.array_equal(t[nb + n:].reshape(n, l_new), f_sm)
        else:
            bt, cl, sm = cache.plan(ids, toks, max_pages, l_new)
            assert np.array_equal(bt, f_bt) and np.array_equal(cl, f_cl) and np.array_equal(sm, f_sm)
            pa.pa_append_kv(dev(k_new), dev(v_new), kp, vp, dev(sm), page_size)
            out = pa.pa_attention(dev(q), kp, vp, dev(bt), dev(cl), page_size, scale=scale,
                                  max_context_len=int(cl.max()))
            check_no_device_error()
        oracle.append_kv(k_new, v_new, kp_h, vp_h, f_sm, page_size)
        assert np.array_equal(host_bits(kp), kp_h) and np.array_equal(host_bits(vp), vp_h)
        ref = oracle.attention(q, kp_h, vp_h, f_bt, f_cl, page_size, scale=scale,
                               n_threads=N_THREADS)
        assert_close(host_f64(out), ref, f"step with {n} request(s), L={l_new}")

    fixture = {}
    waiting, active = list(range(n_req)), {}
    calls = 0
    while waiting or active:
        while waiting and len(active) < batch:
            sid = waiting.pop(0)
            cache.add(sid)
            fixture[sid] = wl.RequestPages(pool)
            active[sid] = [0, 0]
        dec = [s for s, (p, o) in active.items() if p >= prompts[s]]
        pre = [s for s, (p, o) in active.items() if p < prompts[s]]
        if dec:
            call(dec, [1] * len(dec), 1)
            calls += 1
            for s in dec:
                active[s][1] += 1
        for s in pre:
            take = int(min(chunk, prompts[s] - active[s][0]))
            call([s], [take], take)
            calls += 1
            active[s][0] += take
        for s in [s for s, (p, o) in active.items() if o >= outputs[s]]:
            cache.release(s)
            fixture.pop(s).release()
            del active[s]
    assert cache.free_pages == num_pages
    assert calls > n_req
    cache.close()
