"""FP8 (e4m3) page pools with per-tensor scales on the GPU, through the C
ABI, against the fp64 oracle on the same inputs: the quantising append bit
for bit, decode attention within the stated tolerance (max |err| <= 2e-2,
mean |err| <= 2e-3) over the exact decoded page values."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import N_THREADS, assert_close, check_no_device_error, dev, host_f64

pytestmark = pytest.mark.gpu


def _pa():
    import paged_kv_attention_06_gb300 as pa
    return pa


def _u8(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


@pytest.mark.parametrize("ps", [16, 1, 128])
@pytest.mark.parametrize("scales", [(0.05, 0.031), (1.0, 0.25), (0.003, 0.7)])
def test_append_fp8_bit_exact(ps, scales):
    pa = _pa()
    k_scale, v_scale = scales
    rng = np.random.default_rng(ps * 7 + int(k_scale * 1000))
    B, H_kv, L_new, D = 3, 4, 19, 128
    P = (B * L_new) // ps + 8
    key = wl.normal_bf16(rng, (B, H_kv, L_new, D), std=1.0)
    value = wl.normal_bf16(rng, (B, H_kv, L_new, D), std=2.0)
    # saturating, subnormal and zero elements
    key[0, 0, 0, :8] = wl.bf16_bits(np.float32([600, -600, 1e-6, -1e-6, 0.0, -0.0, 20.0, 3e-3]))
    slots = rng.permutation(P * ps)[:B * L_new].reshape(B, L_new).astype(np.int32)
    slots[1, 4] = -1
    slots[2, 7] = -1
    kp0 = wl.random_e4m3_codes(rng, (P, H_kv, ps, D), allow_nan=True)
    vp0 = wl.random_e4m3_codes(rng, (P, H_kv, ps, D), allow_nan=True)
    kp_d, vp_d = _u8(kp0), _u8(vp0)
    pa.pa_append_kv_fp8(dev(key), dev(value), kp_d, vp_d, dev(slots), ps, k_scale, v_scale)
    check_no_device_error()
    kp, vp = kp0.copy(), vp0.copy()
    assert oracle.append_kv_fp8(key, value, kp, vp, slots, ps, k_scale, v_scale) == 0
    assert np.array_equal(kp_d.cpu().numpy(), kp)
    assert np.array_equal(vp_d.cpu().numpy(), vp)


def _fp8_batch(name, B, H_q, H_kv, ps, L, lens, seed, causal=True, placement="permutation"):
    b = wl.build_batch(name, B=B, H_q=H_q, H_kv=H_kv, D=128, page_size=ps, L=L,
                       context_lens=lens, seed=seed, L_new=0, causal=causal,
                       placement=placement)
    rng = np.random.default_rng(seed + 1000)
    kc = wl.random_e4m3_codes(rng, b.key_pages.shape)
    vc = wl.random_e4m3_codes(rng, b.value_pages.shape)
    # stale slots (past every context, in unreferenced pages) hold any byte
    stale = wl.random_e4m3_codes(rng, b.key_pages.shape, allow_nan=True)
    used = np.zeros(b.key_pages.shape[0], bool)
    for r in range(B):
        n = int(b.context_lens[r])
        for j in range(-(-n // ps)):
            used[b.block_table[r, j]] = True
    kc[~used], vc[~used] = stale[~used], stale[~used][::-1]
    for r in range(B):
        n = int(b.context_lens[r])
        if n % ps:
            tail = b.block_table[r, n // ps]
            kc[tail, :, n % ps:] = stale[tail, :, n % ps:]
            vc[tail, :, n % ps:] = 0x7F                         # NaN codes
    return b, kc, vc


def _run(b, kc, vc, k_scale, v_scale, rows=None):
    pa = _pa()
    q = dev(b.query)
    out = pa.pa_decode_fp8(q, _u8(kc), _u8(vc), dev(b.block_table), dev(b.context_lens),
                           b.page_size, k_scale, v_scale, scale=b.scale, causal=b.causal,
                           max_context_len=int(b.context_lens.max()))
    check_no_device_error()
    ref = oracle.attention_fp8(b.query, kc, vc, k_scale, v_scale, b.block_table,
                               b.context_lens, b.page_size, scale=b.scale, causal=b.causal,
                               rows=rows, n_threads=N_THREADS)
    got = host_f64(out)
    if rows is not None:
        got = got[rows[:, 0], rows[:, 1], rows[:, 2]]
    return got, ref


@pytest.mark.parametrize("ps", [16, 128, 4, 1])
@pytest.mark.parametrize("H_q,H_kv", [(28, 4), (8, 8), (32, 4)])
def test_decode_fp8_matches_oracle(ps, H_q, H_kv):
    lens = [1, 63, 64, 65, 127, 300, 1000, 2051]
    b, kc, vc = _fp8_batch("fp8dec", 8, H_q, H_kv, ps, 1, lens, seed=ps + H_q)
    got, ref = _run(b, kc, vc, 0.05, 0.04)
    assert_close(got, ref, f"fp8 decode ps={ps} G={H_q // H_kv}")


@pytest.mark.parametrize("L,causal", [(2, True), (5, True), (8, True), (4, False), (16, True)])
def test_decode_fp8_multi_row(L, causal):
    lens = [L, L + 5, 130, 777, 64 + L]
    b, kc, vc = _fp8_batch("fp8rows", 5, 16, 4, 16, L, lens, seed=40 + L, causal=causal)
    got, ref = _run(b, kc, vc, 0.02, 0.06)
    assert_close(got, ref, f"fp8 decode L={L} causal={causal}")


def test_decode_fp8_headline_shape_every_row():
    """The 7B-class GQA decode batch (B = 32, H_q = 28, H_kv = 4, page_size 16,
    contexts U[128, 4096], shuffled pool) with e4m3 pools."""
    rng = np.random.default_rng(1002)
    lens = [int(x) for x in rng.integers(128, 4097, size=32)]
    b, kc, vc = _fp8_batch("fp8head", 32, 28, 4, 16, 1, lens, seed=1002)
    got, ref = _run(b, kc, vc, 0.05, 0.05)
    assert_close(got, ref, "fp8 headline shape")


def test_decode_fp8_empty_contexts_give_zeros():
    b, kc, vc = _fp8_batch("fp8empty", 3, 8, 2, 16, 3, [0, 2, 40], seed=51)
    got, ref = _run(b, kc, vc, 0.1, 0.1)
    assert np.all(got[0] == 0)
    assert_close(got, ref, "fp8 empty contexts")


def test_append_then_decode_fp8():
    """Append the step's token with the quantising append, then decode over
    the updated e4m3 pools: the oracle does the same with its own append."""
    pa = _pa()
    b = wl.make_workload("decode_b32_gqa7_ps16")
    rng = np.random.default_rng(77)
    kc = wl.random_e4m3_codes(rng, b.key_pages.shape)
    vc = wl.random_e4m3_codes(rng, b.value_pages.shape)
    ks, vs = 0.05, 0.05
    kp_d, vp_d = _u8(kc), _u8(vc)
    pa.pa_append_kv_fp8(dev(b.key_new), dev(b.value_new), kp_d, vp_d, dev(b.slot_mapping),
                        b.page_size, ks, vs)
    out = pa.pa_decode_fp8(dev(b.query), kp_d, vp_d, dev(b.block_table), dev(b.context_lens),
                           b.page_size, ks, vs, scale=b.scale,
                           max_context_len=int(b.context_lens.max()))
    check_no_device_error()
    kp, vp = kc.copy(), vc.copy()
    oracle.append_kv_fp8(b.key_new, b.value_new, kp, vp, b.slot_mapping, b.page_size, ks, vs)
    assert np.array_equal(kp_d.cpu().numpy(), kp) and np.array_equal(vp_d.cpu().numpy(), vp)
    ref = oracle.attention_fp8(b.query, kp, vp, ks, vs, b.block_table, b.context_lens,
                               b.page_size, scale=b.scale, n_threads=N_THREADS)
    assert_close(host_f64(out), ref, "fp8 append + decode")


# ----------------------------------------------------------------------------
# Prefill over e4m3 pools (bf16 copies of the visible tokens + the tensor-core
# prefill kernels)


def _run_prefill(b, kc, vc, k_scale, v_scale, rows=None, max_context_len=None):
    pa = _pa()
    mcl = int(b.context_lens.max()) if max_context_len is None else max_context_len
    out = pa.pa_prefill_fp8(dev(b.query), _u8(kc), _u8(vc), dev(b.block_table),
                            dev(b.context_lens), b.page_size, k_scale, v_scale, scale=b.scale,
                            causal=b.causal, max_context_len=mcl)
    ref = oracle.attention_fp8(b.query, kc, vc, k_scale, v_scale, b.block_table,
                               b.context_lens, b.page_size, scale=b.scale, causal=b.causal,
                               rows=rows, n_threads=N_THREADS)
    got = host_f64(out)
    if rows is not None:
        got = got[rows[:, 0], rows[:, 1], rows[:, 2]]
    return got, ref


@pytest.mark.parametrize("ps", [16, 1, 2, 128, 256])
@pytest.mark.parametrize("L,causal", [(64, True), (130, True), (257, False)])
def test_prefill_fp8_matches_oracle(ps, L, causal):
    """Pool pages of 1, 2, 16, 128 and 256 tokens (the copy gathers every
    size into 128-token pages; at 256 a copy page is half a pool page); row
    tiles with a ragged tail; causal and not."""
    lens = [L, L + 300, 700, 2 * L + 5]
    b, kc, vc = _fp8_batch("fp8pre", 4, 8, 2, ps, L, lens, seed=300 + L + ps, causal=causal)
    got, ref = _run_prefill(b, kc, vc, 0.05, 0.04)
    check_no_device_error()
    assert_close(got, ref, f"fp8 prefill ps={ps} L={L} causal={causal}")


@pytest.mark.parametrize("H_q,H_kv", [(6, 2), (4, 4), (14, 2)])   # groups of 3 and 7 (pairs, last head repeated) / 1 (one head)
def test_prefill_fp8_odd_groups(H_q, H_kv):
    b, kc, vc = _fp8_batch("fp8pre1", 3, H_q, H_kv, 16, 100, [100, 333, 1000], seed=61)
    got, ref = _run_prefill(b, kc, vc, 0.02, 0.09)
    check_no_device_error()
    assert_close(got, ref, f"fp8 prefill G={H_q // H_kv}")


def test_prefill_fp8_head_pairs_kernel_sampled_rows():
    """Enough (request, head pair, 128-row tile) items for the whole-item
    pairs kernel (8 x 4 x 8 = 256 items): sampled rows against the oracle."""
    rng = np.random.default_rng(62)
    lens = [int(x) for x in rng.integers(512, 1600, size=8)]
    b, kc, vc = _fp8_batch("fp8pairs", 8, 16, 4, 16, 512, lens, seed=62)
    rows = np.stack([rng.integers(0, 8, 400), rng.integers(0, 16, 400),
                     rng.integers(0, 512, 400)], axis=1).astype(np.int32)
    rows[:8, 2] = [0, 1, 127, 128, 255, 256, 510, 511]
    got, ref = _run_prefill(b, kc, vc, 0.05, 0.05, rows=rows)
    check_no_device_error()
    assert_close(got, ref, "fp8 prefill pairs kernel")


def test_prefill_fp8_short_and_empty_contexts():
    b, kc, vc = _fp8_batch("fp8pre0", 3, 8, 2, 16, 40, [0, 7, 40], seed=63)
    got, ref = _run_prefill(b, kc, vc, 0.1, 0.1)
    check_no_device_error()
    assert np.all(got[0] == 0)                 # no keys at all
    assert np.all(got[1, :, :33] == 0)         # rows before the first key
    assert_close(got, ref, "fp8 prefill short contexts")


def test_prefill_fp8_nan_code_in_a_visible_slot():
    """A NaN code among the keys a row sees makes that row NaN; rows and
    requests that do not see it stay finite."""
    b, kc, vc = _fp8_batch("fp8nan", 2, 8, 2, 16, 40, [300, 200], seed=67)
    kc = kc.copy()
    pos = 270                                  # visible to rows 10.. of request 0 (causal)
    kc[b.block_table[0, pos // 16], 1, pos % 16, 5] = 0x7F
    got, _ = _run_prefill(b, kc, vc, 0.05, 0.05)
    check_no_device_error()
    first = pos - (300 - 40)                   # first row of request 0 that sees it
    assert np.all(np.isnan(got[0, 4:8, first:]).any(axis=-1))   # heads of KV head 1
    assert np.all(np.isfinite(got[0, 4:8, :first]))
    assert np.all(np.isfinite(got[0, :4])) and np.all(np.isfinite(got[1]))


def test_prefill_fp8_agrees_with_decode_kernel():
    b, kc, vc = _fp8_batch("fp8agree", 2, 8, 2, 16, 48, [48, 900], seed=64)
    pa = _pa()
    got_p, ref = _run_prefill(b, kc, vc, 0.05, 0.05)
    got_d, _ = _run(b, kc, vc, 0.05, 0.05)
    check_no_device_error()
    assert_close(got_p, ref, "prefill kernels")
    assert_close(got_d, ref, "split-KV kernel")


def test_prefill_fp8_context_beyond_bound_is_flagged_and_cut():
    pa = _pa()
    b, kc, vc = _fp8_batch("fp8cut", 2, 8, 2, 16, 16, [200, 130], seed=65)
    got, _ = _run_prefill(b, kc, vc, 0.05, 0.05, max_context_len=100)   # copies 128 tokens
    status, flags = pa.pa_get_device_error()
    assert flags & pa.PA_DEVERR_CONTEXT_LEN
    cut = b.context_lens.copy()
    cut[:] = np.minimum(cut, 128)
    ref = oracle.attention_fp8(b.query, kc, vc, 0.05, 0.05, b.block_table, cut, b.page_size,
                               scale=b.scale, causal=b.causal, n_threads=N_THREADS)
    assert_close(got, ref, "fp8 prefill, contexts cut to the copy")


def test_prefill_fp8_rejects_bad_arguments():
    pa = _pa()
    b, kc, vc = _fp8_batch("fp8bad", 1, 8, 2, 16, 8, [40], seed=66)
    args = (dev(b.query), _u8(kc), _u8(vc), dev(b.block_table), dev(b.context_lens),
            b.page_size)
    shape = pa.make_shape(b.query.shape, kc.shape, b.block_table.shape[1])
    need = pa.pa_prefill_fp8_workspace_bytes(shape, 40)
    assert need > 0
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_prefill_fp8(*args, 0.05, 0.05, max_context_len=40, workspace=small)
    assert e.value.status == pa.PA_ERR_WORKSPACE
    with pytest.raises(pa.PagedAttentionError) as e:
        pa.pa_prefill_fp8(*args, 0.0, 0.05, max_context_len=40)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    check_no_device_error()


def test_prefill_fp8_chunk512_sampled_rows():
    """The bench's prefill workload (4 requests, 512-row chunks after ragged
    prefixes, H_q = 32, H_kv = 8) over e4m3 pools: the quantising append of
    the chunk's K/V, then pa_prefill_fp8 as the bench calls it; sampled rows
    against the oracle run on the oracle's own append."""
    pa = _pa()
    b = wl.make_workload("prefill_chunk512")
    rng = np.random.default_rng(b.seed + 9)
    kc = wl.random_e4m3_codes(rng, b.key_pages.shape)
    vc = wl.random_e4m3_codes(rng, b.value_pages.shape)
    ks, vs = 0.05, 0.05
    kp_d, vp_d = _u8(kc), _u8(vc)
    pa.pa_append_kv_fp8(dev(b.key_new), dev(b.value_new), kp_d, vp_d, dev(b.slot_mapping),
                        b.page_size, ks, vs)
    out = pa.pa_prefill_fp8(dev(b.query), kp_d, vp_d, dev(b.block_table), dev(b.context_lens),
                            b.page_size, ks, vs, scale=b.scale, causal=True,
                            max_context_len=int(b.context_lens.max()))
    check_no_device_error()
    kp, vp = kc.copy(), vc.copy()
    oracle.append_kv_fp8(b.key_new, b.value_new, kp, vp, b.slot_mapping, b.page_size, ks, vs)
    assert np.array_equal(kp_d.cpu().numpy(), kp) and np.array_equal(vp_d.cpu().numpy(), vp)
    rows = []
    for r in range(b.B):
        for i in sorted(set([0, 1, 63, 64, 127, 128, 255, 256, 383, 510, 511] +
                            list(rng.integers(0, b.L, 5)))):
            for h in range(0, b.H_q, 3):
                rows.append((r, h, i))
    rows = np.asarray(rows, dtype=np.int32)
    ref = oracle.attention_fp8(b.query, kp, vp, ks, vs, b.block_table, b.context_lens,
                               b.page_size, scale=b.scale, causal=True, rows=rows,
                               n_threads=N_THREADS)
    got = host_f64(out)[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, ref, "fp8 prefill_chunk512 sampled")


@pytest.mark.parametrize("L", [1, 8, 9, 200])
def test_attention_fp8_dispatch_is_the_routed_call(L):
    """pa_attention_fp8 gives the bits of pa_decode_fp8 for up to 8 query rows
    and of pa_prefill_fp8 beyond, and both match the oracle."""
    pa = _pa()
    b, kc, vc = _fp8_batch("fp8route", 3, 8, 2, 16, L, [L + 40, 700, 2 * L + 3], seed=70 + L)
    args = (dev(b.query), _u8(kc), _u8(vc), dev(b.block_table), dev(b.context_lens), b.page_size,
            0.05, 0.05)
    mcl = int(b.context_lens.max())
    got = pa.pa_attention_fp8(*args, scale=b.scale, max_context_len=mcl)
    routed = (pa.pa_decode_fp8 if L <= 8 else pa.pa_prefill_fp8)(*args, scale=b.scale,
                                                                 max_context_len=mcl)
    check_no_device_error()
    assert torch.equal(got.view(torch.int16), routed.view(torch.int16))
    ref = oracle.attention_fp8(b.query, kc, vc, 0.05, 0.05, b.block_table, b.context_lens,
                               b.page_size, scale=b.scale, causal=True, n_threads=N_THREADS)
    assert_close(host_f64(got), ref, f"pa_attention_fp8 L={L}")
