"""Helpers for the GPU tests: move seeded batches to the device, run the CUDA
path through the C ABI, run the oracle on the same inputs, compare."""
import os

import numpy as np
import torch

import oracle
import workloads as wl

# Tolerance for attention outputs (fp32 accumulation, bf16 out) against the
# fp64 oracle: max |err| and mean |err| over the compared elements.
MAX_ERR = 2e-2
MEAN_ERR = 2e-3

# The same comparison relative to the size of the reference: max |err| <=
# REL * max |ref| and mean |err| <= REL * mean |ref|. With N(0,1) values and
# 16k-40k visible keys an output element is about 0.01, so the absolute bounds
# alone cannot fail there. The kernels' own error is the bf16 rounding of the
# output (relative 2^-9 at most) and of the probabilities fed to P.V (relative
# 2^-9 per term, zero-mean, so about 2^-9/sqrt(3) of the output's size), with
# fp32 accumulation far below both; 2^-6 leaves a margin of 8x over the
# worst element. Dropping a fraction f of a row's keys moves its output by
# about sqrt(f) of its size, so a row that loses more than ~0.03 % of its keys
# fails the mean bound.
REL = 2.0 ** -6

# Every comparison made in this process: (what, max|err|, mean|err|,
# max|ref|, mean|ref|), written out by the session hook in conftest.py when
# PA_PARITY_LOG names a file.
PARITY_LOG = []

N_THREADS = os.cpu_count() or 1


def dev(x, device="cuda"):
    if x.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(x)).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


class DeviceBatch:
    """A PagedBatch resident on the GPU."""

    def __init__(self, b: wl.PagedBatch, device="cuda"):
        self.b = b
        self.query = dev(b.query, device)
        self.key_pages = dev(b.key_pages, device)
        self.value_pages = dev(b.value_pages, device)
        self.block_table = dev(b.block_table, device)
        self.context_lens = dev(b.context_lens, device)
        self.key_new = dev(b.key_new, device)
        self.value_new = dev(b.value_new, device)
        self.slot_mapping = dev(b.slot_mapping, device)


def gpu_step(db: DeviceBatch, route: str = "attention", append: bool = True):
    """append (if the batch has new rows) then attention; returns out tensor."""
    import paged_kv_attention_06_gb300 as pa
    b = db.b
    if append and b.L_new > 0:
        pa.pa_append_kv(db.key_new, db.value_new, db.key_pages, db.value_pages,
                        db.slot_mapping, b.page_size)
    fn = {"attention": pa.pa_attention, "decode": pa.pa_decode, "prefill": pa.pa_prefill,
          "prefill_split": pa.pa_prefill_split}[route]
    kwargs = dict(scale=b.scale, causal=b.causal)
    if route in ("attention", "decode"):
        kwargs["max_context_len"] = int(b.context_lens.max()) if b.B else 0
    return fn(db.query, db.key_pages, db.value_pages, db.block_table, db.context_lens,
              b.page_size, **kwargs)


def oracle_pages(b: wl.PagedBatch):
    kp, vp = b.key_pages.copy(), b.value_pages.copy()
    if b.L_new > 0:
        oracle.append_kv(b.key_new, b.value_new, kp, vp, b.slot_mapping, b.page_size)
    return kp, vp


def oracle_out(b: wl.PagedBatch, kp, vp, rows=None):
    return oracle.attention(b.query, kp, vp, b.block_table, b.context_lens, b.page_size,
                            scale=b.scale, causal=b.causal, rows=rows, n_threads=N_THREADS)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mag = np.abs(ref)
    emax, emean = float(err.max()), float(err.mean())
    rmax, rmean = float(mag.max()), float(mag.mean())
    PARITY_LOG.append((what, emax, emean, rmax, rmean))
    assert emax <= MAX_ERR, f"{what}: max|err| {emax:.3e} > {MAX_ERR}"
    assert emean <= MEAN_ERR, f"{what}: mean|err| {emean:.3e} > {MEAN_ERR}"
    assert emax <= REL * rmax, \
        f"{what}: max|err| {emax:.3e} > 2^-6 * max|ref| ({REL * rmax:.3e})"
    assert emean <= REL * rmean, \
        f"{what}: mean|err| {emean:.3e} > 2^-6 * mean|ref| ({REL * rmean:.3e})"
    return emax, emean


def check_no_device_error():
    import paged_kv_attention_06_gb300 as pa
    st, flags = pa.pa_get_device_error()
    assert st == 0 and flags == 0, f"device error status {st} flags {flags:#x}"
