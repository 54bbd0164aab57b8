"""Seeded synthetic inputs for paged attention.

This module is the ONE piece shared by the tests, the smoke check, the
benchmark and the oracle's callers. It draws random numbers and lays K/V out in
a page pool; it holds none of the attention arithmetic (no scores, no softmax,
no weighted sums), and it imports neither the oracle nor the CUDA library.

Contents:
  * bf16 <-> fp32 bit conversion (round to nearest even);
  * ``PageFreeList`` / ``RequestPages``: the page allocator and per-request
    page list whose behaviour Tutorial 13: Paged Attention and Memory
    Management states in section 3 "The Page Pool" and section 4 "The
    Request Cache" (last returned page reused first, fresh ids when none is
    returned, tail page filled first). Used to produce block tables and
    slot_mapping;
  * ``slot_of``: the flat-slot encoding of Reading vLLM's PagedAttention
    Kernel, 3.2 "Writing into the cache" (physical_block * block_size +
    offset_in_block), used to build slot_mapping inputs;
  * ``build_batch`` and the named workloads (shapes and value distributions of
    the pages' workloads).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

# ----------------------------------------------------------------------------
# bf16 bit helpers


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest even.
    NaN stays NaN (quiet bit forced)."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    nan = np.isnan(f)
    if nan.any():
        rounded = rounded.copy()
        rounded[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return rounded


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


_CHUNK = 1 << 22


def random_e4m3_codes(rng: np.random.Generator, shape, max_magnitude_code: int = 0x5F,
                      allow_nan: bool = False) -> np.ndarray:
    """Seeded e4m3 byte codes: a uniform magnitude code in [0, max_magnitude_code]
    (0x5F is 1.875 * 2^4 = 30) and a random sign; with allow_nan, any of the 256
    byte values (stale FP8 slots). Bytes only, no arithmetic of the method."""
    if allow_nan:
        return rng.integers(0, 256, size=shape, dtype=np.uint8)
    mag = rng.integers(0, max_magnitude_code + 1, size=shape, dtype=np.uint8)
    sign = (rng.integers(0, 2, size=shape, dtype=np.uint8) << 7).astype(np.uint8)
    return mag | sign


def normal_bf16(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    """bf16 bit patterns of N(0, std^2) draws.

    Large arrays are filled in fixed 4 Mi-element chunks, each from its own
    generator seeded by one draw of ``rng``, on a thread pool; the result
    depends only on ``rng``'s state, not on the thread count."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    n_chunks = max(1, -(-n // _CHUNK))
    seeds = rng.integers(0, 2**63 - 1, size=n_chunks)

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        x = np.random.default_rng(int(seeds[c])).standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            x *= np.float32(std)
        out[lo:hi] = bf16_bits(x)

    if n_chunks == 1:
        fill(0)
    else:
        workers = min(n_chunks, os.cpu_count() or 1)
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


# ----------------------------------------------------------------------------
# Page allocator fixture (Tutorial 13, sections 3 and 4, from the behaviour
# the tutorial states: a page given back is the first one handed out again;
# with none given back the pool hands out the next id it never used; a page
# cannot be given back twice; new tokens go into the request's last page
# while it has room, else onto a new page)


class DoubleFree(RuntimeError):
    """Raised when a page is given back to the pool twice."""


class PageFreeList:
    """Hands out page ids: the most recently returned id first, else the
    lowest id never handed out (``fresh`` counts those)."""

    def __init__(self, page_size: int):
        self.page_size = int(page_size)
        self.returned: List[int] = []  # stack, top = last returned
        self.in_use: set = set()
        self.fresh = 0

    def take(self) -> int:
        if self.returned:
            pid = self.returned[-1]
            del self.returned[-1]
        else:
            pid, self.fresh = self.fresh, self.fresh + 1
        self.in_use.add(pid)
        return pid

    def give_back(self, pid: int) -> None:
        if pid not in self.in_use:
            raise DoubleFree(f"page {pid} is not in use")
        self.in_use.discard(pid)
        self.returned.append(pid)


@dataclass
class RequestPages:
    """The pages one request holds in a pool, in logical order.

    ``policy="tail_fill"``: a token goes into the last page while that page
    has room, otherwise onto a fresh page (Tutorial 13, section 4; Week 3
    Day 4, "Decode Metadata": allocate only when the tail page is full).
    ``policy="new_page_per_chunk"``: each call's first token starts a fresh
    page, as the printed walkthrough of Tutorial 13 shows; the holes this
    leaves cannot be described by a block table plus a context length, so it
    serves only to reproduce that walkthrough.
    ``pages``: page ids; ``fill``: tokens held in each page; ``length``: tokens
    placed so far."""

    pool: PageFreeList
    policy: str = "tail_fill"
    pages: List[int] = field(default_factory=list)
    fill: List[int] = field(default_factory=list)
    length: int = 0

    def append(self, n_tokens: int) -> List[int]:
        """Place n_tokens new tokens, one at a time; returns their flat slots."""
        if self.policy not in ("tail_fill", "new_page_per_chunk"):
            raise ValueError(f"unknown policy {self.policy}")
        ps = self.pool.page_size
        out: List[int] = []
        for t in range(n_tokens):
            room = bool(self.pages) and self.fill[-1] < ps
            if not room or (t == 0 and self.policy == "new_page_per_chunk"):
                self.pages.append(self.pool.take())
                self.fill.append(0)
            out.append(slot_of(self.pages[-1], self.fill[-1], ps))
            self.fill[-1] += 1
        self.length += n_tokens
        return out

    def release(self) -> None:
        """Give every page of this request back to the pool exactly once."""
        held, self.pages, self.fill, self.length = self.pages, [], [], 0
        for pid in held:
            self.pool.give_back(pid)


def slot_of(page_id: int, offset_in_page: int, page_size: int) -> int:
    """Flat physical slot of a token: page_id * page_size + offset."""
    return int(page_id) * int(page_size) + int(offset_in_page)


# ----------------------------------------------------------------------------
# Batches


@dataclass
class PagedBatch:
    """One attention call's inputs plus the write that precedes it.

    Layouts: query [B, H_q, L, D]; pages [num_pages, H_kv, page_size, D]
    (bf16 bits); block_table [B, max_pages] and context_lens [B] int32;
    key_new/value_new [B, H_kv, L_new, D]; slot_mapping [B, L_new] int32.
    context_lens already count the L_new tokens that the append writes."""

    name: str
    B: int
    H_q: int
    H_kv: int
    D: int
    page_size: int
    L: int
    num_pages: int
    max_pages: int
    scale: float
    causal: bool
    query: np.ndarray
    key_pages: np.ndarray
    value_pages: np.ndarray
    block_table: np.ndarray
    context_lens: np.ndarray
    key_new: np.ndarray
    value_new: np.ndarray
    slot_mapping: np.ndarray
    seed: int = 0
    recipe: str = ""

    @property
    def L_new(self) -> int:
        return int(self.slot_mapping.shape[1])

    def kv_bytes(self) -> int:
        """Bytes of K and V that attention over context_lens has to read."""
        return int(self.context_lens.astype(np.int64).sum()) * self.H_kv * self.D * 2 * 2


def _page_tables_permutation(rng, n_pages_per_req: Sequence[int], num_pages: int):
    perm = rng.permutation(num_pages)
    tables, k = [], 0
    for n in n_pages_per_req:
        tables.append([int(x) for x in perm[k:k + n]])
        k += n
    return tables


def _page_tables_churn(rng, lens: Sequence[int], page_size: int, num_pages: int,
                       freed_fraction: float, step_tokens: int):
    """Shuffled pool with a fraction of ids freed and handed out again.

    Every pool id is allocated once and freed in random order (a shuffled free
    list); transient requests then take ``freed_fraction`` of the pages needed
    and release them (those ids go back on top of the returned stack); the
    real requests are then prefilled round-robin in chunks of ``step_tokens``
    with the tail-fill policy, so the first pages they get are the freed and
    reused ids. Returns (tables, transient page ids)."""
    pool = PageFreeList(page_size)
    ids = [pool.take() for _ in range(num_pages)]
    for i in rng.permutation(len(ids)):
        pool.give_back(ids[int(i)])
    need = sum(math.ceil(n / page_size) for n in lens)
    transient = RequestPages(pool)
    transient.append(int(freed_fraction * need) * page_size)
    ghost_ids = list(transient.pages)
    order = list(rng.permutation(len(ghost_ids)))
    for j in order:                       # release in random order
        pool.give_back(ghost_ids[int(j)])
    transient.pages = []
    caches = [RequestPages(pool) for _ in lens]
    remaining = list(lens)
    while any(r > 0 for r in remaining):
        for b, cache in enumerate(caches):
            if remaining[b] > 0:
                t = min(step_tokens, remaining[b])
                cache.append(t)
                remaining[b] -= t
    if pool.fresh != num_pages:
        raise AssertionError("pool grew beyond its sizing")
    return [c.pages for c in caches], ghost_ids


def build_batch(name: str, B: int, H_q: int, H_kv: int, D: int, page_size: int,
                L: int, context_lens: Sequence[int], seed: int,
                L_new: Optional[int] = None, placement: str = "permutation",
                pool_slack: float = 0.10, num_pages: Optional[int] = None,
                tables: Optional[List[List[int]]] = None, causal: bool = True,
                garbage_std: float = 10.0, pad_value: int = -1,
                freed_fraction: float = 0.20, step_tokens: int = 128,
                recipe: str = "") -> PagedBatch:
    """Seeded paged batch.

    Valid K/V (positions < context_len - L_new), query and the new rows are
    bf16 N(0,1). Every other slot of the pool (unreferenced pages, tail slots
    past the context, and the slots the append is about to write) holds
    seeded garbage N(0, garbage_std^2). block_table entries past a request's
    last page hold ``pad_value``."""
    rng = np.random.default_rng(seed)
    lens = [int(n) for n in context_lens]
    if L_new is None:
        L_new = L
    if any(n < L_new for n in lens):
        raise ValueError("every context must hold at least the L_new new tokens")
    pages_per_req = [max(1, math.ceil(n / page_size)) if n > 0 else 0 for n in lens]
    need = sum(pages_per_req)
    if num_pages is None:
        num_pages = max(1, math.ceil((1.0 + pool_slack) * need))
    if tables is None:
        if placement == "permutation":
            tables = _page_tables_permutation(rng, pages_per_req, num_pages)
        elif placement == "churn":
            tables, _ = _page_tables_churn(rng, lens, page_size, num_pages,
                                           freed_fraction, step_tokens)
        elif placement == "sequential":
            tables, k = [], 0
            for n in pages_per_req:
                tables.append(list(range(k, k + n)))
                k += n
        else:
            raise ValueError(placement)
    max_pages = max(1, max(len(t) for t in tables))
    block_table = np.full((B, max_pages), pad_value, dtype=np.int32)
    for b, t in enumerate(tables):
        block_table[b, :len(t)] = t

    shape = (num_pages, H_kv, page_size, D)
    key_pages = normal_bf16(rng, shape)
    value_pages = normal_bf16(rng, shape)
    # Garbage everywhere that holds no valid prefix token.
    valid = np.zeros((num_pages, page_size), dtype=bool)
    for b, t in enumerate(tables):
        prefix = lens[b] - L_new
        for pos in range(0, prefix, page_size):
            valid[t[pos // page_size], :min(page_size, prefix - pos)] = True
    bad_pages, bad_slots = np.nonzero(~valid)
    if bad_pages.size:
        g = garbage_std
        n_bad = bad_pages.size * H_kv * D
        gk = normal_bf16(rng, (bad_pages.size, H_kv, D), g)
        gv = normal_bf16(rng, (bad_pages.size, H_kv, D), g)
        key_pages[bad_pages, :, bad_slots, :] = gk
        value_pages[bad_pages, :, bad_slots, :] = gv
        del n_bad

    query = normal_bf16(rng, (B, H_q, L, D))
    key_new = normal_bf16(rng, (B, H_kv, L_new, D))
    value_new = normal_bf16(rng, (B, H_kv, L_new, D))
    slot_mapping = np.full((B, L_new), -1, dtype=np.int32)
    for b, t in enumerate(tables):
        for i in range(L_new):
            pos = lens[b] - L_new + i
            slot_mapping[b, i] = slot_of(t[pos // page_size], pos % page_size, page_size)
    return PagedBatch(name=name, B=B, H_q=H_q, H_kv=H_kv, D=D, page_size=page_size,
                      L=L, num_pages=num_pages, max_pages=max_pages,
                      scale=1.0 / math.sqrt(D), causal=causal, query=query,
                      key_pages=key_pages, value_pages=value_pages,
                      block_table=block_table,
                      context_lens=np.asarray(lens, dtype=np.int32),
                      key_new=key_new, value_new=value_new,
                      slot_mapping=slot_mapping, seed=seed, recipe=recipe)


# ----------------------------------------------------------------------------
# Named workloads (shapes of the pages' workloads; see the module docstring)

WORKLOADS = (
    "tiny_decode",            # B=2 H_q=4 H_kv=2 D=64 ps=4, ctx [10, 7], 16 pages
    "decode_b32_gqa7_ps16",   # B=32 H_q=28 H_kv=4 D=128 ps=16, ctx U[128, 4096]
    "decode_b64_ps128",       # B=64 H_q=32 H_kv=8 D=128 ps=128, ctx log-U[64, 8192]
    "prefill_chunk512",       # B=4 H_q=32 H_kv=8 D=128 ps=16, L=512 after U[0,2048] prefix
    "decode_long_b8",         # B=8 H_q=32 H_kv=8 D=128 ps=16, ctx U[16384, 32768]
)

_SEEDS = {name: 1001 + i for i, name in enumerate(WORKLOADS)}


def make_workload(name: str, pad_value: int = -1, seed: Optional[int] = None) -> PagedBatch:
    """The named seeded workloads (decode steps append one token per request
    before attending; the chunked prefill appends its 512 rows first)."""
    s = _SEEDS[name] if seed is None else seed
    rng = np.random.default_rng(s + 7919)          # lengths and table draws
    if name == "tiny_decode":
        # Request 0 is the mapping example of Week 3 Day 4 ("Why block_table
        # Matters"): pages [12, 5, 3], 10 tokens, page size 4. Request 1 takes
        # two other distinct ids.
        others = [int(x) for x in rng.permutation([i for i in range(16) if i not in (12, 5, 3)])[:2]]
        return build_batch(name, B=2, H_q=4, H_kv=2, D=64, page_size=4, L=1,
                           context_lens=[10, 7], seed=s, num_pages=16,
                           tables=[[12, 5, 3], others], pad_value=pad_value,
                           recipe="ctx [10,7]; request 0 pages [12,5,3]; 16 pages; "
                                  "values N(0,1), garbage N(0,10^2)")
    if name == "decode_b32_gqa7_ps16":
        lens = rng.integers(128, 4096, size=32, endpoint=True)
        return build_batch(name, B=32, H_q=28, H_kv=4, D=128, page_size=16, L=1,
                           context_lens=lens, seed=s, placement="permutation",
                           pad_value=pad_value,
                           recipe="ctx U[128,4096]; pool = total pages +10%, random "
                                  "permutation; values N(0,1)")
    if name == "decode_b64_ps128":
        lens = np.exp(rng.uniform(math.log(64), math.log(8192), size=64)).astype(np.int64)
        lens = np.clip(lens, 64, 8192)
        return build_batch(name, B=64, H_q=32, H_kv=8, D=128, page_size=128, L=1,
                           context_lens=lens, seed=s, placement="churn",
                           freed_fraction=0.20, step_tokens=128, pad_value=pad_value,
                           recipe="ctx log-U[64,8192]; shuffled pool, 20% of ids freed "
                                  "and reused (LIFO); values N(0,1)")
    if name == "prefill_chunk512":
        prefix = rng.integers(0, 2048, size=4, endpoint=True)
        return build_batch(name, B=4, H_q=32, H_kv=8, D=128, page_size=16, L=512,
                           context_lens=prefix + 512, seed=s, placement="churn",
                           freed_fraction=0.20, step_tokens=128, pad_value=pad_value,
                           recipe="prefix U[0,2048] + 512 new rows appended through "
                                  "slot_mapping (tail fill); causal; values N(0,1)")
    if name == "decode_long_b8":
        lens = rng.integers(16384, 32768, size=8, endpoint=True)
        return build_batch(name, B=8, H_q=32, H_kv=8, D=128, page_size=16, L=1,
                           context_lens=lens, seed=s, placement="permutation",
                           pad_value=pad_value,
                           recipe="ctx U[16384,32768]; fully shuffled pool, ragged "
                                  "tails; values N(0,1)")
    raise KeyError(name)
