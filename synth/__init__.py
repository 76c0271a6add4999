"""Seeded synthetic inputs shared by the CUDA path's tests, the oracle's tests and
the benchmark.

This module holds no attention or quantisation arithmetic: it only draws random
numbers, rounds them to bf16 storage, and lays out ragged batches (sequence
lengths, prefix sums, shuffled paged block tables).  Both sides receive exactly
the arrays produced here.

bf16 values are carried as ``numpy.uint16`` bit patterns (numpy has no bf16
dtype).  ``bf16_bits_to_f32`` is the exact widening used to look at them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

from .configs import CONFIGS, Workload, layer_kinds, layer_to_cache_map  # noqa: F401


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even) and return the bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    # keep NaN a NaN (not used by the generators, which only draw finite values)
    nan = np.isnan(x)
    if nan.any():
        r[nan] = 0x7FC0
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def bf16_normal(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    """N(0, scale^2) drawn in float32 and rounded to bf16 (bits)."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x = x * np.float32(scale)
    return f32_to_bf16_bits(x)


@dataclass
class PagedBatch:
    """A ragged batch laid out over a paged pool.

    ``block_table[b, i]`` is the physical block holding tokens
    ``[i*page_size, (i+1)*page_size)`` of sequence ``b``; unused entries are -1.
    """

    seq_lens: np.ndarray          # int32 [batch], tokens in cache (incl. the newest)
    block_table: np.ndarray       # int32 [batch, max_blocks]
    num_blocks: int               # pool size (physical blocks)
    page_size: int
    shared_prefix_blocks: int = 0  # leading table entries shared inside a group
    groups: np.ndarray | None = field(default=None)  # int32 [batch] group id

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])


def make_paged_batch(rng: np.random.Generator | None, seq_lens, page_size: int,
                     shuffle: bool = True, slack: float = 0.10,
                     max_blocks: int | None = None) -> PagedBatch:
    """Give every sequence its own blocks, drawn from a pool of
    ``ceil((1+slack) * sum ceil(L/P))`` blocks; ``shuffle`` permutes the physical ids."""
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    need = [(int(L) + page_size - 1) // page_size for L in seq_lens]
    total = int(sum(need))
    pool = max(total + 1, int(math.ceil(total * (1.0 + slack))))
    ids = rng.permutation(pool).astype(np.int32) if shuffle else np.arange(pool, dtype=np.int32)
    mb = max(need) if max_blocks is None else max_blocks
    table = np.full((len(seq_lens), max(mb, 1)), -1, dtype=np.int32)
    cur = 0
    for b, n in enumerate(need):
        table[b, :n] = ids[cur:cur + n]
        cur += n
    return PagedBatch(seq_lens=seq_lens, block_table=table, num_blocks=pool, page_size=page_size)


def make_prefix_shared_batch(rng: np.random.Generator, num_groups: int, seqs_per_group: int,
                             prefix_len: int, new_len: int, page_size: int,
                             slack: float = 0.10) -> PagedBatch:
    """Groups of sequences whose first ``prefix_len`` tokens live in blocks shared
    by the whole group (read-only), followed by private blocks for ``new_len``
    appended tokens.  ``prefix_len`` must be a multiple of ``page_size``."""
    assert prefix_len % page_size == 0
    pre = prefix_len // page_size
    priv = (new_len + page_size - 1) // page_size
    batch = num_groups * seqs_per_group
    total = num_groups * pre + batch * priv
    pool = max(total + 1, int(math.ceil(total * (1.0 + slack))))
    ids = rng.permutation(pool).astype(np.int32)
    table = np.full((batch, pre + priv), -1, dtype=np.int32)
    cur = 0
    groups = np.repeat(np.arange(num_groups, dtype=np.int32), seqs_per_group)
    for g in range(num_groups):
        shared = ids[cur:cur + pre]
        cur += pre
        for s in range(seqs_per_group):
            table[g * seqs_per_group + s, :pre] = shared
    for b in range(batch):
        table[b, pre:] = ids[cur:cur + priv]
        cur += priv
    seq_lens = np.full(batch, prefix_len + new_len, dtype=np.int32)
    return PagedBatch(seq_lens=seq_lens, block_table=table, num_blocks=pool, page_size=page_size,
                      shared_prefix_blocks=pre, groups=groups)


def cu_from_counts(counts) -> np.ndarray:
    """Exclusive prefix sums with a trailing total: ``cu[b+1] - cu[b] = counts[b]``."""
    counts = np.asarray(counts, dtype=np.int64)
    cu = np.zeros(len(counts) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(counts)
    return cu


def seq_lens_for(w: "Workload", rng: np.random.Generator) -> np.ndarray:
    """Context lengths drawn as the workload's recipe states."""
    if w.len_kind == "fixed":
        return np.asarray(w.len_values, dtype=np.int32)
    if w.len_kind == "uniform":
        lo, hi = w.len_values
        return rng.integers(lo, hi + 1, size=w.batch, dtype=np.int64).astype(np.int32)
    if w.len_kind == "lognormal":
        median, sigma, cap = w.len_values
        x = np.exp(rng.normal(math.log(median), sigma, size=w.batch))
        return np.clip(np.rint(x), 1, cap).astype(np.int32)
    if w.len_kind == "prefix":
        prefix, new = w.len_values
        return np.full(w.batch, prefix + new, dtype=np.int32)
    raise ValueError(w.len_kind)


def sample_rows(rng: np.random.Generator, n_total: int, n: int) -> np.ndarray:
    """``n`` distinct row indices out of ``n_total`` (sorted)."""
    n = min(n, n_total)
    return np.sort(rng.choice(n_total, size=n, replace=False)).astype(np.int64)
