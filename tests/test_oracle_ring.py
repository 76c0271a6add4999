"""Pins of the oracle's window-bounded (ring) cache addressing.

A local layer attends over a window of W keys ("Character.AI inference
article", secret 1: most layers use a 1024-token sliding window), so a cache
that serves only local layers needs to keep just the pages that a window can
touch: with R table entries per sequence, logical page p lives in entry p % R
and overwrites page p - R.  The ring is a pure re-addressing of the paged
cache, so attention over it must equal attention over a full table holding
the same tokens, exactly, whenever the keys it reads are resident.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def ring_and_linear(rng, lens, page, d, ring, chunk):
    """The same tokens appended chunk by chunk into a linear cache (full table)
    and a ring cache (ring entries per sequence); returns both setups."""
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    need = [(int(L) + page - 1) // page for L in lens]
    lin_pool = sum(need)
    lin_table = np.full((B, max(need)), -1, np.int32)
    ids = rng.permutation(lin_pool).astype(np.int32)
    cur = 0
    for b, n in enumerate(need):
        lin_table[b, :n] = ids[cur:cur + n]
        cur += n
    ring_table = rng.permutation(B * ring).astype(np.int32).reshape(B, ring)
    lin = oracle.Cache.empty(lin_pool, page, d)
    rc = oracle.Cache.empty(B * ring, page, d)
    k_all = [synth.bf16_normal(rng, (int(L), d)) for L in lens]
    v_all = [synth.bf16_normal(rng, (int(L), d)) for L in lens]
    done = np.zeros(B, np.int32)
    while (done < lens).any():
        n = np.minimum(lens - done, chunk).astype(np.int32)
        cu = synth.cu_from_counts(n)
        k = np.concatenate([k_all[b][done[b]:done[b] + n[b]] for b in range(B)])
        v = np.concatenate([v_all[b][done[b]:done[b] + n[b]] for b in range(B)])
        cur_lens = done + n
        oracle.quant_append(lin, lin_table, cur_lens, cu, k, v)
        oracle.quant_append(rc, ring_table, cur_lens, cu, k, v, ring_blocks=ring)
        done = cur_lens
    return lin, lin_table, rc, ring_table, k_all, v_all


@pytest.mark.parametrize("page,W", [(16, 64), (64, 1024), (16, 40)])
def test_ring_decode_equals_full_table_exactly(page, W):
    rng = np.random.default_rng(page + W)
    d, H = 16, 4
    ring = (W - 1) // page + 2  # the pages a window of W keys can touch
    lens = [1, page - 1, page, ring * page, ring * page + 1, 3 * ring * page + 17, 5 * W + 3]
    lin, lt, rc, rt, _, _ = ring_and_linear(rng, lens, page, d, ring, chunk=ring * page)
    q = synth.bf16_normal(rng, (len(lens), H, d))
    a, la = oracle.decode(lin, lt, lens, q, W, 1 / math.sqrt(d))
    b, lb = oracle.decode(rc, rt, lens, q, W, 1 / math.sqrt(d), ring_blocks=ring)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_ring_prefill_rows_equal_full_table_exactly():
    rng = np.random.default_rng(3)
    d, H, page, W, qlen = 16, 2, 16, 48, 20
    ring = (W + qlen - 2) // page + 2  # a chunk of qlen queries and their windows
    lens = [qlen, 100, 333, 517]
    lin, lt, rc, rt, _, _ = ring_and_linear(rng, lens, page, d, ring, chunk=37)
    cu_q = synth.cu_from_counts([qlen] * len(lens))
    rs, rp = oracle.prefill_rows(cu_q, lens)
    q = synth.bf16_normal(rng, (len(rs), H, d))
    a, _ = oracle.attention(lin, lt, lens, q, rs, rp, W, 0.25)
    b, _ = oracle.attention(rc, rt, lens, q, rs, rp, W, 0.25, ring_blocks=ring)
    assert np.array_equal(a, b)


def test_ring_slots_hold_the_newest_tokens():
    rng = np.random.default_rng(4)
    d, page, ring = 8, 16, 3
    L = 7 * page + 5  # pages 0..7; entry p % 3 holds the last page p mapped to it
    _, _, rc, rt, k_all, _ = ring_and_linear(rng, [L], page, d, ring, chunk=ring * page)
    codes, scales = oracle.quantize_tokens(k_all[0])
    last_page = (L - 1) // page
    for p in range(last_page - ring + 1, last_page + 1):
        blk = rt[0, p % ring]
        n = min(page, L - p * page)
        assert np.array_equal(rc.k_codes[blk, :n], codes[p * page:p * page + n])
        assert np.array_equal(rc.k_scale[blk, :n].view(np.uint32), scales[p * page:p * page + n].view(np.uint32))


def test_ring_rejects_keys_that_are_no_longer_resident():
    rng = np.random.default_rng(5)
    d, page, ring = 8, 16, 3
    L = 10 * page
    _, _, rc, rt, _, _ = ring_and_linear(rng, [L], page, d, ring, chunk=ring * page)
    q = synth.bf16_normal(rng, (1, 1, d))
    oracle.decode(rc, rt, [L], q, (ring - 1) * page, 1.0, ring_blocks=ring)  # resident: fine
    with pytest.raises(ValueError):
        oracle.decode(rc, rt, [L], q, ring * page + 1, 1.0, ring_blocks=ring)  # reaches an evicted page
    with pytest.raises(ValueError):
        oracle.decode(rc, rt, [L], q, 0, 1.0, ring_blocks=ring)  # global: evicted pages


def test_ring_without_wrap_is_the_full_table():
    """Before the ring wraps (L <= R * page) every page is resident and the ring
    cache is an ordinary paged cache: global attention agrees too."""
    rng = np.random.default_rng(6)
    d, page, ring = 8, 16, 5
    lens = [1, 17, 5 * 16]
    lin, lt, rc, rt, _, _ = ring_and_linear(rng, lens, page, d, ring, chunk=ring * page)
    q = synth.bf16_normal(rng, (3, 2, d))
    for W in (0, 7, 30):
        a, _ = oracle.decode(lin, lt, lens, q, W, 0.5)
        b, _ = oracle.decode(rc, rt, lens, q, W, 0.5, ring_blocks=ring)
        assert np.array_equal(a, b)


def test_ring_append_rejects_chunks_longer_than_the_ring():
    rng = np.random.default_rng(7)
    d, page, ring = 8, 16, 2
    c = oracle.Cache.empty(4, page, d)
    table = np.array([[0, 1]], np.int32)
    n = ring * page + 1
    with pytest.raises(ValueError):
        oracle.quant_append(c, table, [n], synth.cu_from_counts([n]), synth.bf16_normal(rng, (n, d)),
                            synth.bf16_normal(rng, (n, d)), ring_blocks=ring)
