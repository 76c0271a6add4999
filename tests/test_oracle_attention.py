"""Pins for the oracle's attention and split-combine (CPU only).

Each pin checks the oracle against something other than itself: closed forms,
torch's fp64 scaled_dot_product_attention on a dense layout with K/V repeated
per head (MQA = MHA with shared K/V), a dense brute-force loop, and
invariants of the method (window semantics, cache sharing, paging, prefix
sharing, split partitions).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import (bf16_bits_to_f32, bf16_normal, cu_from_counts, f32_to_bf16_bits,
                   make_paged_batch, make_prefix_shared_batch)


def build_cache(rng, seq_lens, d, P, shuffle=True, pb=None, kv=None):
    pb = pb or make_paged_batch(rng, seq_lens, P, shuffle=shuffle)
    cache = oracle.Cache.empty(pb.num_blocks, P, d)
    cu = cu_from_counts(pb.seq_lens)
    if kv is None:
        k = bf16_normal(rng, (int(cu[-1]), d))
        v = bf16_normal(rng, (int(cu[-1]), d))
    else:
        k, v = kv
    oracle.quant_append(cache, pb.block_table, pb.seq_lens, cu, k, v)
    return cache, pb, (k, v)


def dense_kv(cache, pb, b):
    """Dequantised K^/V^ of sequence b as dense fp64 [L, d]."""
    L = int(pb.seq_lens[b])
    P = cache.page_size
    idx = [(pb.block_table[b, j // P], j % P) for j in range(L)]
    kc = np.stack([cache.k_codes[i, o] for i, o in idx]).astype(np.float64)
    vc = np.stack([cache.v_codes[i, o] for i, o in idx]).astype(np.float64)
    ks = np.array([cache.k_scale[i, o] for i, o in idx], np.float64)
    vs = np.array([cache.v_scale[i, o] for i, o in idx], np.float64)
    return kc * ks[:, None], vc * vs[:, None]


def qf64(q):
    return bf16_bits_to_f32(q).astype(np.float64)


@pytest.mark.parametrize("window", [0, 1, 7, 32])
def test_matches_torch_sdpa_fp64(window):
    rng = np.random.default_rng(11 + window)
    d, P, H = 16, 4, 4
    seq_lens = np.array([1, 9, 23, 40], np.int32)
    cache, pb, _ = build_cache(rng, seq_lens, d, P)
    # prefill-style rows: the last 5 positions of each sequence (or fewer)
    qlen = np.minimum(seq_lens, 5)
    cu_q = cu_from_counts(qlen)
    q = bf16_normal(rng, (int(cu_q[-1]), H, d))
    rs, rp = oracle.prefill_rows(cu_q, seq_lens)
    scale = 1.0 / math.sqrt(d)
    out, lse = oracle.attention(cache, pb.block_table, seq_lens, q, rs, rp, window, scale)
    for b in range(len(seq_lens)):
        K, V = dense_kv(cache, pb, b)
        L = K.shape[0]
        rows = np.arange(cu_q[b], cu_q[b + 1])
        pos = rp[rows]
        j = np.arange(L)
        allow = (j[None, :] <= pos[:, None])
        if window > 0:
            allow &= j[None, :] > pos[:, None] - window
        Q = torch.from_numpy(qf64(q[rows])).permute(1, 0, 2)            # [H, n, d]
        Kt = torch.from_numpy(K)[None].expand(H, L, d)                    # MQA: K repeated per head
        Vt = torch.from_numpy(V)[None].expand(H, L, d)
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, Kt, Vt, attn_mask=torch.from_numpy(allow)[None], scale=scale)
        np.testing.assert_allclose(out[rows], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
        # lse against torch.logsumexp of the masked scores
        S = torch.einsum("hnd,hld->hnl", Q, Kt) * scale
        S = S.masked_fill(~torch.from_numpy(allow)[None], -math.inf)
        np.testing.assert_allclose(lse[rows], torch.logsumexp(S, -1).T.numpy(), rtol=0, atol=1e-12)


def test_matches_dense_brute_force_loop():
    rng = np.random.default_rng(12)
    d, P, H, W = 8, 4, 3, 6
    seq_lens = np.array([13, 40], np.int32)
    cache, pb, _ = build_cache(rng, seq_lens, d, P)
    q = bf16_normal(rng, (2, H, d))
    out, lse = oracle.decode(cache, pb.block_table, seq_lens, q, W, 0.3)
    for b in range(2):
        K, V = dense_kv(cache, pb, b)
        i = seq_lens[b] - 1
        for h in range(H):
            js = [j for j in range(i + 1) if j > i - W]
            sc = [0.3 * sum(qf64(q)[b, h, k] * K[j, k] for k in range(d)) for j in js]
            mx = max(sc)
            w = [math.exp(s - mx) for s in sc]
            den = sum(w)
            ref = [sum(w[a] * V[js[a], k] for a in range(len(js))) / den for k in range(d)]
            assert np.allclose(out[b, h], ref, rtol=0, atol=1e-13)
            assert abs(lse[b, h] - (mx + math.log(den))) < 1e-13


def test_single_key_returns_its_value():
    rng = np.random.default_rng(13)
    cache, pb, _ = build_cache(rng, np.array([1, 1], np.int32), 64, 16)
    q = bf16_normal(rng, (2, 8, 64))
    out, lse = oracle.decode(cache, pb.block_table, pb.seq_lens, q, 0, 0.125)
    for b in range(2):
        K, V = dense_kv(cache, pb, b)
        assert np.array_equal(out[b], np.broadcast_to(V[0], out[b].shape))
        np.testing.assert_allclose(lse[b], 0.125 * (qf64(q)[b] @ K[0]), rtol=0, atol=1e-13)


@pytest.mark.parametrize("window", [0, 5])
def test_zero_query_gives_window_mean(window):
    rng = np.random.default_rng(14)
    seq_lens = np.array([12, 30], np.int32)
    cache, pb, _ = build_cache(rng, seq_lens, 32, 4)
    q = np.zeros((2, 2, 32), np.uint16)
    out, lse = oracle.decode(cache, pb.block_table, seq_lens, q, window, 0.2)
    for b in range(2):
        _, V = dense_kv(cache, pb, b)
        L = seq_lens[b]
        lo = max(0, L - window) if window else 0
        np.testing.assert_allclose(out[b, 0], V[lo:L].mean(0), rtol=0, atol=1e-13)
        assert abs(lse[b, 0] - math.log(L - lo)) < 1e-13


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(15)
    d, L = 16, 20
    k = bf16_normal(rng, (L, d), scale=0.01)
    v = bf16_normal(rng, (L, d))
    k[7] = f32_to_bf16_bits(np.full(d, 8.0, np.float32))  # <q,k_7> = 8*8*16 = 1024 vs ~0
    cache, pb, _ = build_cache(rng, np.array([L], np.int32), d, 4, kv=(k, v))
    q = f32_to_bf16_bits(np.full((1, 1, d), 8.0, np.float32))
    out, _ = oracle.decode(cache, pb.block_table, pb.seq_lens, q, 0, 1.0 / 16)
    _, V = dense_kv(cache, pb, 0)
    np.testing.assert_allclose(out[0, 0], V[7], rtol=0, atol=1e-12)


def test_softmax_rows_sum_to_one_and_respect_window():
    rng = np.random.default_rng(16)
    seq_lens = np.array([50, 3, 17], np.int32)
    cache, pb, _ = build_cache(rng, seq_lens, 16, 4)
    q = bf16_normal(rng, (3, 4, 16), scale=4.0)
    W = 10
    out, lse, probs = oracle.attention(cache, pb.block_table, seq_lens, q, np.arange(3),
                                       seq_lens - 1, W, 0.5, want_probs=True)
    assert np.all(probs >= 0)
    np.testing.assert_allclose(probs.sum(-1), 1.0, rtol=0, atol=1e-12)
    for b in range(3):
        i = seq_lens[b] - 1
        outside = [j for j in range(probs.shape[-1]) if not (i - W < j <= i)]
        assert np.all(probs[b][:, outside] == 0)


def test_local_equals_global_when_context_fits_window():
    rng = np.random.default_rng(17)
    seq_lens = np.array([100, 128, 7], np.int32)
    cache, pb, _ = build_cache(rng, seq_lens, 64, 16)
    q = bf16_normal(rng, (3, 8, 64))
    g = oracle.decode(cache, pb.block_table, seq_lens, q, 0, 0.125)
    l = oracle.decode(cache, pb.block_table, seq_lens, q, 128, 0.125)
    assert np.array_equal(g[0], l[0]) and np.array_equal(g[1], l[1])
    l2 = oracle.decode(cache, pb.block_table, seq_lens, q, 127, 0.125)
    assert not np.array_equal(g[0][1], l2[0][1])  # 128 keys, window 127: differs


def test_mqa_equals_mha_with_repeated_kv():
    """MQA over one K/V head equals per-head attention where each head is given its
    own copy of that K/V head (the heads then share nothing but the data)."""
    rng = np.random.default_rng(18)
    seq_lens = np.array([33, 8], np.int32)
    cache, pb, _ = build_cache(rng, seq_lens, 32, 8)
    H = 4
    q = bf16_normal(rng, (2, H, 32))
    mqa_out, mqa_lse = oracle.decode(cache, pb.block_table, seq_lens, q, 0, 0.17)
    for h in range(H):
        head_cache = oracle.Cache(cache.k_codes.copy(), cache.v_codes.copy(),
                                  cache.k_scale.copy(), cache.v_scale.copy())
        o, l = oracle.decode(head_cache, pb.block_table, seq_lens,
                             np.ascontiguousarray(q[:, h:h + 1]), 0, 0.17)
        assert np.array_equal(o[:, 0], mqa_out[:, h]) and np.array_equal(l[:, 0], mqa_lse[:, h])


def test_shared_cache_map_equals_duplicated_caches():
    """Two layers reading one cache through the layer->cache map give the same
    results as two layers reading two identical caches."""
    rng = np.random.default_rng(19)
    seq_lens = np.array([70, 20], np.int32)
    cache, pb, _ = build_cache(rng, seq_lens, 64, 16)
    dup = oracle.Cache(cache.k_codes.copy(), cache.v_codes.copy(), cache.k_scale.copy(),
                       cache.v_scale.copy())
    q = [bf16_normal(rng, (2, 8, 64)) for _ in range(2)]
    windows = [16, 0]
    shared = [oracle.decode([cache, dup][m], pb.block_table, seq_lens, q[l], windows[l], 0.125)
              for l, m in enumerate([0, 0])]
    separate = [oracle.decode([cache, dup][m], pb.block_table, seq_lens, q[l], windows[l], 0.125)
                for l, m in enumerate([0, 1])]
    for a, b in zip(shared, separate):
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_shuffled_block_table_equals_identity():
    rng = np.random.default_rng(20)
    seq_lens = np.array([45, 64, 3], np.int32)
    d, P = 32, 16
    k = bf16_normal(rng, (int(seq_lens.sum()), d))
    v = bf16_normal(rng, (int(seq_lens.sum()), d))
    c1, pb1, _ = build_cache(rng, seq_lens, d, P, shuffle=False, kv=(k, v))
    c2, pb2, _ = build_cache(rng, seq_lens, d, P, shuffle=True, kv=(k, v))
    assert not np.array_equal(pb1.block_table, pb2.block_table)
    q = bf16_normal(rng, (3, 8, d))
    for W in (0, 20):
        a = oracle.decode(c1, pb1.block_table, seq_lens, q, W, 0.2)
        b = oracle.decode(c2, pb2.block_table, seq_lens, q, W, 0.2)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_prefix_shared_blocks_equal_private_copies():
    rng = np.random.default_rng(21)
    d, P, H = 32, 16, 4
    groups, per, prefix, new = 2, 3, 32, 10
    pbs = make_prefix_shared_batch(rng, groups, per, prefix, new, P)
    cache = oracle.Cache.empty(pbs.num_blocks, P, d)
    # write each group's prefix once (through its first sequence), then each tail
    pre_k = [bf16_normal(rng, (prefix, d)) for _ in range(groups)]
    pre_v = [bf16_normal(rng, (prefix, d)) for _ in range(groups)]
    firsts = np.arange(groups) * per
    oracle.quant_append(cache, pbs.block_table[firsts], np.full(groups, prefix, np.int32),
                        cu_from_counts([prefix] * groups), np.concatenate(pre_k), np.concatenate(pre_v))
    tail_k = bf16_normal(rng, (groups * per * new, d))
    tail_v = bf16_normal(rng, (groups * per * new, d))
    oracle.quant_append(cache, pbs.block_table, pbs.seq_lens, cu_from_counts([new] * groups * per),
                        tail_k, tail_v)
    # private layout: every sequence owns a copy of its prefix
    full_k = np.concatenate([np.concatenate([pre_k[b // per], tail_k[b * new:(b + 1) * new]])
                             for b in range(groups * per)])
    full_v = np.concatenate([np.concatenate([pre_v[b // per], tail_v[b * new:(b + 1) * new]])
                             for b in range(groups * per)])
    priv, pbp, _ = build_cache(rng, pbs.seq_lens, d, P, kv=(full_k, full_v))
    cu_q = cu_from_counts([new] * groups * per)
    q = bf16_normal(rng, (int(cu_q[-1]), H, d))
    rs, rp = oracle.prefill_rows(cu_q, pbs.seq_lens)
    for W in (0, 12):
        a = oracle.attention(cache, pbs.block_table, pbs.seq_lens, q, rs, rp, W, 0.2)
        b = oracle.attention(priv, pbp.block_table, pbp.seq_lens, q, rs, rp, W, 0.2)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("window", [0, 19])
def test_split_partition_then_combine_equals_unsplit(window):
    rng = np.random.default_rng(22 + window)
    seq_lens = np.array([77, 31, 5], np.int32)
    cache, pb, _ = build_cache(rng, seq_lens, 16, 8)
    H, d = 4, 16
    q = bf16_normal(rng, (3, H, d), scale=2.0)
    full, full_lse = oracle.decode(cache, pb.block_table, seq_lens, q, window, 0.3)
    for b in range(3):
        L = int(seq_lens[b])
        cuts = np.sort(rng.choice(np.arange(1, L + 1), size=min(4, L), replace=False))
        edges = [0] + [int(c) for c in cuts if c < L] + [L, L]  # includes an empty part
        parts, lses = [], []
        for s in range(len(edges) - 1):
            o, l = oracle.attention(cache, pb.block_table, seq_lens, q[b:b + 1], np.array([b]),
                                    np.array([L - 1]), window, 0.3, key_range=(edges[s], edges[s + 1]))
            parts.append(o.reshape(H, d))
            lses.append(l.reshape(H))
        o, l = oracle.combine(np.stack(parts), np.stack(lses))
        np.testing.assert_allclose(o, full[b], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, full_lse[b], rtol=0, atol=1e-12)


def test_combine_of_all_empty_parts_is_zero():
    parts = np.ones((3, 2, 4))
    lse = np.full((3, 2), -np.inf)
    o, l = oracle.combine(parts, lse)
    assert np.all(o == 0) and np.all(np.isneginf(l))


def test_combine_closed_form_two_parts():
    # two parts with equal lse average their outputs; lse grows by ln 2
    parts = np.stack([np.full((1, 3), 1.0), np.full((1, 3), 3.0)])
    lse = np.array([[0.7], [0.7]])
    o, l = oracle.combine(parts, lse)
    np.testing.assert_allclose(o, 2.0, atol=1e-15)
    np.testing.assert_allclose(l, 0.7 + math.log(2), atol=1e-15)
