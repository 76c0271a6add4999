"""GPU test of the host prefix cache: pages offloaded from device caches into
the pinned pool and uploaded back into other blocks are bit-identical, and a
prefill that starts from an uploaded prefix (the step the cache saves) matches
the oracle computed over the whole sequence."""
import numpy as np
import pytest
import torch

import oracle
import synth
import mqa_decode_attention_kv_gb300 as mk
from gpu_common import assert_close, sm_scale, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


def fill_caches(rng, caches, table, lens, d):
    """kv_quant_append of random bf16 K/V rows for every sequence, into every
    cache; returns the bf16 rows per cache."""
    cu = synth.cu_from_counts(lens)
    T = int(cu[-1])
    batch = mk.Batch.from_host(table, lens)
    rows = []
    for gc in caches:
        k = synth.bf16_normal(rng, (T, d))
        v = synth.bf16_normal(rng, (T, d))
        mk.kv_quant_append(gc, batch, to_dev_i32(cu), T, to_dev_bf16(k), to_dev_bf16(v))
        rows.append((k, v))
    return rows


@pytest.mark.parametrize("page,d,heads", [(64, 128, 32), (16, 64, 8)])
def test_offload_upload_roundtrip_and_prefill_after_upload(page, d, heads):
    rng = np.random.default_rng(page + d)
    num_caches, num_blocks = 2, 64
    caches = [mk.KVCache.empty(num_blocks, page, d) for _ in range(num_caches)]
    # conversation A: 5 whole pages plus a partial one, in blocks 10..15 (shuffled)
    n_a = 5 * page + page // 2
    table_a = np.array([[13, 10, 15, 11, 14, 12]], np.int32)
    rows_a = fill_caches(rng, caches, table_a, np.array([n_a], np.int32), d)
    tokens_a = rng.integers(0, 30000, n_a).astype(np.int32)

    pc = mk.PrefixCache(page, d, num_caches, host_pages=32)
    idx, slots = pc.insert(tokens_a)
    assert idx.tolist() == [0, 1, 2, 3, 4]
    pc.offload(caches, table_a[0, idx], slots)

    # request B: A's first 4 pages (and 7 tokens of page 4), then its own tokens
    n_keep = 4 * page + 7
    n_new = 2 * page + 3
    tokens_b = np.concatenate([tokens_a[:n_keep], rng.integers(30000, 40000, n_new).astype(np.int32)])
    hit = pc.match(tokens_b)
    assert hit.tolist() == slots[:4].tolist()
    # upload the hit into fresh blocks 40.. and check the bytes
    blocks_b = np.array([40, 47, 43, 41, 50, 52, 45], np.int32)
    pc.upload(caches, hit, blocks_b[:4])
    torch.cuda.synchronize()
    for gc in caches:
        for name in ("k_codes", "v_codes", "k_scale", "v_scale"):
            t = getattr(gc, name)
            src = t[torch.from_numpy(table_a[0, :4].astype(np.int64)).cuda()]
            dst = t[torch.from_numpy(blocks_b[:4].astype(np.int64)).cuda()]
            assert torch.equal(src.view(torch.int8) if src.dtype != torch.int8 else src,
                               dst.view(torch.int8) if dst.dtype != torch.int8 else dst), name
    st = pc.stats()
    assert st["cached_pages"] == 5 and st["pages_matched"] == 4

    # prefill of B's tokens after the hit: append them, attend them over the uploaded prefix
    L_b = len(tokens_b)
    q_len = L_b - 4 * page
    table_b = blocks_b[None, :]
    batch_b = mk.Batch.from_host(table_b, np.array([L_b], np.int32))
    cu_q = synth.cu_from_counts([q_len])
    kv_new = []
    for gc in caches:
        k = synth.bf16_normal(rng, (q_len, d))
        v = synth.bf16_normal(rng, (q_len, d))
        mk.kv_quant_append(gc, batch_b, to_dev_i32(cu_q), q_len, to_dev_bf16(k), to_dev_bf16(v))
        kv_new.append((k, v))
    q = synth.bf16_normal(rng, (q_len, heads, d))
    for c in range(num_caches):
        out = mk.mqa_prefill_attn(caches, [0, 1], c, 0, batch_b, to_dev_i32(cu_q), to_dev_bf16(q), q_len,
                                  sm_scale=sm_scale(d))
        torch.cuda.synchronize()
        # the oracle: B's whole sequence = A's first 4 pages of rows, then the new rows
        ka, va = rows_a[c]
        kb = np.concatenate([ka[:4 * page], kv_new[c][0]])
        vb = np.concatenate([va[:4 * page], kv_new[c][1]])
        oc = oracle.Cache.empty(len(blocks_b), page, d)
        otab = np.arange(len(blocks_b), dtype=np.int32)[None, :]
        oracle.quant_append(oc, otab, [L_b], synth.cu_from_counts([L_b]), kb, vb)
        rs, rp = oracle.prefill_rows(cu_q, [L_b])
        ref, _ = oracle.attention(oc, otab, [L_b], q, rs, rp, 0, sm_scale(d))
        assert_close(out, ref, f"prefill after upload, cache {c}")
    pc.close()


def test_upload_rejects_bad_indices():
    caches = [mk.KVCache.empty(8, 64, 128)]
    pc = mk.PrefixCache(64, 128, 1, host_pages=4)
    with pytest.raises(mk.MQAError):
        pc.upload(caches, [4], [0])          # slot outside the pool
    with pytest.raises(mk.MQAError):
        pc.upload(caches, [0], [8])          # block outside the cache
    with pytest.raises(mk.MQAError):
        pc.upload(caches + caches, [0], [0])  # the pool holds one cache per page
    pc.close()
