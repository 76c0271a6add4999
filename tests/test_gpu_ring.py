"""GPU parity of window-bounded (ring) caches for local layers.

A local layer attends over a window of W keys ("Character.AI inference
article", secret 1), so its cache need keep only the pages such a window can
reach: with ring_blocks = R, page p of a sequence lives in block-table entry
p % R.  The tests append whole histories into ring caches chunk by chunk
(kv_quant_append), then check
  * the ring cache bytes against the oracle's ring append, bit for bit;
  * decode and chunked-prefill attention over the ring against the oracle
    (which reads the ring through the same addressing) and, bit for bit,
    against the same kernels over an ordinary paged cache holding every token
    (the ring only changes which block a page is fetched from);
  * the device-side rejection of an append chunk longer than the ring.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import mqa_decode_attention_kv_gb300 as mk
from gpu_common import assert_close, caches_equal, sm_scale, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


def ring_setup(rng, lens, page, d, ring, max_chunk):
    """The tokens of every sequence appended into a ring cache chunk by chunk
    (GPU and oracle) and, in one call, into a linear cache (GPU)."""
    lens = np.asarray(lens, np.int32)
    B = len(lens)
    cu_all = synth.cu_from_counts(lens)
    T = int(cu_all[-1])
    k_all = synth.bf16_normal(rng, (T, d))
    v_all = synth.bf16_normal(rng, (T, d))

    # linear cache: a full table, every token
    lin_pb = synth.make_paged_batch(rng, lens, page, shuffle=True)
    lin = mk.KVCache.empty(lin_pb.num_blocks, page, d)
    lin_batch = mk.Batch.from_host(lin_pb.block_table, lens)
    mk.kv_quant_append(lin, lin_batch, to_dev_i32(cu_all), T, to_dev_bf16(k_all), to_dev_bf16(v_all))

    # ring cache: R entries per sequence, a shuffled pool of B * R blocks
    table = rng.permutation(B * ring).astype(np.int32).reshape(B, ring)
    gc = mk.KVCache.empty(B * ring, page, d)
    oc = oracle.Cache.empty(B * ring, page, d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    done = np.zeros(B, np.int32)
    while (done < lens).any():
        want = rng.integers(1, max_chunk + 1, size=B)
        n = np.minimum(lens - done, want).astype(np.int32)
        cur = done + n
        cu = synth.cu_from_counts(n)
        rows = np.concatenate([np.arange(cu_all[b] + done[b], cu_all[b] + cur[b]) for b in range(B)])
        k, v = np.ascontiguousarray(k_all[rows]), np.ascontiguousarray(v_all[rows])
        batch = mk.Batch.from_host(table, cur, ring_blocks=ring)
        mk.kv_quant_append(gc, batch, to_dev_i32(cu), int(cu[-1]), to_dev_bf16(k), to_dev_bf16(v),
                           dev_status=status)
        oracle.quant_append(oc, table, cur, cu, k, v, ring_blocks=ring)
        done = cur
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return dict(lens=lens, table=table, gc=gc, oc=oc, lin=lin, lin_pb=lin_pb, k_all=k_all, v_all=v_all)


DECODE_CASES = [
    # heads, d, page, window: 64-token and 16-token pages, two-token rows (d=64)
    # and zero-query columns (d=128 with 16 heads)
    (32, 128, 64, 1024),
    (32, 128, 16, 300),
    (8, 64, 16, 200),
    (16, 128, 64, 500),
]


@pytest.mark.parametrize("heads,d,page,window", DECODE_CASES)
def test_ring_decode(heads, d, page, window):
    rng = np.random.default_rng(heads * 7 + d + page + window)
    ring = (window - 1) // page + 2
    span = ring * page
    lens = [1, page - 1, page, span - 1, span, span + 1, 2 * span + 5, window, window + 1, 3 * window + 7,
            5 * span + page // 2]
    st = ring_setup(rng, lens, page, d, ring, max_chunk=span)
    assert caches_equal(st["gc"], st["oc"]), "ring cache bytes differ from the oracle's"
    B = len(lens)
    q_bits = synth.bf16_normal(rng, (B, heads, d))
    q = to_dev_bf16(q_bits)
    rb = mk.Batch.from_host(st["table"], st["lens"], ring_blocks=ring)
    lb = mk.Batch.from_host(st["lin_pb"].block_table, st["lens"])
    for w in (window, max(1, window // 3)):
        ref, _ = oracle.decode(st["oc"], st["table"], st["lens"], q_bits, w, sm_scale(d), ring_blocks=ring)
        for splits in (0, 1, 3):
            got = mk.mqa_decode_attn([st["gc"]], [0], 0, w, rb, q, num_splits=splits)
            lin = mk.mqa_decode_attn([st["lin"]], [0], 0, w, lb, q, num_splits=splits)
            torch.cuda.synchronize()
            assert_close(got, ref, f"ring decode H={heads} d={d} P={page} W={w} splits={splits}")
            assert torch.equal(got.view(torch.int16), lin.view(torch.int16)), \
                f"ring decode differs from the full-table decode (W={w}, splits={splits})"


def test_ring_decode_rejects_uncovered_windows():
    rng = np.random.default_rng(11)
    page, d, ring = 64, 128, 17
    st = ring_setup(rng, [3000, 70], page, d, ring, max_chunk=ring * page)
    q = to_dev_bf16(synth.bf16_normal(rng, (2, 32, d)))
    rb = mk.Batch.from_host(st["table"], st["lens"], ring_blocks=ring)
    mk.mqa_decode_attn([st["gc"]], [0], 0, (ring - 1) * page, rb, q)  # the widest resident window
    for w in ((ring - 1) * page + 1, 0):
        with pytest.raises(mk.MQAError):
            mk.mqa_decode_attn([st["gc"]], [0], 0, w, rb, q)


PREFILL_CASES = [(32, 128, 64, 1024, 200), (16, 128, 16, 256, 100), (8, 64, 16, 256, 90)]


@pytest.mark.parametrize("heads,d,page,window,qlen", PREFILL_CASES)
def test_ring_chunked_prefill(heads, d, page, window, qlen):
    """Chunked prefill of four sequences through a ring: append qlen tokens,
    attend their queries, repeat; bitwise equal to the same prefill over a
    full table, and equal to the oracle on sampled rows of every chunk."""
    rng = np.random.default_rng(heads + d + page + qlen)
    ring = (window + qlen - 2) // page + 2
    B = 4
    total = np.array([5 * qlen + 3, 3 * qlen, 2 * qlen + 1, qlen // 2 + 1], np.int32)
    cu_all = synth.cu_from_counts(total)
    T = int(cu_all[-1])
    k_all = synth.bf16_normal(rng, (T, d))
    v_all = synth.bf16_normal(rng, (T, d))
    lin_pb = synth.make_paged_batch(rng, total, page, shuffle=True)
    lin = mk.KVCache.empty(lin_pb.num_blocks, page, d)
    mk.kv_quant_append(lin, mk.Batch.from_host(lin_pb.block_table, total), to_dev_i32(cu_all), T,
                       to_dev_bf16(k_all), to_dev_bf16(v_all))
    table = rng.permutation(B * ring).astype(np.int32).reshape(B, ring)
    gc = mk.KVCache.empty(B * ring, page, d)
    oc = oracle.Cache.empty(B * ring, page, d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    done = np.zeros(B, np.int32)
    step = 0
    while (done < total).any():
        n = np.minimum(total - done, qlen).astype(np.int32)
        seqs = np.nonzero(n > 0)[0]  # sequences that finished leave the batch
        cur = done[seqs] + n[seqs]
        cu = synth.cu_from_counts(n[seqs])
        rows = np.concatenate([np.arange(cu_all[b] + done[b], cu_all[b] + done[b] + n[b]) for b in seqs])
        k, v = np.ascontiguousarray(k_all[rows]), np.ascontiguousarray(v_all[rows])
        sub_table = np.ascontiguousarray(table[seqs])
        rb = mk.Batch.from_host(sub_table, cur, ring_blocks=ring)
        cu_dev = to_dev_i32(cu)
        mk.kv_quant_append(gc, rb, cu_dev, int(cu[-1]), to_dev_bf16(k), to_dev_bf16(v), dev_status=status)
        oracle.quant_append(oc, sub_table, cur, cu, k, v, ring_blocks=ring)
        q_bits = synth.bf16_normal(rng, (int(cu[-1]), heads, d))
        q = to_dev_bf16(q_bits)
        mq = int(n[seqs].max())
        got = mk.mqa_prefill_attn([gc], [0], 0, window, rb, cu_dev, q, mq, dev_status=status)
        lb = mk.Batch.from_host(np.ascontiguousarray(lin_pb.block_table[seqs]), cur)
        ref_lin = mk.mqa_prefill_attn([lin], [0], 0, window, lb, cu_dev, q, mq)
        torch.cuda.synchronize()
        assert int(status.item()) == 0, f"device status {int(status.item()):#x}"
        assert torch.equal(got.view(torch.int16), ref_lin.view(torch.int16)), \
            f"step {step}: ring prefill differs from the full-table prefill"
        rs, rp = oracle.prefill_rows(cu, cur)
        pick = synth.sample_rows(np.random.default_rng(step), len(rs), min(len(rs), 48))
        ref, _ = oracle.attention(oc, sub_table, cur, np.ascontiguousarray(q_bits[pick]), rs[pick], rp[pick],
                                  window, sm_scale(d), ring_blocks=ring)
        assert_close(got[torch.from_numpy(np.asarray(pick, np.int64)).cuda()], ref,
                     f"ring prefill H={heads} d={d} P={page} W={window} step {step}")
        done[seqs] = cur
        step += 1
    assert caches_equal(gc, oc)


def test_ring_append_chunk_longer_than_ring_is_flagged():
    """A sequence appending more than R * page tokens in one call would
    overwrite its own new tokens: the kernel flags MQA_DEV_BAD_CU and skips
    that sequence; the others are written."""
    rng = np.random.default_rng(12)
    page, d, ring = 16, 64, 3
    counts = np.array([ring * page + 1, 5], np.int32)
    table = np.array([[0, 1, 2], [3, 4, 5]], np.int32)
    cu = synth.cu_from_counts(counts)
    k = synth.bf16_normal(rng, (int(cu[-1]), d))
    v = synth.bf16_normal(rng, (int(cu[-1]), d))
    gc = mk.KVCache.empty(6, page, d)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mk.kv_quant_append(gc, mk.Batch.from_host(table, counts, ring_blocks=ring), to_dev_i32(cu), int(cu[-1]),
                       to_dev_bf16(k), to_dev_bf16(v), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mk.MQA_DEV_BAD_CU
    assert not gc.k_codes[:3].any().item() and not gc.k_scale[:3].any().item()
    codes, scales = oracle.quantize_tokens(k[cu[1]:cu[2]])
    assert np.array_equal(gc.k_codes[3, :5].cpu().numpy(), codes)
    assert np.array_equal(gc.k_scale[3, :5].cpu().numpy().view(np.uint32), scales.view(np.uint32))
