"""GPU parity of chunked causal prefill over prefix-shared int8 caches."""
import numpy as np
import pytest
import torch

import oracle
import synth
import mqa_decode_attention_kv_gb300 as mk
from gpu_common import assert_close, build_caches, caches_equal, sm_scale, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu


def build_prefix_setup(rng, groups, per, prefix, new_counts, page, d, heads):
    """Prefix blocks shared inside each group, written once through the group's
    first sequence; then every sequence appends its own new tokens."""
    new_counts = np.asarray(new_counts, np.int64)
    max_new = int(new_counts.max())
    pbs = synth.make_prefix_shared_batch(rng, groups, per, prefix, max_new, page)
    B = groups * per
    seq_lens = (prefix + new_counts).astype(np.int32)
    gc = mk.KVCache.empty(pbs.num_blocks, page, d)
    oc = oracle.Cache.empty(pbs.num_blocks, page, d)
    # 1) shared prefixes
    leaders = np.arange(groups) * per
    lead_table = np.ascontiguousarray(pbs.block_table[leaders])
    lead_lens = np.full(groups, prefix, np.int32)
    cu_p = synth.cu_from_counts(lead_lens)
    kp = synth.bf16_normal(rng, (int(cu_p[-1]), d))
    vp = synth.bf16_normal(rng, (int(cu_p[-1]), d))
    lead_batch = mk.Batch.from_host(lead_table, lead_lens)
    mk.kv_quant_append(gc, lead_batch, to_dev_i32(cu_p), int(cu_p[-1]), to_dev_bf16(kp), to_dev_bf16(vp))
    oracle.quant_append(oc, lead_table, lead_lens, cu_p, kp, vp)
    # 2) new tokens of every sequence
    batch = mk.Batch.from_host(pbs.block_table, seq_lens)
    cu_q = synth.cu_from_counts(new_counts)
    T = int(cu_q[-1])
    kn = synth.bf16_normal(rng, (T, d))
    vn = synth.bf16_normal(rng, (T, d))
    cu_dev = to_dev_i32(cu_q)
    mk.kv_quant_append(gc, batch, cu_dev, T, to_dev_bf16(kn), to_dev_bf16(vn))
    oracle.quant_append(oc, pbs.block_table, seq_lens, cu_q, kn, vn)
    q = synth.bf16_normal(rng, (T, heads, d))
    torch.cuda.synchronize()
    return dict(pbs=pbs, seq_lens=seq_lens, gc=gc, oc=oc, batch=batch, cu_q=cu_q, cu_dev=cu_dev, q=q,
                max_new=max_new, d=d)


def run(st, window, rows=None):
    out = mk.mqa_prefill_attn([st["gc"]], [0], 0, window, st["batch"], st["cu_dev"], to_dev_bf16(st["q"]),
                              st["max_new"], sm_scale=sm_scale(st["d"]))
    torch.cuda.synchronize()
    rs, rp = oracle.prefill_rows(st["cu_q"], st["seq_lens"])
    if rows is not None:
        rs, rp = rs[rows], rp[rows]
    q = st["q"] if rows is None else np.ascontiguousarray(st["q"][rows])
    ref, _ = oracle.attention(st["oc"], st["pbs"].block_table, st["seq_lens"], q, rs, rp, window,
                              sm_scale(st["d"]))
    got = out if rows is None else out[torch.from_numpy(rows).cuda()]
    return got, ref


@pytest.mark.parametrize("heads,d,page", [(32, 128, 64), (8, 64, 16), (16, 128, 16), (64, 128, 64), (8, 128, 64)])
def test_prefill_prefix_shared_ragged(heads, d, page):
    rng = np.random.default_rng(heads + d + page)
    counts = [100, 37, 64, 1, 129, 65]
    st = build_prefix_setup(rng, 3, 2, 256, counts, page, d, heads)
    assert caches_equal(st["gc"], st["oc"])
    for window in (0, 1, 50, 300):
        got, ref = run(st, window)
        assert_close(got, ref, f"prefill H={heads} d={d} P={page} W={window}")


def test_prefill_prefix_reuse_full_size_sampled():
    """32 groups x 8 sequences sharing 8192-token prefixes, 512 new tokens each,
    32 heads, d=128, page 64; local (1024) and global; sampled query rows."""
    w = synth.CONFIGS["prefix_prefill"]
    rng = np.random.default_rng(w.seed)
    prefix, new = w.len_values
    st = build_prefix_setup(rng, w.groups, w.batch // w.groups, prefix, [new] * w.batch, w.page_size,
                            w.head_dim, w.num_q_heads)
    T = int(st["cu_q"][-1])
    rows = np.unique(np.concatenate([np.arange(0, new, 37), T - 1 - np.arange(0, new, 41),
                                     synth.sample_rows(rng, T, 24)]))
    for window in w.windows:
        got, ref = run(st, window, rows)
        assert_close(got, ref, f"prefix_prefill W={window}")


@pytest.mark.parametrize("num_decode,chunks", [(36, [64, 200, 1, 513]), (600, [3, 130])])
def test_mixed_decode_rows_and_prefill_chunks_one_launch(num_decode, chunks):
    """Continuous batching (LLM-inference workshop transcript, 01:03:27-01:04:33):
    one mqa_prefill_attn launch over sequences that decode one token (q_len = 1)
    next to sequences that prefill a chunk; every row against the oracle, the
    decode rows also against the decode kernel.  600 sequences take the tile
    scan over more than one pass of the CTA."""
    rng = np.random.default_rng(num_decode)
    H, d, page = 32, 128, 64
    dec_lens = rng.integers(1, 700 if num_decode < 100 else 200, num_decode)
    ch_q = np.asarray(chunks, np.int64)
    ch_lens = ch_q + rng.integers(0, 300, len(chunks))
    lens = np.concatenate([dec_lens, ch_lens]).astype(np.int32)
    q_lens = np.concatenate([np.ones(num_decode, np.int64), ch_q])
    order = rng.permutation(len(lens))  # decode rows and chunks interleaved in the batch
    lens, q_lens = lens[order], q_lens[order]
    st = build_caches(rng, lens, page, d, 1)
    cu_q = synth.cu_from_counts(q_lens)
    T = int(cu_q[-1])
    q_bits = synth.bf16_normal(rng, (T, H, d))
    q_dev = to_dev_bf16(q_bits)
    for window in (0, 100, 1024):
        out = mk.mqa_prefill_attn(st.gpu_caches, [0], 0, window, st.batch, to_dev_i32(cu_q), q_dev,
                                  int(q_lens.max()), sm_scale=sm_scale(d))
        torch.cuda.synchronize()
        rs, rp = oracle.prefill_rows(cu_q, lens)
        ref, _ = oracle.attention(st.ora_caches[0], st.pb.block_table, lens, q_bits, rs, rp, window, sm_scale(d))
        assert_close(out, ref, f"mixed batch W={window}")
        # the decode rows through the decode kernel agree with the same rows of the mixed launch
        dec = np.nonzero(q_lens == 1)[0]
        rows = torch.from_numpy(cu_q[dec].astype(np.int64)).cuda()
        qd = torch.zeros((len(lens), H, d), dtype=torch.bfloat16, device="cuda")
        qd[torch.from_numpy(dec).cuda()] = q_dev[rows]
        od = mk.mqa_decode_attn(st.gpu_caches, [0], 0, window, st.batch, qd, sm_scale=sm_scale(d))
        torch.cuda.synchronize()
        assert_close(od[torch.from_numpy(dec).cuda()], ref[cu_q[dec]], f"decode kernel rows W={window}")


def _prefill_vs_oracle(st, lens, q_lens, q_bits, window, d):
    cu_q = synth.cu_from_counts(q_lens)
    out = mk.mqa_prefill_attn(st.gpu_caches, [0], 0, window, st.batch, to_dev_i32(cu_q), to_dev_bf16(q_bits),
                              int(np.max(q_lens)), sm_scale=sm_scale(d))
    torch.cuda.synchronize()
    rs, rp = oracle.prefill_rows(cu_q, lens)
    ref, _ = oracle.attention(st.ora_caches[0], st.pb.block_table, lens, q_bits, rs, rp, window, sm_scale(d))
    return out, ref


@pytest.mark.parametrize("d", [128, 64])
def test_prefill_large_magnitudes_stay_finite(d):
    """V scales far above fp16's range, tiny queries, and V magnitudes that grow
    along the sequence (the power-of-two bound of the V scales moves block after
    block): every intermediate stays finite and the rows match the oracle."""
    rng = np.random.default_rng(51 + d)
    page, H = 64, 32 if d == 128 else 8
    lens = np.array([700, 1500, 130], np.int32)
    q_lens = np.array([300, 129, 130], np.int64)
    T = int(lens.sum())
    k = rng.standard_normal((T, d), dtype=np.float32) * np.float32(3e5)
    growth = np.exp(np.linspace(0.0, 12.0, T, dtype=np.float32))[:, None]
    v = rng.standard_normal((T, d), dtype=np.float32) * np.float32(3e5) * growth
    st = build_caches(rng, lens, page, d, 1, kv_bits=[(synth.f32_to_bf16_bits(k), synth.f32_to_bf16_bits(v))])
    q = synth.bf16_normal(rng, (int(q_lens.sum()), H, d), 1e-5)
    for window in (0, 256):
        out, ref = _prefill_vs_oracle(st, lens, q_lens, q, window, d)
        g = out.float().cpu().numpy()
        assert np.all(np.isfinite(g))
        scale = np.abs(ref).max()
        rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
        assert rel <= 5e-3 and np.abs(g - ref).max() <= 1e-2 * scale, (window, rel)


@pytest.mark.parametrize("k_offset", [1.0, 30.0])
def test_prefill_one_signed_queries_and_skewed_keys(k_offset):
    """Queries of one sign and keys whose codes sit near one end of the int8
    range: the K images carry their codes' exponent bias, which the softmax
    takes off in fp32, so this is where that correction is largest."""
    rng = np.random.default_rng(61)
    d, page, H = 128, 64, 32
    lens = np.array([1, 129, 1500, 700], np.int32)
    q_lens = np.array([1, 129, 200, 64], np.int64)
    T = int(lens.sum())
    k = rng.standard_normal((T, d), dtype=np.float32) * np.float32(0.1 * k_offset) + np.float32(k_offset)
    v = rng.standard_normal((T, d), dtype=np.float32)
    st = build_caches(rng, lens, page, d, 1, kv_bits=[(synth.f32_to_bf16_bits(k), synth.f32_to_bf16_bits(v))])
    for sign in (1.0, -1.0):
        qf = (np.abs(rng.standard_normal((int(q_lens.sum()), H, d), dtype=np.float32)) + np.float32(0.5)) * \
            np.float32(sign * 2.0)
        q = synth.f32_to_bf16_bits(qf)
        for window in (0, 1024):
            out, ref = _prefill_vs_oracle(st, lens, q_lens, q, window, d)
            assert_close(out, ref, f"prefill one-signed q sign {sign} window {window} k_offset {k_offset}")
