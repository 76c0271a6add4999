"""GPU parity: kv_quant_append (bit-exact), decode attention and split-KV
combine (within the bf16 tolerances) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
import mqa_decode_attention_kv_gb300 as mk
from gpu_common import (assert_close, build_caches, caches_equal, sm_scale, to_dev_bf16, to_dev_i32)

pytestmark = pytest.mark.gpu


# ----------------------------------------------------------------- quantise + append
@pytest.mark.parametrize("d,page", [(64, 16), (128, 64), (128, 16), (64, 64)])
def test_append_full_sequences_bit_exact(d, page):
    rng = np.random.default_rng(100 + d + page)
    lens = np.array([1, 15, 16, 17, 64, 65, 300, 1000], np.int32)
    s = build_caches(rng, lens, page, d, 1, kv_scale=2.0)
    assert caches_equal(s.gpu_caches[0], s.ora_caches[0])


def test_append_decode_step_and_ties_bit_exact():
    """One token per sequence at its last position (a decode step), with rows
    that hit rounding ties, zero vectors and huge/tiny magnitudes."""
    rng = np.random.default_rng(7)
    d, page = 128, 64
    lens = np.array([5, 64, 65, 129, 700], np.int32)
    s = build_caches(rng, lens, page, d, 1)
    B = len(lens)
    k = synth.bf16_normal(rng, (B, d))
    v = synth.bf16_normal(rng, (B, d))
    # row 0: ties around a scale of exactly 1 (amax 127); row 1: zeros; rows 2/3: extreme magnitudes
    tie = np.zeros(d, np.float32)
    tie[:6] = [127.0, 2.5, 3.5, -2.5, 0.5, -126.5]
    k[0] = synth.f32_to_bf16_bits(tie)
    v[1] = 0
    k[2] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(k[2]) * np.float32(1e30))
    v[3] = synth.f32_to_bf16_bits(synth.bf16_bits_to_f32(v[3]) * np.float32(1e-30))
    cu = synth.cu_from_counts(np.ones(B))
    mk.kv_quant_append(s.gpu_caches[0], s.batch, to_dev_i32(cu), B, to_dev_bf16(k), to_dev_bf16(v))
    oracle.quant_append(s.ora_caches[0], s.pb.block_table, lens, cu, k, v)
    torch.cuda.synchronize()
    assert caches_equal(s.gpu_caches[0], s.ora_caches[0])


def test_append_ragged_chunk_with_empty_sequences():
    rng = np.random.default_rng(8)
    d, page = 64, 16
    lens = np.array([40, 3, 90, 17], np.int32)
    s = build_caches(rng, lens, page, d, 1)
    counts = np.array([7, 0, 33, 1])
    cu = synth.cu_from_counts(counts)
    T = int(cu[-1])
    k = synth.bf16_normal(rng, (T, d), 5.0)
    v = synth.bf16_normal(rng, (T, d), 0.01)
    mk.kv_quant_append(s.gpu_caches[0], s.batch, to_dev_i32(cu), T, to_dev_bf16(k), to_dev_bf16(v))
    oracle.quant_append(s.ora_caches[0], s.pb.block_table, lens, cu, k, v)
    torch.cuda.synchronize()
    assert caches_equal(s.gpu_caches[0], s.ora_caches[0])


# ----------------------------------------------------------------- decode
def run_decode(s, q_bits, window, layer_map=(0,), layer=0, num_splits=0, heads=None):
    q = to_dev_bf16(q_bits)
    out = mk.mqa_decode_attn(s.gpu_caches, list(layer_map), layer, window, s.batch, q,
                             sm_scale=sm_scale(s.head_dim), num_splits=num_splits)
    torch.cuda.synchronize()
    ref, _ = oracle.decode(s.ora_caches[layer_map[layer]], s.pb.block_table, s.seq_lens, q_bits, window,
                           sm_scale(s.head_dim))
    return out, ref


@pytest.mark.parametrize("num_splits", [1, 0, 3])
def test_decode_tiny_config(num_splits):
    """Batch 4, 8 heads, d=64, lengths {17,100,250,512}, page 16, identity table;
    layer 0 local (window 128), layer 1 global; map [0,1] and shared map [0,0]."""
    w = synth.CONFIGS["tiny"]
    rng = np.random.default_rng(w.seed)
    s = build_caches(rng, synth.seq_lens_for(w, rng), w.page_size, w.head_dim, w.num_caches, shuffle=False)
    for layer_map in ((0, 1), (0, 0)):
        for layer, window in enumerate(w.windows):
            q = synth.bf16_normal(rng, (w.batch, w.num_q_heads, w.head_dim))
            out, ref = run_decode(s, q, window, layer_map, layer, num_splits)
            assert_close(out, ref, f"tiny layer {layer} map {layer_map} splits {num_splits}")


@pytest.mark.parametrize("heads", [8, 16, 32, 64])
@pytest.mark.parametrize("d,page", [(128, 64), (64, 16), (128, 16)])
def test_decode_shapes_and_edges(heads, d, page):
    rng = np.random.default_rng(heads * 7 + d + page)
    # edge lengths: 1 token, page/tile boundaries, ragged tails
    lens = np.array([1, 2, 63, 64, 65, 127, 128, 129, 1000, 1500], np.int32)
    s = build_caches(rng, lens, page, d, 1)
    for window in (0, 1, 100, 1024):
        q_bits = synth.bf16_normal(rng, (len(lens), heads, d))
        ref, _ = oracle.decode(s.ora_caches[0], s.pb.block_table, s.seq_lens, q_bits, window, sm_scale(d))
        q = to_dev_bf16(q_bits)
        for splits in (1, 0, 4):
            out = mk.mqa_decode_attn(s.gpu_caches, [0], 0, window, s.batch, q, sm_scale=sm_scale(d),
                                     num_splits=splits)
            torch.cuda.synchronize()
            assert_close(out, ref, f"H={heads} d={d} P={page} W={window} S={splits}")


def test_decode_local_b64_full_size():
    """Single local layer: batch 64, 32 heads, d=128, ragged 1k-8k, window 1024,
    page 64, shuffled block table (the full workload)."""
    w = synth.CONFIGS["local_b64"]
    rng = np.random.default_rng(w.seed)
    s = build_caches(rng, synth.seq_lens_for(w, rng), w.page_size, w.head_dim, 1)
    assert caches_equal(s.gpu_caches[0], s.ora_caches[0])
    q = synth.bf16_normal(rng, (w.batch, w.num_q_heads, w.head_dim))
    for splits in (0, 1):
        out, ref = run_decode(s, q, w.windows[0], num_splits=splits)
        assert_close(out, ref, f"local_b64 splits={splits}")


def test_decode_global_long_full_size():
    """Single global layer, long context: batch 8, 32 heads, d=128,
    32k-128k tokens, page 64, split-KV with combine (the full workload)."""
    w = synth.CONFIGS["global_long_b8"]
    rng = np.random.default_rng(w.seed)
    s = build_caches(rng, synth.seq_lens_for(w, rng), w.page_size, w.head_dim, 1)
    q = synth.bf16_normal(rng, (w.batch, w.num_q_heads, w.head_dim))
    splits = mk.mqa_decode_auto_splits(s.batch, 0, w.num_q_heads, w.head_dim, w.page_size)
    assert splits > 1
    out, ref = run_decode(s, q, 0, num_splits=0)
    assert_close(out, ref, f"global_long splits={splits}")


def test_decode_large_magnitudes_stay_finite():
    """V scales far above fp16's range and tiny K scales: the power-of-two
    rescaling of P' keeps every intermediate finite."""
    rng = np.random.default_rng(31)
    d, page = 128, 64
    lens = np.array([300, 2000, 77], np.int32)
    s = build_caches(rng, lens, page, d, 1, kv_scale=3e5)
    q = synth.bf16_normal(rng, (3, 32, d), 1e-3)
    out, ref = run_decode(s, q, 0, num_splits=0)
    scale = np.abs(ref).max()
    g = out.float().cpu().numpy()
    assert np.all(np.isfinite(g))
    rel = np.linalg.norm(g - ref) / np.linalg.norm(ref)
    assert rel <= 5e-3 and np.abs(g - ref).max() <= 1e-2 * scale


@pytest.mark.parametrize("k_offset", [1.0, 30.0])
def test_decode_one_signed_queries_and_skewed_keys(k_offset):
    """Queries whose 128 entries all share one sign and keys whose codes sit near
    one end of the int8 range (a common offset ten times their spread): sum_d
    Q[h][d] is as large as it gets, so the K conversion's bias (1152 per code,
    taken off the scores in fp32) is at its largest against the scores it rides on."""
    rng = np.random.default_rng(41)
    d, page = 128, 64
    lens = np.array([1, 129, 1500, 4096], np.int32)
    T = int(lens.sum())
    k = rng.standard_normal((T, d), dtype=np.float32) * np.float32(0.1 * k_offset) + np.float32(k_offset)
    v = rng.standard_normal((T, d), dtype=np.float32)
    s = build_caches(rng, lens, page, d, 1, kv_bits=[(synth.f32_to_bf16_bits(k), synth.f32_to_bf16_bits(v))])
    for sign in (1.0, -1.0):
        qf = (np.abs(rng.standard_normal((4, 32, d), dtype=np.float32)) + np.float32(0.5)) * np.float32(sign * 2.0)
        q = synth.f32_to_bf16_bits(qf)
        for window in (0, 1024):
            out, ref = run_decode(s, q, window, num_splits=0)
            assert_close(out, ref, f"one-signed q sign {sign} window {window} k_offset {k_offset}")


def test_decode_is_deterministic():
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 5000, size=16).astype(np.int32)
    s = build_caches(rng, lens, 64, 128, 1)
    q = to_dev_bf16(synth.bf16_normal(rng, (16, 32, 128)))
    a = mk.mqa_decode_attn(s.gpu_caches, [0], 0, 0, s.batch, q, num_splits=0)
    b = mk.mqa_decode_attn(s.gpu_caches, [0], 0, 0, s.batch, q, num_splits=0)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_decode_without_host_lengths():
    rng = np.random.default_rng(6)
    lens = np.array([10, 3000, 600, 1], np.int32)
    s = build_caches(rng, lens, 64, 128, 1, with_host_lens=False)
    q = synth.bf16_normal(rng, (4, 32, 128))
    for window in (0, 1024):
        out, ref = run_decode(s, q, window, num_splits=0)
        assert_close(out, ref, f"no host lens W={window}")


def test_device_checks_flag_bad_inputs_without_faulting():
    rng = np.random.default_rng(9)
    lens = np.array([100, 200], np.int32)
    s = build_caches(rng, lens, 64, 128, 1)
    q = to_dev_bf16(synth.bf16_normal(rng, (2, 32, 128)))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_table = s.pb.block_table.copy()
    bad_table[1, 1] = s.pb.num_blocks + 5  # outside the pool
    bad = mk.Batch.from_host(bad_table, lens)
    mk.mqa_decode_attn(s.gpu_caches, [0], 0, 0, bad, q, num_splits=1, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mk.MQA_DEV_BAD_BLOCK
    # a device length beyond max_seq_len (no host copy to catch it)
    status.zero_()
    long_lens = to_dev_i32(np.array([100, 5000], np.int32))
    b2 = mk.Batch(bad.block_table, long_lens, None, 200)
    out = mk.mqa_decode_attn(s.gpu_caches, [0], 0, 0, b2, q, num_splits=1, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mk.MQA_DEV_BAD_SEQLEN
    assert torch.all(out[1].float() == 0)


def test_decode_batch_above_one_pass_partition():
    """More sequences (400) than the tensor-core kernel's threads: its work
    partition takes the multi-pass path; ragged short lengths, both windows."""
    rng = np.random.default_rng(12)
    lens = rng.integers(1, 700, size=400).astype(np.int32)
    s = build_caches(rng, lens, 64, 128, 1)
    for window in (0, 256):
        q = synth.bf16_normal(rng, (len(lens), 32, 128))
        out, ref = run_decode(s, q, window, num_splits=4)  # explicit: balanced shares, never whole pairs
        assert_close(out, ref, f"batch 400 W={window}")


@pytest.mark.parametrize("heads", [32, 64])
def test_decode_one_long_sequence_cut_into_many_pieces(heads):
    """Batch 1, 40k tokens: the balanced split cuts the sequence into one piece
    per CTA (far more than 32), all merged by the last one."""
    rng = np.random.default_rng(13 + heads)
    lens = np.array([40000], np.int32)
    s = build_caches(rng, lens, 64, 128, 1)
    q = synth.bf16_normal(rng, (1, heads, 128))
    out, ref = run_decode(s, q, 0, num_splits=0)
    assert_close(out, ref, f"one long sequence H={heads}")


def test_back_to_back_calls_keep_every_handoff_in_step():
    """Many decode calls in a row, alternating a local and a global layer over
    two caches (the warp-specialised kernel's barriers are exercised hundreds
    of thousands of times): no call may report a timeout, and the outputs
    still match the oracle."""
    rng = np.random.default_rng(15)
    # the 24-layer workload's length mix: batch 128, lognormal around 4k, many short
    # sequences (pieces of a single block follow one another)
    lens = synth.seq_lens_for(synth.CONFIGS["stack24_b128"], rng)
    s = build_caches(rng, lens, 64, 128, 2)
    q_bits = synth.bf16_normal(rng, (2, len(lens), 32, 128))
    qs = [to_dev_bf16(q_bits[i]) for i in range(2)]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = {}
    for it in range(48):
        layer = it % 2
        window = 1024 if layer == 0 else 0
        outs[layer] = mk.mqa_decode_attn(s.gpu_caches, [0, 1], layer, window, s.batch, qs[layer],
                                         sm_scale=sm_scale(128), num_splits=0, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item()):#x}"
    for layer, window in ((0, 1024), (1, 0)):
        ref, _ = oracle.decode(s.ora_caches[layer], s.pb.block_table, s.seq_lens, q_bits[layer], window,
                               sm_scale(128))
        assert_close(outs[layer], ref, f"back-to-back layer {layer}")


def test_device_length_check_in_balanced_mode():
    """A device length beyond max_seq_len with automatic splitting: that
    sequence is zero-filled and flagged, the others are computed."""
    rng = np.random.default_rng(14)
    lens = np.array([100, 200, 3000], np.int32)
    s = build_caches(rng, lens, 64, 128, 1)
    q_bits = synth.bf16_normal(rng, (3, 32, 128))
    q = to_dev_bf16(q_bits)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dev_lens = to_dev_i32(np.array([100, 5000, 3000], np.int32))
    b2 = mk.Batch(s.batch.block_table, dev_lens, None, 3000)
    out = mk.mqa_decode_attn(s.gpu_caches, [0], 0, 0, b2, q, num_splits=0, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & mk.MQA_DEV_BAD_SEQLEN
    assert torch.all(out[1].float() == 0)
    ref, _ = oracle.decode(s.ora_caches[0], s.pb.block_table, lens, q_bits, 0, sm_scale(128))
    assert_close(out[[0, 2]], ref[[0, 2]], "balanced mode, valid sequences")


# ----------------------------------------------------------------- combine
@pytest.mark.parametrize("d", [64, 128])
def test_split_kv_combine_matches_oracle(d):
    rng = np.random.default_rng(40 + d)
    B, S, H = 5, 7, 32
    parts = rng.standard_normal((B, S, H, d)).astype(np.float32)
    lse = (rng.standard_normal((B, S, H)) * 3).astype(np.float32)
    lse[0, 2:, :] = -np.inf          # empty splits
    lse[1, :, 0] = -np.inf           # a (sequence, head) with nothing at all
    out = mk.split_kv_combine(torch.from_numpy(parts).cuda(), torch.from_numpy(lse).cuda())
    torch.cuda.synchronize()
    for b in range(B):
        o, _ = oracle.combine(parts[b].reshape(S, H, d).astype(np.float64), lse[b].astype(np.float64))
        assert_close(out[b], o.reshape(H, d), f"combine b={b}")
    assert torch.all(out[1, 0].float() == 0)
