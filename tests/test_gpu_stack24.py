"""GPU parity of one whole decode step of the 24-layer local/global stack
(batch 128, 32 heads, d=128, page 64, lognormal lengths, 12 caches) against
the CPU oracle, through the C ABI.

The step is issued exactly as a serving loop (and the benchmark) issues it:
for every layer in order, the new token of cache c is quantised and appended
(kv_quant_append) just before the first layer that reads cache c, then the
layer's decode attention runs with its window (1024 on local layers, 0 on the
layers l % 6 == 5).  Two layer -> cache maps are checked: the stack's own
pairing (consecutive local layers share a cache, global layers are tied across
blocks) and the plain adjacent pairing map[l] = l // 2 (Character.AI inference
article, secret 1, cross-layer KV sharing; the pages leave the exact pairing
open, and both readings must give the same attention).

The GPU holds all 128 sequences, so every call runs the automatic plan of the
real workload; the oracle recomputes a seeded sample of sequences (plus the
shortest and the longest) on compact caches holding the same token bits.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import mqa_decode_attention_kv_gb300 as mk
from gpu_common import assert_close, sm_scale, to_dev_bf16, to_dev_i32

pytestmark = pytest.mark.gpu

N_SAMPLE = 32


def rolled(pool: np.ndarray, c: int) -> np.ndarray:
    """Token rows of cache c: the shared random pool rotated by a cache-specific
    offset, so that every cache holds different K/V rows."""
    return np.roll(pool, 7919 * (c + 1), axis=0)


def append_order(layer_map):
    """layer -> cache whose new token is appended just before that layer (the
    first layer reading the cache)."""
    first = {}
    for l, c in enumerate(layer_map):
        first.setdefault(c, l)
    return {l: c for c, l in first.items()}


@pytest.mark.parametrize("map_kind", ["stack_pairs", "half"])
def test_stack24_step_matches_oracle(map_kind):
    w = synth.CONFIGS["stack24_b128"]
    rng = np.random.default_rng(w.seed)
    lens = synth.seq_lens_for(w, rng)
    B, H, d, P = w.batch, w.num_q_heads, w.head_dim, w.page_size
    L = w.num_layers
    layer_map = list(w.layer_map) if map_kind == "stack_pairs" else [l // 2 for l in range(L)]
    num_caches = max(layer_map) + 1
    assert num_caches == 12
    pb = synth.make_paged_batch(rng, lens, P, shuffle=True)
    cu = synth.cu_from_counts(lens)
    T = int(cu[-1])
    k_pool = synth.bf16_normal(rng, (T, d))
    v_pool = synth.bf16_normal(rng, (T, d))
    q_bits = synth.bf16_normal(rng, (L, B, H, d))
    kn = synth.bf16_normal(rng, (num_caches, B, d))
    vn = synth.bf16_normal(rng, (num_caches, B, d))

    # the oracle's sample: seeded sequences plus the shortest and the longest
    pick = set(synth.sample_rows(np.random.default_rng(400), B, N_SAMPLE).tolist())
    pick |= {int(np.argmin(lens)), int(np.argmax(lens))}
    sample = np.array(sorted(pick), np.int64)
    lens_s = lens[sample]
    pb_s = synth.make_paged_batch(None, lens_s, P, shuffle=False)
    cu_s = synth.cu_from_counts(lens_s)
    rows_s = np.concatenate([np.arange(cu[b], cu[b + 1]) for b in sample])

    # caches: every token of every sequence on the GPU, the sample in the oracle
    batch = mk.Batch.from_host(pb.block_table, lens)
    cu_dev = to_dev_i32(cu)
    gpu, ora = [], []
    for c in range(num_caches):
        kc, vc = rolled(k_pool, c), rolled(v_pool, c)
        gc = mk.KVCache.empty(pb.num_blocks, P, d)
        mk.kv_quant_append(gc, batch, cu_dev, T, to_dev_bf16(kc), to_dev_bf16(vc))
        oc = oracle.Cache.empty(pb_s.num_blocks, P, d)
        oracle.quant_append(oc, pb_s.block_table, lens_s, cu_s, np.ascontiguousarray(kc[rows_s]),
                            np.ascontiguousarray(vc[rows_s]))
        gpu.append(gc)
        ora.append(oc)
    torch.cuda.synchronize()

    # one step, in the serving order
    before = append_order(layer_map)
    cu_step = to_dev_i32(np.arange(B + 1))
    cu_step_s = synth.cu_from_counts(np.ones(len(sample)))
    kn_dev, vn_dev, q_dev = to_dev_bf16(kn), to_dev_bf16(vn), to_dev_bf16(q_bits)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for l in range(L):
        c = before.get(l)
        if c is not None:
            mk.kv_quant_append(gpu[c], batch, cu_step, B, kn_dev[c], vn_dev[c], dev_status=status)
            oracle.quant_append(ora[c], pb_s.block_table, lens_s, cu_step_s, np.ascontiguousarray(kn[c][sample]),
                                np.ascontiguousarray(vn[c][sample]))
        outs.append(mk.mqa_decode_attn(gpu, layer_map, l, w.windows[l], batch, q_dev[l], sm_scale=sm_scale(d),
                                       num_splits=0, dev_status=status))
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item()):#x}"

    # every layer's output on the sample
    for l in range(L):
        ref, _ = oracle.decode(ora[layer_map[l]], pb_s.block_table, lens_s,
                               np.ascontiguousarray(q_bits[l][sample]), w.windows[l], sm_scale(d))
        assert_close(outs[l][torch.from_numpy(sample).cuda()], ref, f"{map_kind} layer {l} window {w.windows[l]}")

    # the cache bytes after the step: the appended slot of all 128 sequences
    # against the oracle's quantiser, and every slot of the sampled sequences
    last = lens - 1
    blk = torch.from_numpy(pb.block_table[np.arange(B), last // P].astype(np.int64)).cuda()
    off = torch.from_numpy((last % P).astype(np.int64)).cuda()
    for c in range(num_caches):
        kc_, ks_ = oracle.quantize_tokens(kn[c])
        vc_, vs_ = oracle.quantize_tokens(vn[c])
        g = gpu[c]
        assert np.array_equal(g.k_codes[blk, off].cpu().numpy(), kc_), f"cache {c}: appended K codes"
        assert np.array_equal(g.v_codes[blk, off].cpu().numpy(), vc_), f"cache {c}: appended V codes"
        assert np.array_equal(g.k_scale[blk, off].cpu().numpy().view(np.uint32), ks_.view(np.uint32))
        assert np.array_equal(g.v_scale[blk, off].cpu().numpy().view(np.uint32), vs_.view(np.uint32))
        nblk_s = (lens_s + P - 1) // P
        for i, b in enumerate(sample):
            gb = torch.from_numpy(pb.block_table[b, :nblk_s[i]].astype(np.int64)).cuda()
            ob = pb_s.block_table[i, :nblk_s[i]]
            n = int(lens_s[i])
            gk = g.k_codes[gb].reshape(-1, d)[:n].cpu().numpy()
            ok = ora[c].k_codes[ob].reshape(-1, d)[:n]
            gv = g.v_codes[gb].reshape(-1, d)[:n].cpu().numpy()
            ov = ora[c].v_codes[ob].reshape(-1, d)[:n]
            gks = g.k_scale[gb].reshape(-1)[:n].cpu().numpy().view(np.uint32)
            oks = ora[c].k_scale[ob].reshape(-1)[:n].view(np.uint32)
            gvs = g.v_scale[gb].reshape(-1)[:n].cpu().numpy().view(np.uint32)
            ovs = ora[c].v_scale[ob].reshape(-1)[:n].view(np.uint32)
            assert np.array_equal(gk, ok) and np.array_equal(gv, ov), f"cache {c} seq {b}: codes"
            assert np.array_equal(gks, oks) and np.array_equal(gvs, ovs), f"cache {c} seq {b}: scales"
