"""GPU test of mqa_decode_attn_noalloc, the decode entry point for callers that
cannot allocate device memory (it keeps split-KV partials in a library-owned
32 MiB device array instead of a caller workspace).

Collected last on purpose: if it fails, a run that stops at the first failure
has already run every other test.  It builds its own inputs, so it passes both
alone in a fresh process and after the other tests.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import synth
import mqa_decode_attention_kv_gb300 as mk
from gpu_common import assert_close, build_caches, to_dev_bf16

pytestmark = pytest.mark.gpu


def noalloc_call(s, q, window, num_splits, heads, d):
    out = torch.empty_like(q)
    carr = mk._caches_array(s.gpu_caches)
    lmap = (ctypes.c_int32 * 1)(0)
    bt = s.batch.c()
    rc = mk.lib().mqa_decode_attn_noalloc(carr, 1, lmap, 1, 0, window, ctypes.byref(bt), q.data_ptr(),
                                          out.data_ptr(), heads, 1.0 / math.sqrt(d), num_splits, None,
                                          torch.cuda.current_stream().cuda_stream)
    assert rc == mk.MQA_OK, mk.status_str(rc)
    return out


@pytest.mark.parametrize("window,lens", [(1024, (1500, 3000, 700, 9000, 64, 1)), (0, (40000, 2500, 17, 12000))])
def test_noalloc_matches_workspace_entry_point_twice(window, lens):
    rng = np.random.default_rng(77 + window)
    d, H = 128, 32
    s = build_caches(rng, np.array(lens, np.int32), 64, d, 1)
    for call in range(2):  # the scratch array keeps the previous call's contents
        q_bits = synth.bf16_normal(rng, (len(lens), H, d))
        q = to_dev_bf16(q_bits)
        ref = mk.mqa_decode_attn(s.gpu_caches, [0], 0, window, s.batch, q, sm_scale=1.0 / math.sqrt(d))
        got = noalloc_call(s, q, window, 0, H, d)
        forced = noalloc_call(s, q, window, 4, H, d)
        torch.cuda.synchronize()
        for g in (got, forced):
            assert_close(g, ref.float().cpu().numpy().astype(np.float64), f"noalloc call {call} vs mqa_decode_attn")
        # and directly against the oracle
        exact, _ = oracle.decode(s.ora_caches[0], s.pb.block_table, s.seq_lens, q_bits, window, 1.0 / math.sqrt(d))
        assert_close(got, exact, f"noalloc call {call} vs oracle")
        assert_close(forced, exact, f"noalloc (4 splits) call {call} vs oracle")


def test_noalloc_rejects_split_counts_beyond_its_scratch():
    rng = np.random.default_rng(5)
    lens = np.full(64, 131072, np.int32)
    pb = synth.make_paged_batch(rng, lens, 64)
    cache = mk.KVCache.empty(16, 64, 128)  # never read: the call is rejected before any launch
    batch = mk.Batch.from_host(pb.block_table, lens)
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    carr = mk._caches_array([cache])
    lmap = (ctypes.c_int32 * 1)(0)
    bt = batch.c()
    # 64 sequences x 1024 splits x 32 heads x 128 x 4 B = 1 GiB of partials > 32 MiB
    rc = mk.lib().mqa_decode_attn_noalloc(carr, 1, lmap, 1, 0, 0, ctypes.byref(bt), q.data_ptr(), out.data_ptr(),
                                          32, 0.088, 1024, None, None)
    assert rc == mk.MQA_ERR_WORKSPACE
