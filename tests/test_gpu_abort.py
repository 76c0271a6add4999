"""GPU test of the decode kernel's abort path: every wait is bounded, and a wait
that runs out makes the whole CTA leave (after letting its own copies and MMAs
in flight land) and report MQA_DEV_TIMEOUT, with the GPU still usable.

A test-only build of the library (MQA_TEST_WAIT_LIMIT_NS=1) makes every
pipeline wait give up almost at once, so the first wait that is not already
satisfied runs out; drains keep their normal limit.  Nothing here blocks: the
waits give up, they never hang.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import synth
import mqa_decode_attention_kv_gb300 as mk
from mqa_decode_attention_kv_gb300 import build as mk_build
from gpu_common import assert_close, build_caches, sm_scale, to_dev_bf16

pytestmark = pytest.mark.gpu


def short_wait_lib():
    return mk.declare(ctypes.CDLL(mk_build.build_variant("shortwait", ["-DMQA_TEST_WAIT_LIMIT_NS=1"])))


@pytest.mark.parametrize("window,lens", [(1024, (1500, 3000, 700, 9000)), (0, (40000, 2500, 17, 12000))])
def test_timeout_reports_status_and_gpu_keeps_working(window, lens):
    rng = np.random.default_rng(91 + window)
    d, H = 128, 32
    s = build_caches(rng, np.array(lens, np.int32), 64, d, 1)
    q_bits = synth.bf16_normal(rng, (len(lens), H, d))
    q = to_dev_bf16(q_bits)
    L = short_wait_lib()
    carr = mk._caches_array(s.gpu_caches)
    lmap = (ctypes.c_int32 * 1)(0)
    bt = s.batch.c()
    stream = torch.cuda.current_stream().cuda_stream
    for splits in (1, 4):  # one CTA per (sequence, head group), then balanced shares + merge
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        out = torch.empty_like(q)
        ws = torch.empty(max(16, mk.mqa_decode_workspace_size(len(lens), H, d, splits)), dtype=torch.uint8,
                         device="cuda")
        rc = L.mqa_decode_attn(carr, 1, lmap, 1, 0, window, ctypes.byref(bt), q.data_ptr(), out.data_ptr(), H,
                               1.0 / math.sqrt(d), splits, ws.data_ptr(), ws.numel(),
                               ctypes.c_void_p(status.data_ptr()), stream)
        assert rc == mk.MQA_OK, mk.status_str(rc)
        torch.cuda.synchronize()  # the call ended: no wait hung
        assert int(status.item()) & mk.MQA_DEV_TIMEOUT, f"splits={splits}: no timeout reported"
    # the GPU still answers: the product library on the same inputs and stream
    ok_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mk.mqa_decode_attn(s.gpu_caches, [0], 0, window, s.batch, q, sm_scale=sm_scale(d), dev_status=ok_status)
    torch.cuda.synchronize()
    assert int(ok_status.item()) == 0
    ref, _ = oracle.decode(s.ora_caches[0], s.pb.block_table, s.seq_lens, q_bits, window, sm_scale(d))
    assert_close(out, ref, f"after aborted calls, window {window}")


@pytest.mark.parametrize("d,H,window", [(128, 32, 0), (64, 8, 256)])
def test_prefill_timeout_reports_status_and_gpu_keeps_working(d, H, window):
    """The same for the prefill kernels: with near-zero wait limits a chunked
    prefill gives up, reports MQA_DEV_TIMEOUT and leaves (its copies and MMAs
    drained); the GPU then runs the product library's prefill correctly."""
    rng = np.random.default_rng(93 + d)
    lens = np.array([900, 130, 2000], np.int32)
    q_lens = np.array([300, 130, 64], np.int64)
    s = build_caches(rng, lens, 64, d, 1)
    cu_q = synth.cu_from_counts(q_lens)
    T = int(cu_q[-1])
    q_bits = synth.bf16_normal(rng, (T, H, d))
    q = to_dev_bf16(q_bits)
    cu_dev = torch.from_numpy(cu_q).cuda()
    L = short_wait_lib()
    carr = mk._caches_array(s.gpu_caches)
    lmap = (ctypes.c_int32 * 1)(0)
    bt = s.batch.c()
    stream = torch.cuda.current_stream().cuda_stream
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    ws = torch.empty(max(16, mk.mqa_prefill_workspace_size(len(lens), int(lens.max()), window, int(q_lens.max()), d)),
                     dtype=torch.uint8, device="cuda")
    rc = L.mqa_prefill_attn(carr, 1, lmap, 1, 0, window, ctypes.byref(bt), cu_dev.data_ptr(), T, int(q_lens.max()),
                            q.data_ptr(), out.data_ptr(), H, 1.0 / math.sqrt(d), ws.data_ptr(), ws.numel(),
                            ctypes.c_void_p(status.data_ptr()), stream)
    assert rc == mk.MQA_OK, mk.status_str(rc)
    torch.cuda.synchronize()  # the call ended: no wait hung
    assert int(status.item()) & mk.MQA_DEV_TIMEOUT, "no timeout reported"
    ok_status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = mk.mqa_prefill_attn(s.gpu_caches, [0], 0, window, s.batch, cu_dev, q, int(q_lens.max()),
                              sm_scale=sm_scale(d), dev_status=ok_status)
    torch.cuda.synchronize()
    assert int(ok_status.item()) == 0
    rs, rp = oracle.prefill_rows(cu_q, lens)
    ref, _ = oracle.attention(s.ora_caches[0], s.pb.block_table, lens, q_bits, rs, rp, window, sm_scale(d))
    assert_close(out, ref, f"prefill after an aborted call, d={d} window {window}")
