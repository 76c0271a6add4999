"""Host-side tests of the C ABI (no GPU needed).

The library must load, export every function include/mqa_kv.h declares, and
reject bad arguments with a negative status before touching the GPU.  Device
pointers here are fake (never dereferenced): each call fails validation first.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import mqa_decode_attention_kv_gb300 as mk
from mqa_decode_attention_kv_gb300 import build as mkbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]
FAKE = 0x10000  # a 16-byte aligned non-null "device" address, never dereferenced


@pytest.fixture(scope="module")
def L():
    mkbuild.build()
    return mk.lib()


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*([a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert set(names) >= {"kv_quant_append", "mqa_decode_attn", "mqa_prefill_attn", "split_kv_combine"}
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    assert set(mk.EXPORTED) == set(names)


def test_status_strings(L):
    for s in (0, -1, -2, -3, -4):
        assert mk.status_str(s)
    assert mk.status_str(123) == "unknown status"


def test_workspace_size_formula(L):
    assert mk.mqa_decode_workspace_size(8, 32, 128, 1) == 0
    n = mk.mqa_decode_workspace_size(8, 32, 128, 10)
    r256 = lambda x: (x + 255) // 256 * 256
    part = 8 * 10 * 32 * 128 * 4           # fp32 partial outputs
    lse = 8 * 10 * 32 * 4                  # fp32 log-sum-exps
    descs = 2 * 1024 * 8 * 4               # merge descriptors of up to 1024 CTAs
    assert n == r256(r256(part) + lse) + descs


def cache(num_blocks=16, page=16, d=64, **kw):
    c = mk._Cache(FAKE, FAKE, FAKE, FAKE, num_blocks, page, d)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def batch(n=2, max_blocks=4, max_seq_len=64, lens=None, **kw):
    host = None
    keep = None
    if lens is not None:
        keep = np.asarray(lens, np.int32)
        host = keep.ctypes.data
    b = mk._Batch(FAKE, FAKE, host, n, max_blocks, max_seq_len)
    for k, v in kw.items():
        setattr(b, k, v)
    return b, keep


def decode(L, c, b, layer_map=(0,), layer=0, window=0, heads=8, splits=1, ws=None, ws_bytes=0, q=FAKE, out=FAKE,
           num_caches=1, scale=0.125):
    arr = (mk._Cache * num_caches)(*([c] * num_caches))
    lm = (ctypes.c_int32 * len(layer_map))(*layer_map)
    return L.mqa_decode_attn(arr, num_caches, lm, len(layer_map), layer, window, ctypes.byref(b), q, out, heads,
                             scale, splits, ws, ws_bytes, None, None)


def test_decode_argument_validation(L):
    b, keep = batch(lens=[10, 20])
    assert decode(L, cache(d=96), b) == mk.MQA_ERR_UNSUPPORTED
    assert decode(L, cache(page=32), b) == mk.MQA_ERR_UNSUPPORTED
    assert decode(L, cache(), b, heads=12) == mk.MQA_ERR_UNSUPPORTED
    assert decode(L, cache(k_codes=None), b) == mk.MQA_ERR_INVALID_ARG
    assert decode(L, cache(k_scale=FAKE + 4), b) == mk.MQA_ERR_INVALID_ARG      # misaligned
    assert decode(L, cache(num_blocks=0), b) == mk.MQA_ERR_INVALID_ARG
    assert decode(L, cache(), b, q=None) == mk.MQA_ERR_INVALID_ARG
    assert decode(L, cache(), b, out=FAKE + 2) == mk.MQA_ERR_INVALID_ARG
    assert decode(L, cache(), b, layer_map=(1,)) == mk.MQA_ERR_INVALID_ARG    # map out of range
    assert decode(L, cache(), b, layer=1) == mk.MQA_ERR_INVALID_ARG           # layer out of range
    assert decode(L, cache(), b, window=-1) == mk.MQA_ERR_INVALID_ARG
    assert decode(L, cache(), b, splits=-1) == mk.MQA_ERR_INVALID_ARG
    assert decode(L, cache(), b, splits=mk.MQA_MAX_SPLITS + 1) == mk.MQA_ERR_INVALID_ARG
    assert decode(L, cache(), b, scale=float("nan")) == mk.MQA_ERR_INVALID_ARG
    # seq_len 0, or above max_seq_len, in the host copy
    b0, k0 = batch(lens=[0, 20])
    assert decode(L, cache(), b0) == mk.MQA_ERR_INVALID_ARG
    b1, k1 = batch(lens=[65, 20])
    assert decode(L, cache(), b1) == mk.MQA_ERR_INVALID_ARG
    # max_seq_len beyond the block table's reach (4 blocks x 16 = 64)
    b2, k2 = batch(max_seq_len=65, lens=[10, 20])
    assert decode(L, cache(), b2) == mk.MQA_ERR_INVALID_ARG
    b3, _ = batch(block_table=None)
    assert decode(L, cache(), b3) == mk.MQA_ERR_INVALID_ARG
    # split-KV without (enough) workspace
    b4, k4 = batch(max_blocks=16, max_seq_len=256, lens=[256, 256])  # 4 tiles of 64: two splits
    assert decode(L, cache(), b4, splits=2) == mk.MQA_ERR_WORKSPACE
    need = mk.mqa_decode_workspace_size(2, 8, 64, 2)
    assert decode(L, cache(), b4, splits=2, ws=FAKE, ws_bytes=need - 1) == mk.MQA_ERR_WORKSPACE
    # an empty batch is a valid no-op
    be, _ = batch(n=0)
    assert decode(L, cache(), be) == mk.MQA_OK


def test_append_argument_validation(L):
    b, keep = batch(lens=[10, 20])
    c = cache()
    f = L.kv_quant_append
    assert f(ctypes.byref(c), ctypes.byref(b), FAKE, 0, FAKE, FAKE, None, None) == mk.MQA_OK  # no-op
    assert f(ctypes.byref(c), ctypes.byref(b), FAKE, -1, FAKE, FAKE, None, None) == mk.MQA_ERR_INVALID_ARG
    assert f(ctypes.byref(c), ctypes.byref(b), None, 3, FAKE, FAKE, None, None) == mk.MQA_ERR_INVALID_ARG
    assert f(ctypes.byref(c), ctypes.byref(b), FAKE, 3, FAKE + 8, FAKE, None, None) == mk.MQA_ERR_INVALID_ARG
    c96 = cache(d=96)
    assert f(ctypes.byref(c96), ctypes.byref(b), FAKE, 3, FAKE, FAKE, None, None) == mk.MQA_ERR_UNSUPPORTED
    b0, k0 = batch(lens=[0, 20])
    assert f(ctypes.byref(c), ctypes.byref(b0), FAKE, 3, FAKE, FAKE, None, None) == mk.MQA_ERR_INVALID_ARG
    assert f(None, ctypes.byref(b), FAKE, 3, FAKE, FAKE, None, None) == mk.MQA_ERR_INVALID_ARG


def test_combine_and_prefill_validation(L):
    assert L.split_kv_combine(FAKE, FAKE, 2, 3, 8, 96, FAKE, None) == mk.MQA_ERR_UNSUPPORTED
    assert L.split_kv_combine(FAKE, FAKE, 2, 0, 8, 64, FAKE, None) == mk.MQA_ERR_INVALID_ARG
    assert L.split_kv_combine(None, FAKE, 2, 3, 8, 64, FAKE, None) == mk.MQA_ERR_INVALID_ARG
    assert L.split_kv_combine(FAKE, FAKE, 0, 3, 8, 64, FAKE, None) == mk.MQA_OK
    b, keep = batch(lens=[10, 20])
    arr = (mk._Cache * 1)(cache())
    lm = (ctypes.c_int32 * 1)(0)
    P = L.mqa_prefill_attn
    assert P(arr, 1, lm, 1, 0, 0, ctypes.byref(b), FAKE, 0, 0, FAKE, FAKE, 8, 0.1, None, 0, None, None) == mk.MQA_OK
    assert P(arr, 1, lm, 1, 0, 0, ctypes.byref(b), None, 5, 3, FAKE, FAKE, 8, 0.1, None, 0, None, None) == mk.MQA_ERR_INVALID_ARG
    assert P(arr, 1, lm, 1, 0, 0, ctypes.byref(b), FAKE, 5, 65, FAKE, FAKE, 8, 0.1, None, 0, None, None) == mk.MQA_ERR_INVALID_ARG
    assert P(arr, 1, lm, 1, 0, -3, ctypes.byref(b), FAKE, 5, 3, FAKE, FAKE, 8, 0.1, None, 0, None, None) == mk.MQA_ERR_INVALID_ARG
    assert P(arr, 1, lm, 1, 0, 0, ctypes.byref(b), FAKE, 5, 3, FAKE, FAKE, 24, 0.1, None, 0, None, None) == mk.MQA_ERR_UNSUPPORTED
    # the key tiles are converted into a workspace first: missing or short -> rejected
    arr128 = (mk._Cache * 1)(cache(d=128, page=64))
    b128, k128 = batch(max_blocks=4, max_seq_len=256, lens=[200, 130])
    need = mk.mqa_prefill_workspace_size(2, 256, 0, 3, 128)
    assert need > 0 and mk.mqa_prefill_workspace_size(2, 256, 0, 3, 96) == 0
    assert P(arr128, 1, lm, 1, 0, 0, ctypes.byref(b128), FAKE, 5, 3, FAKE, FAKE, 32, 0.1, None, 0, None,
             None) == mk.MQA_ERR_WORKSPACE
    assert P(arr128, 1, lm, 1, 0, 0, ctypes.byref(b128), FAKE, 5, 3, FAKE, FAKE, 32, 0.1, FAKE, need - 1, None,
             None) == mk.MQA_ERR_WORKSPACE
    arr64 = (mk._Cache * 1)(cache(d=64, page=16))
    b64, k64 = batch(max_blocks=16, max_seq_len=256, lens=[200, 130])
    assert P(arr64, 1, lm, 1, 0, 0, ctypes.byref(b64), FAKE, 5, 3, FAKE, FAKE, 8, 0.1, None, 0, None,
             None) == mk.MQA_ERR_WORKSPACE


def test_prefill_workspace_formula(L):
    r256 = lambda x: (x + 255) // 256 * 256
    # per sequence: the tiles of the key range plus one all-invalid tile; 256 * head_dim byte images,
    # 528-byte records
    for B, Lmax, W, Q in ((3, 8704, 0, 512), (256, 8704, 1024, 512), (5, 100, 1024, 7), (2, 64, 0, 64)):
        tiles = -(-Lmax // 64)
        if W > 0:
            tiles = min(tiles, (W + Q - 2) // 64 + 2)
        n = B * (tiles + 1)
        for d in (64, 128):
            assert mk.mqa_prefill_workspace_size(B, Lmax, W, Q, d) == r256(n * 256 * d) + n * 528


def test_auto_splits_validation(L):
    b, keep = batch(lens=[10, 20])
    assert L.mqa_decode_auto_splits(ctypes.byref(b), 0, 8, 96, 16) == mk.MQA_ERR_UNSUPPORTED
    assert L.mqa_decode_auto_splits(ctypes.byref(b), -5, 8, 64, 16) == mk.MQA_ERR_INVALID_ARG


def test_ring_argument_validation(L):
    """Window-bounded caches (ring_blocks = R > 0): R within the table, a
    window on every read, and enough resident pages for that window."""
    c = cache(page=16)
    # R outside [0, max_blocks]
    b, k = batch(lens=[10, 20], ring_blocks=-1)
    assert decode(L, c, b, window=16) == mk.MQA_ERR_INVALID_ARG
    b, k = batch(lens=[10, 20], ring_blocks=5)
    assert decode(L, c, b, window=16) == mk.MQA_ERR_INVALID_ARG
    # a ring may serve sequences longer than its table (4 entries x 16 tokens)
    be, _ = batch(n=0, max_seq_len=10000, ring_blocks=4)
    assert decode(L, c, be, window=48) == mk.MQA_OK              # (48 - 1) / 16 + 2 = 4 pages
    assert decode(L, c, be, window=49) == mk.MQA_ERR_INVALID_ARG  # needs 5
    assert decode(L, c, be, window=0) == mk.MQA_ERR_INVALID_ARG   # global attention reads evicted pages
    # ... but a full table may not
    bf, kf = batch(lens=[10, 20], max_seq_len=10000)
    assert decode(L, c, bf, window=48) == mk.MQA_ERR_INVALID_ARG
    # prefill: the chunk's keys and the windows of all its queries must be resident
    arr = (mk._Cache * 1)(c)
    lm = (ctypes.c_int32 * 1)(0)

    def prefill(b, window, max_q):
        return L.mqa_prefill_attn(arr, 1, lm, 1, 0, window, ctypes.byref(b), FAKE, 10, max_q, FAKE, FAKE, 8,
                                  0.125, None, 0, None, None)
    br, kr = batch(lens=[100, 90], max_seq_len=100, ring_blocks=4)
    assert prefill(br, 16, 34) == mk.MQA_ERR_INVALID_ARG   # (16 + 34 - 2) / 16 + 2 = 5 pages > 4
    assert prefill(br, 49, 1) == mk.MQA_ERR_INVALID_ARG    # (49 + 1 - 2) / 16 + 2 = 5 pages > 4
    assert prefill(br, 0, 1) == mk.MQA_ERR_INVALID_ARG     # global attention reads evicted pages
    # append accepts the ring (its per-sequence chunk bound is checked on the device)
    b, k = batch(lens=[10, 20], ring_blocks=5)
    assert L.kv_quant_append(ctypes.byref(c), ctypes.byref(b), FAKE, 3, FAKE, FAKE, None, None) \
        == mk.MQA_ERR_INVALID_ARG
