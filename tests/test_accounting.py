"""Pins for the byte/flop accounting: the workshop's printed KV-size example
(tests/golden/kv_size_mistral7b.txt) and brute-force counts of attended keys."""
import os

import numpy as np

from mqa_decode_attention_kv_gb300 import accounting as acc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_size_mistral7b.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = float(v)
    return vals


def test_workshop_kv_size_example():
    g = _golden()
    per_tok = acc.kv_bytes_per_token(int(g["layers"]), int(g["kv_heads"]), int(g["head_dim"]),
                                     g["bytes_per_elem"])
    assert per_tok == 131072
    assert round(per_tok / 1000) == g["per_token_kbytes"]
    assert abs(per_tok * 4096 / 1e9 - g["ctx4k_gb"]) / g["ctx4k_gb"] < 0.1      # 0.537 vs "half a GB"
    assert abs(per_tok * 16384 / 1e9 - g["ctx16k_gb"]) / g["ctx16k_gb"] < 0.05  # 2.15 vs 2.1
    assert abs(80 * per_tok * 4096 / 1e9 - g["users80_ctx4k_gb"]) / g["users80_ctx4k_gb"] < 0.05


def test_mqa_vs_gqa8_is_eight_times_smaller():
    # Character.AI article, secret 1: MQA cuts the KV cache 8x relative to GQA (8 KV heads)
    assert acc.kv_bytes_per_token(1, 8, 128, 2) / acc.kv_bytes_per_token(1, 1, 128, 2) == 8


def test_decode_counts_match_brute_force():
    L = np.array([1, 5, 1024, 1025, 3000])
    for W in (0, 1024, 7):
        n = sum(len([j for j in range(l) if W == 0 or j > l - 1 - W]) for l in L)
        assert acc.keys_attended(L, W).sum() == n
        assert acc.decode_kv_bytes(L, W, 128) == n * 264
        assert acc.decode_flops(L, W, 32, 128) == 4 * 128 * 32 * n


def test_prefill_pairs_match_brute_force():
    L = np.array([10, 40, 7])
    q = np.array([3, 40, 1])
    for W in (0, 5):
        n = 0
        for l, m in zip(L, q):
            for i in range(l - m, l):
                n += len([j for j in range(i + 1) if W == 0 or j > i - W])
        assert acc.prefill_pairs(L, q, W) == n
