"""Algorithmic byte and flop counts used to report throughput and roofline
fractions.  These count what the method must touch, not what a kernel happens
to move: the int8 codes plus fp32 scales of exactly the keys each query row
attends to, and 4*d flops per (query head, key) pair (QK^T and PV, one
multiply-add each per element).
"""
from __future__ import annotations

import numpy as np


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: float) -> float:
    """KV-cache bytes per token of a dense cache: K and V, each
    layers x kv_heads x head_dim elements (LLM-inference workshop transcript,
    00:14:45-00:15:23, the per-token KV size of Mistral 7B)."""
    return 2.0 * layers * kv_heads * head_dim * bytes_per_elem


def int8_token_bytes(head_dim: int) -> int:
    """Bytes one cached token occupies in one int8 cache: K and V codes
    (head_dim bytes each) plus one fp32 scale each."""
    return 2 * (head_dim + 4)


def keys_attended(seq_lens, window: int) -> np.ndarray:
    """Keys seen by the decode query at position L-1: min(L, W) for a local
    layer, L for a global one."""
    L = np.asarray(seq_lens, dtype=np.int64)
    return np.minimum(L, window) if window > 0 else L


def decode_kv_bytes(seq_lens, window: int, head_dim: int) -> int:
    return int(keys_attended(seq_lens, window).sum()) * int8_token_bytes(head_dim)


def decode_flops(seq_lens, window: int, num_q_heads: int, head_dim: int) -> int:
    return 4 * head_dim * num_q_heads * int(keys_attended(seq_lens, window).sum())


def prefill_pairs(seq_lens, q_lens, window: int) -> int:
    """(query row, key) pairs of a causal prefill chunk: query t of a chunk of
    q_len new tokens sits at position i = L - q_len + t and sees keys
    max(0, i-W+1)..i (all of 0..i when global)."""
    total = 0
    for L, n in zip(np.asarray(seq_lens, np.int64), np.asarray(q_lens, np.int64)):
        i = np.arange(L - n, L, dtype=np.int64)
        cnt = i + 1
        if window > 0:
            cnt = np.minimum(cnt, window)
        total += int(cnt.sum())
    return total


def prefill_flops(seq_lens, q_lens, window: int, num_q_heads: int, head_dim: int) -> int:
    return 4 * head_dim * num_q_heads * prefill_pairs(seq_lens, q_lens, window)
