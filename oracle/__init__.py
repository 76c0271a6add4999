"""CPU oracle for int8 paged multi-query attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product library never does, and this
package never imports the product.  The arithmetic lives in ``mqa_oracle.c``
(single-threaded, fp64 attention, fp32 quantisation); this module only
marshals numpy arrays into it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile ``mqa_oracle.c`` with gcc into ``liboracle.so`` (portable C: no
    intrinsics, no -march flags, so it builds the same on x86-64 and aarch64)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32 = ctypes.c_int32
            lib.oracle_quantize_token.argtypes = [P, i32, P, P]
            lib.oracle_quantize_token.restype = None
            lib.oracle_quant_append.argtypes = [P, P, P, P, i32, i32, i32, P, i32, P, i32, P, P, P, i32]
            lib.oracle_quant_append.restype = i32
            lib.oracle_attention.argtypes = [P, P, P, P, i32, i32, i32, P, i32, P, i32, i32,
                                             P, i32, P, P, i32, ctypes.c_double, i32, i32,
                                             P, P, P, ctypes.c_int64, P, i32]
            lib.oracle_attention.restype = i32
            lib.oracle_combine.argtypes = [P, P, i32, ctypes.c_int64, i32, P, P]
            lib.oracle_combine.restype = None
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Cache:
    """One physical KV cache (one shared K/V head) in host memory."""

    k_codes: np.ndarray  # int8 [num_blocks, page_size, d]
    v_codes: np.ndarray
    k_scale: np.ndarray  # float32 [num_blocks, page_size]
    v_scale: np.ndarray

    @classmethod
    def empty(cls, num_blocks: int, page_size: int, d: int) -> "Cache":
        return cls(np.zeros((num_blocks, page_size, d), np.int8),
                   np.zeros((num_blocks, page_size, d), np.int8),
                   np.zeros((num_blocks, page_size), np.float32),
                   np.zeros((num_blocks, page_size), np.float32))

    @property
    def num_blocks(self) -> int:
        return self.k_codes.shape[0]

    @property
    def page_size(self) -> int:
        return self.k_codes.shape[1]

    @property
    def head_dim(self) -> int:
        return self.k_codes.shape[2]


def quantize_tokens(x_bits: np.ndarray):
    """Per-token symmetric int8 quantisation of bf16 rows ``[T, d]`` (uint16 bits).
    Returns ``(codes int8 [T, d], scales float32 [T])``."""
    lib = _load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, d = x.shape
    codes = np.empty((T, d), np.int8)
    scales = np.empty(T, np.float32)
    for t in range(T):
        lib.oracle_quantize_token(ctypes.c_void_p(x.ctypes.data + 2 * t * d), d,
                                  ctypes.c_void_p(codes.ctypes.data + t * d),
                                  ctypes.c_void_p(scales.ctypes.data + 4 * t))
    return codes, scales


def quant_append(cache: Cache, block_table: np.ndarray, seq_lens: np.ndarray,
                 cu_new: np.ndarray, k_new: np.ndarray, v_new: np.ndarray, ring_blocks: int = 0) -> None:
    """Quantise ``k_new``/``v_new`` (bf16 bits ``[T, d]``) and store them at the
    last ``cu_new[b+1]-cu_new[b]`` positions of each sequence, in place.  With
    ``ring_blocks = R > 0`` page ``p // page_size`` lives in table entry
    ``(p // page_size) % R`` (a window-bounded cache keeping R pages)."""
    lib = _load()
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    cu = np.ascontiguousarray(cu_new, np.int32)
    k = np.ascontiguousarray(k_new, np.uint16)
    v = np.ascontiguousarray(v_new, np.uint16)
    rc = lib.oracle_quant_append(_p(cache.k_codes), _p(cache.v_codes), _p(cache.k_scale),
                                 _p(cache.v_scale), cache.num_blocks, cache.page_size,
                                 cache.head_dim, _p(bt), bt.shape[1], _p(sl), sl.shape[0],
                                 _p(cu), _p(k), _p(v), int(ring_blocks))
    if rc != 0:
        raise ValueError("oracle_quant_append: index out of range")


def attention(cache: Cache, block_table: np.ndarray, seq_lens: np.ndarray, q: np.ndarray,
              row_seq: np.ndarray, row_pos: np.ndarray, window: int, sm_scale: float,
              key_range: tuple[int, int] | None = None, want_probs: bool = False, ring_blocks: int = 0):
    """Exact attention of query rows ``q`` (bf16 bits ``[rows, H, d]``).
    Returns ``(out fp64 [rows,H,d], lse fp64 [rows,H])`` and, with ``want_probs``,
    the weights ``fp64 [rows, H, max_len]`` (zero outside each row's key set).
    ``ring_blocks``: as for ``quant_append``; a key whose page is not among the
    sequence's R most recent raises ValueError."""
    lib = _load()
    q = np.ascontiguousarray(q, np.uint16)
    rows, H, d = q.shape
    assert d == cache.head_dim
    bt = np.ascontiguousarray(block_table, np.int32)
    sl = np.ascontiguousarray(seq_lens, np.int32)
    rs = np.ascontiguousarray(row_seq, np.int32)
    rp = np.ascontiguousarray(row_pos, np.int32)
    out = np.zeros((rows, H, d), np.float64)
    lse = np.zeros((rows, H), np.float64)
    max_keys = int(rp.max()) + 1 if rows else 1
    scratch = np.empty(max_keys * H + (H + 1) * d, np.float64)
    probs = None
    stride = 0
    if want_probs:
        stride = int(sl.max())
        probs = np.zeros((rows, H, stride), np.float64)
    kb, ke = key_range if key_range is not None else (0, -1)
    rc = lib.oracle_attention(_p(cache.k_codes), _p(cache.v_codes), _p(cache.k_scale),
                              _p(cache.v_scale), cache.num_blocks, cache.page_size, d,
                              _p(bt), bt.shape[1], _p(sl), sl.shape[0], H, _p(q), rows,
                              _p(rs), _p(rp), int(window), float(sm_scale), int(kb), int(ke),
                              _p(out), _p(lse), _p(probs) if probs is not None else None,
                              stride, _p(scratch), int(ring_blocks))
    if rc != 0:
        raise ValueError("oracle_attention: index out of range")
    return (out, lse, probs) if want_probs else (out, lse)


def decode(cache: Cache, block_table, seq_lens, q, window: int, sm_scale: float,
           seqs: np.ndarray | None = None, ring_blocks: int = 0):
    """Decode: the query of sequence b (``q[b]``, bf16 bits ``[B, H, d]``) sits at
    position ``seq_lens[b]-1``.  ``seqs`` restricts to a subset of sequences."""
    sl = np.asarray(seq_lens, np.int32)
    seqs = np.arange(sl.shape[0]) if seqs is None else np.asarray(seqs)
    qq = np.ascontiguousarray(np.asarray(q)[seqs])
    return attention(cache, block_table, sl, qq, seqs.astype(np.int32),
                     (sl[seqs] - 1).astype(np.int32), window, sm_scale, ring_blocks=ring_blocks)


def prefill_rows(cu_q: np.ndarray, seq_lens: np.ndarray):
    """Row -> (sequence, absolute position) for a ragged chunk of new queries:
    the q_len = cu_q[b+1]-cu_q[b] queries of sequence b are its last q_len
    positions."""
    cu = np.asarray(cu_q, np.int64)
    sl = np.asarray(seq_lens, np.int64)
    rows = int(cu[-1])
    row_seq = np.empty(rows, np.int32)
    row_pos = np.empty(rows, np.int32)
    for b in range(len(sl)):
        n = cu[b + 1] - cu[b]
        row_seq[cu[b]:cu[b + 1]] = b
        row_pos[cu[b]:cu[b + 1]] = np.arange(sl[b] - n, sl[b])
    return row_seq, row_pos


def combine(parts: np.ndarray, part_lse: np.ndarray):
    """Merge partials ``parts [S, n, d]`` with ``part_lse [S, n]`` (fp64)."""
    lib = _load()
    parts = np.ascontiguousarray(parts, np.float64)
    part_lse = np.ascontiguousarray(part_lse, np.float64)
    S, n, d = parts.shape
    out = np.zeros((n, d), np.float64)
    lse = np.zeros(n, np.float64)
    lib.oracle_combine(_p(parts), _p(part_lse), S, n, d, _p(out), _p(lse))
    return out, lse
