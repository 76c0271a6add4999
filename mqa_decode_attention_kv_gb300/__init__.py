"""Python binding of libmqa_kv (int8 paged multi-query attention for GB300).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libmqa_kv.so`` behind the C ABI declared in ``include/mqa_kv.h``.
PyTorch supplies device memory and the current CUDA stream.  There is no CPU
fallback: if the library is not built, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmqa_kv.so")

MQA_OK = 0
MQA_ERR_INVALID_ARG = -1
MQA_ERR_UNSUPPORTED = -2
MQA_ERR_WORKSPACE = -3
MQA_ERR_CUDA = -4
MQA_DEV_BAD_BLOCK = 1
MQA_DEV_BAD_SEQLEN = 2
MQA_DEV_BAD_CU = 4
MQA_DEV_TIMEOUT = 8
MQA_MAX_SPLITS = 1024

EXPORTED = ("kv_quant_append", "mqa_decode_attn", "mqa_decode_auto_splits", "mqa_decode_workspace_size",
            "split_kv_combine", "mqa_prefill_attn", "mqa_prefill_workspace_size", "mqa_status_str",
            "mqa_decode_attn_noalloc",
            "mqa_pc_create", "mqa_pc_destroy", "mqa_pc_match", "mqa_pc_insert", "mqa_pc_offload",
            "mqa_pc_upload", "mqa_pc_stats")


class MQAError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {status_str(status)} ({status})")
        self.status = status


class _Cache(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


class _Batch(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
                ("seq_lens_host", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("max_seq_len", ctypes.c_int32),
                ("ring_blocks", ctypes.c_int32)]


_lib_handle = None


def declare(L: ctypes.CDLL) -> ctypes.CDLL:
    """Set the argument and return types of every entry point on a loaded
    libmqa_kv handle (64-bit pointers must never pass as default C ints)."""
    P, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    L.kv_quant_append.argtypes = [P, P, P, i32, P, P, P, P]
    L.kv_quant_append.restype = ctypes.c_int
    L.mqa_decode_attn.argtypes = [P, i32, P, i32, i32, i32, P, P, P, i32, ctypes.c_float, i32, P, sz, P, P]
    L.mqa_decode_attn.restype = ctypes.c_int
    L.mqa_decode_auto_splits.argtypes = [P, i32, i32, i32, i32]
    L.mqa_decode_auto_splits.restype = ctypes.c_int
    L.mqa_decode_workspace_size.argtypes = [i32, i32, i32, i32]
    L.mqa_decode_workspace_size.restype = sz
    L.split_kv_combine.argtypes = [P, P, i32, i32, i32, i32, P, P]
    L.split_kv_combine.restype = ctypes.c_int
    L.mqa_prefill_attn.argtypes = [P, i32, P, i32, i32, i32, P, P, i32, i32, P, P, i32, ctypes.c_float, P, sz,
                                   P, P]
    L.mqa_prefill_attn.restype = ctypes.c_int
    L.mqa_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    L.mqa_prefill_workspace_size.restype = sz
    L.mqa_decode_attn_noalloc.argtypes = [P, i32, P, i32, i32, i32, P, P, P, i32, ctypes.c_float, i32, P, P]
    L.mqa_decode_attn_noalloc.restype = ctypes.c_int
    L.mqa_status_str.argtypes = [ctypes.c_int]
    L.mqa_status_str.restype = ctypes.c_char_p
    i64 = ctypes.c_int64
    L.mqa_pc_create.argtypes = [i32, i32, i32, i64, i32, P]
    L.mqa_pc_create.restype = ctypes.c_int
    L.mqa_pc_destroy.argtypes = [P]
    L.mqa_pc_destroy.restype = None
    L.mqa_pc_match.argtypes = [P, P, i64, P, i64]
    L.mqa_pc_match.restype = i64
    L.mqa_pc_insert.argtypes = [P, P, i64, P, P, i64]
    L.mqa_pc_insert.restype = i64
    L.mqa_pc_offload.argtypes = [P, P, i32, P, P, i64, P]
    L.mqa_pc_offload.restype = ctypes.c_int
    L.mqa_pc_upload.argtypes = [P, P, i32, P, P, i64, P]
    L.mqa_pc_upload.restype = ctypes.c_int
    L.mqa_pc_stats.argtypes = [P, P]
    L.mqa_pc_stats.restype = ctypes.c_int
    return L


def lib() -> ctypes.CDLL:
    """Load libmqa_kv.so (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m mqa_decode_attention_kv_gb300.build`")
        _lib_handle = declare(ctypes.CDLL(LIB_PATH))
    return _lib_handle


def status_str(status: int) -> str:
    return lib().mqa_status_str(int(status)).decode()


def _check(fn: str, rc: int) -> None:
    if rc != MQA_OK:
        raise MQAError(fn, rc)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return int(t.data_ptr())


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


@dataclass
class KVCache:
    """One physical int8 KV cache (one shared K/V head) in device memory."""

    k_codes: "object"  # torch.int8 [num_blocks, page_size, head_dim]
    v_codes: "object"
    k_scale: "object"  # torch.float32 [num_blocks, page_size]
    v_scale: "object"

    @classmethod
    def empty(cls, num_blocks: int, page_size: int, head_dim: int, device="cuda") -> "KVCache":
        import torch
        return cls(torch.zeros((num_blocks, page_size, head_dim), dtype=torch.int8, device=device),
                   torch.zeros((num_blocks, page_size, head_dim), dtype=torch.int8, device=device),
                   torch.zeros((num_blocks, page_size), dtype=torch.float32, device=device),
                   torch.zeros((num_blocks, page_size), dtype=torch.float32, device=device))

    @property
    def num_blocks(self) -> int:
        return int(self.k_codes.shape[0])

    @property
    def page_size(self) -> int:
        return int(self.k_codes.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.k_codes.shape[2])

    def c(self) -> _Cache:
        return _Cache(_ptr(self.k_codes), _ptr(self.v_codes), _ptr(self.k_scale), _ptr(self.v_scale),
                      self.num_blocks, self.page_size, self.head_dim)


@dataclass
class Batch:
    """A ragged batch over paged caches: device block table and lengths plus a
    host copy of the lengths (used for validation and split planning)."""

    block_table: "object"        # torch.int32 [batch, max_blocks] (device)
    seq_lens: "object"           # torch.int32 [batch] (device)
    seq_lens_host: np.ndarray | None
    max_seq_len: int
    ring_blocks: int = 0         # > 0: window-bounded cache, page i in table entry i % ring_blocks

    @classmethod
    def from_host(cls, block_table: np.ndarray, seq_lens: np.ndarray, device="cuda",
                  with_host_lens: bool = True, max_seq_len: int | None = None,
                  ring_blocks: int = 0) -> "Batch":
        import torch
        bt = torch.from_numpy(np.ascontiguousarray(block_table, np.int32)).to(device)
        sl_np = np.ascontiguousarray(seq_lens, np.int32)
        sl = torch.from_numpy(sl_np).to(device)
        mx = int(sl_np.max()) if max_seq_len is None else int(max_seq_len)
        return cls(bt, sl, sl_np.copy() if with_host_lens else None, mx, int(ring_blocks))

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    def c(self) -> _Batch:
        host = None
        if self.seq_lens_host is not None:
            self._host_keep = np.ascontiguousarray(self.seq_lens_host, np.int32)
            host = self._host_keep.ctypes.data
        return _Batch(_ptr(self.block_table), _ptr(self.seq_lens), host, self.batch,
                      int(self.block_table.shape[1]), int(self.max_seq_len), int(self.ring_blocks))


def _caches_array(caches: Sequence[KVCache]):
    arr = (_Cache * len(caches))(*[c.c() for c in caches])
    return arr


def kv_quant_append(cache: KVCache, batch: Batch, cu_new, num_new_tokens: int, k_new, v_new,
                    dev_status=None, stream=None) -> None:
    """Quantise ``k_new``/``v_new`` (bf16 [T, d]) and store them at the last
    ``cu_new[b+1]-cu_new[b]`` positions of each sequence."""
    c = cache.c()
    bt = batch.c()
    rc = lib().kv_quant_append(ctypes.byref(c), ctypes.byref(bt), _ptr(cu_new), int(num_new_tokens),
                               _ptr(k_new), _ptr(v_new), _ptr(dev_status), _stream(stream))
    _check("kv_quant_append", rc)


def mqa_decode_workspace_size(batch: int, num_q_heads: int, head_dim: int, num_splits: int) -> int:
    return int(lib().mqa_decode_workspace_size(batch, num_q_heads, head_dim, num_splits))


def mqa_decode_auto_splits(batch: Batch, window: int, num_q_heads: int, head_dim: int, page_size: int) -> int:
    bt = batch.c()
    rc = lib().mqa_decode_auto_splits(ctypes.byref(bt), int(window), int(num_q_heads), int(head_dim),
                                      int(page_size))
    if rc < 0:
        raise MQAError("mqa_decode_auto_splits", rc)
    return int(rc)


def mqa_decode_attn(caches: Sequence[KVCache], layer_to_kv: Sequence[int], layer: int, window: int,
                    batch: Batch, q, out=None, sm_scale: float | None = None, num_splits: int = 0,
                    workspace=None, dev_status=None, stream=None):
    """Decode attention of layer ``layer`` (reads cache ``layer_to_kv[layer]``).
    ``q``: bf16 [batch, num_q_heads, head_dim].  Returns ``out``."""
    import torch
    B, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    cache = caches[layer_to_kv[layer]]
    splits = num_splits if num_splits > 0 else mqa_decode_auto_splits(batch, window, H, D, cache.page_size)
    if workspace is None and splits > 1:
        workspace = torch.empty(mqa_decode_workspace_size(B, H, D, splits), dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    carr = _caches_array(caches)
    lmap = (ctypes.c_int32 * len(layer_to_kv))(*layer_to_kv)
    bt = batch.c()
    rc = lib().mqa_decode_attn(carr, len(caches), lmap, len(layer_to_kv), int(layer), int(window),
                               ctypes.byref(bt), _ptr(q), _ptr(out), int(H), float(sm_scale), int(splits),
                               _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check("mqa_decode_attn", rc)
    return out


def split_kv_combine(o_partial, lse, out=None, stream=None):
    """Merge fp32 partials [batch, splits, heads, d] with lse [batch, splits, heads]."""
    import torch
    B, S, H, D = o_partial.shape
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=o_partial.device)
    rc = lib().split_kv_combine(_ptr(o_partial), _ptr(lse), B, S, H, D, _ptr(out), _stream(stream))
    _check("split_kv_combine", rc)
    return out


def mqa_prefill_workspace_size(batch: int, max_seq_len: int, window: int, max_q_len: int, head_dim: int) -> int:
    return int(lib().mqa_prefill_workspace_size(batch, max_seq_len, window, max_q_len, head_dim))


def mqa_prefill_attn(caches: Sequence[KVCache], layer_to_kv: Sequence[int], layer: int, window: int,
                     batch: Batch, cu_q, q, max_q_len: int, out=None, sm_scale: float | None = None,
                     workspace=None, dev_status=None, stream=None):
    """Causal prefill attention of the ``cu_q``-described new tokens (bf16 q
    [total_q, num_q_heads, head_dim]).  ``workspace`` (uint8, on the device)
    is allocated for the call when not given.  Returns ``out``."""
    import torch
    T, H, D = q.shape
    if out is None:
        out = torch.empty_like(q)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(D)
    need = mqa_prefill_workspace_size(batch.batch, batch.max_seq_len, window, max_q_len, D)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    carr = _caches_array(caches)
    lmap = (ctypes.c_int32 * len(layer_to_kv))(*layer_to_kv)
    bt = batch.c()
    rc = lib().mqa_prefill_attn(carr, len(caches), lmap, len(layer_to_kv), int(layer), int(window),
                                ctypes.byref(bt), _ptr(cu_q), int(T), int(max_q_len), _ptr(q), _ptr(out),
                                int(H), float(sm_scale), _ptr(workspace),
                                0 if workspace is None else workspace.numel() * workspace.element_size(),
                                _ptr(dev_status), _stream(stream))
    _check("mqa_prefill_attn", rc)
    return out


class PrefixCache:
    """Host-memory prefix cache (mqa_prefix_cache.h): whole pages of every cache
    of a layer stack, in a prefix tree keyed by a rolling hash of the tokens,
    with LRU eviction of leaf pages.  ``pinned=False`` keeps only the tree
    bookkeeping (no GPU needed; offload and upload are refused)."""

    def __init__(self, page_size: int, head_dim: int, num_caches: int, host_pages: int, pinned: bool = True):
        h = ctypes.c_void_p()
        _check("mqa_pc_create", lib().mqa_pc_create(int(page_size), int(head_dim), int(num_caches),
                                                    int(host_pages), int(bool(pinned)), ctypes.byref(h)))
        self._h = h
        self.page_size, self.head_dim, self.num_caches = int(page_size), int(head_dim), int(num_caches)

    def close(self) -> None:
        if self._h is not None and self._h.value:
            lib().mqa_pc_destroy(self._h)
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def match(self, tokens: np.ndarray) -> np.ndarray:
        """Slots of the longest cached whole-page prefix of ``tokens`` (int32)."""
        t = np.ascontiguousarray(tokens, np.int32)
        cap = len(t) // self.page_size
        slots = np.zeros(max(cap, 1), np.int64)
        k = lib().mqa_pc_match(self._h, t.ctypes.data, len(t), slots.ctypes.data, cap)
        if k < 0:
            raise MQAError("mqa_pc_match", int(k))
        return slots[:k].copy()

    def insert(self, tokens: np.ndarray):
        """Insert the whole pages of ``tokens``; returns (page indices, slots) of
        the pages that are new (to be filled with ``offload``)."""
        t = np.ascontiguousarray(tokens, np.int32)
        cap = len(t) // self.page_size
        idx = np.zeros(max(cap, 1), np.int64)
        slots = np.zeros(max(cap, 1), np.int64)
        n = lib().mqa_pc_insert(self._h, t.ctypes.data, len(t), idx.ctypes.data, slots.ctypes.data, cap)
        if n < 0:
            raise MQAError("mqa_pc_insert", int(n))
        return idx[:n].copy(), slots[:n].copy()

    def offload(self, caches, src_blocks, slots, stream=None) -> None:
        """Device blocks -> pool slots (every cache), enqueued on ``stream``."""
        b = np.ascontiguousarray(src_blocks, np.int32)
        sl = np.ascontiguousarray(slots, np.int64)
        assert len(b) == len(sl)
        _check("mqa_pc_offload", lib().mqa_pc_offload(self._h, _caches_array(caches), len(caches), b.ctypes.data,
                                                      sl.ctypes.data, len(b), _stream(stream)))

    def upload(self, caches, slots, dst_blocks, stream=None) -> None:
        """Pool slots -> device blocks (every cache), enqueued on ``stream``."""
        b = np.ascontiguousarray(dst_blocks, np.int32)
        sl = np.ascontiguousarray(slots, np.int64)
        assert len(b) == len(sl)
        _check("mqa_pc_upload", lib().mqa_pc_upload(self._h, _caches_array(caches), len(caches), sl.ctypes.data,
                                                    b.ctypes.data, len(b), _stream(stream)))

    def stats(self) -> dict:
        out = np.zeros(8, np.int64)
        _check("mqa_pc_stats", lib().mqa_pc_stats(self._h, out.ctypes.data))
        keys = ("cached_pages", "free_slots", "capacity", "match_calls", "pages_matched", "pages_inserted",
                "pages_evicted", "slot_bytes")
        return dict(zip(keys, (int(x) for x in out)))
