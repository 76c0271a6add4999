"""Shared set-up for the GPU parity tests: build identical caches on the GPU
(through kv_quant_append) and in the oracle, from the same seeded bf16 inputs."""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

import oracle
import synth
import mqa_decode_attention_kv_gb300 as mk

# tolerances for attention outputs (bf16 result vs fp64 oracle)
MAX_ABS = 1e-2
REL_L2 = 5e-3


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev_i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) around |x|: the
    largest error of rounding the exact value to the bf16 output."""
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def abs_tolerance(ref: np.ndarray) -> np.ndarray:
    """Per-element max-abs bound: MAX_ABS, plus bf16's own half-ulp where
    |ref| >= 4.  There the output format alone (half-ulp 0.0156 on [4, 8))
    cannot meet 1e-2; below 4 its half-ulp is at most 0.0078 and the bound is
    the plain 1e-2."""
    return MAX_ABS + np.where(np.abs(ref) >= 4.0, bf16_half_ulp(ref), 0.0)


def errors(gpu_out: torch.Tensor, ref: np.ndarray):
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    diff = g - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(diff) / den) if den > 0 else float(np.linalg.norm(diff))
    return max_abs, rel, float(np.abs(ref).max()) if ref.size else 0.0


def assert_close(gpu_out, ref, what=""):
    max_abs, rel, ref_max = errors(gpu_out, ref)
    assert np.isfinite(max_abs), f"{what}: non-finite output"
    g = gpu_out.float().cpu().numpy().astype(np.float64)
    excess = float((np.abs(g - ref) - abs_tolerance(ref)).max()) if ref.size else 0.0
    assert excess <= 0.0 and rel <= REL_L2, \
        f"{what}: max_abs={max_abs:.3e} (over the bound by {excess:.3e}) rel_l2={rel:.3e} (max|ref|={ref_max:.3f})"
    return max_abs, rel


@dataclass
class Setup:
    seq_lens: np.ndarray
    pb: synth.PagedBatch
    head_dim: int
    gpu_caches: list
    ora_caches: list
    batch: mk.Batch
    kv_bits: list  # per cache (k, v) bf16 bits [sum L, d]


def build_caches(rng, seq_lens, page_size, head_dim, num_caches, shuffle=True, with_host_lens=True,
                 pb: synth.PagedBatch | None = None, kv_scale: float = 1.0, kv_bits=None) -> Setup:
    """Caches filled by kv_quant_append (GPU) and the oracle's quantiser (CPU) from the
    same bf16 K/V rows: N(0, kv_scale^2) draws, or kv_bits[c] = (k, v) when given."""
    seq_lens = np.asarray(seq_lens, np.int32)
    pb = pb or synth.make_paged_batch(rng, seq_lens, page_size, shuffle=shuffle)
    cu = synth.cu_from_counts(seq_lens)
    T = int(cu[-1])
    batch = mk.Batch.from_host(pb.block_table, seq_lens, with_host_lens=with_host_lens)
    cu_dev = to_dev_i32(cu)
    gpu, ora, bits = [], [], []
    for c in range(num_caches):
        if kv_bits is not None:
            k, v = kv_bits[c]
        else:
            k = synth.bf16_normal(rng, (T, head_dim), kv_scale)
            v = synth.bf16_normal(rng, (T, head_dim), kv_scale)
        gc = mk.KVCache.empty(pb.num_blocks, page_size, head_dim)
        mk.kv_quant_append(gc, batch, cu_dev, T, to_dev_bf16(k), to_dev_bf16(v))
        oc = oracle.Cache.empty(pb.num_blocks, page_size, head_dim)
        oracle.quant_append(oc, pb.block_table, seq_lens, cu, k, v)
        gpu.append(gc)
        ora.append(oc)
        bits.append((k, v))
    torch.cuda.synchronize()
    return Setup(seq_lens, pb, head_dim, gpu, ora, batch, bits)


def caches_equal(gc: mk.KVCache, oc: oracle.Cache) -> bool:
    return (np.array_equal(gc.k_codes.cpu().numpy(), oc.k_codes)
            and np.array_equal(gc.v_codes.cpu().numpy(), oc.v_codes)
            and np.array_equal(gc.k_scale.cpu().numpy().view(np.uint32), oc.k_scale.view(np.uint32))
            and np.array_equal(gc.v_scale.cpu().numpy().view(np.uint32), oc.v_scale.view(np.uint32)))


def sm_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)
