"""The five synthetic workloads (shapes, length mixes and seeds) used by the
tests and the benchmark.  Pure data: no attention arithmetic here."""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    head_dim: int
    page_size: int
    len_kind: str            # "fixed" | "uniform" | "lognormal" | "prefix"
    len_values: tuple
    windows: tuple           # per layer: 0 = global, >0 = local window
    num_caches: int
    layer_map: tuple         # layer -> cache index
    shuffle: bool
    seed: int
    groups: int = 0          # prefix-sharing groups (prefill workload)
    new_tokens: int = 0      # tokens appended per sequence (prefill workload)

    @property
    def num_layers(self) -> int:
        return len(self.windows)


def layer_kinds(num_layers: int, period: int = 6) -> list[bool]:
    """True where the layer is global: one layer in ``period``, the last of each group."""
    return [(l % period) == period - 1 for l in range(num_layers)]


def layer_to_cache_map(num_layers: int, period: int = 6) -> tuple[list[int], int]:
    """Adjacent-layer cache sharing for a local/global stack.

    Local layers are paired consecutively in local order; global layers are
    paired consecutively among the globals (so globals are tied across blocks).
    Local pairs get cache ids 0..n_local_pairs-1, global pairs the ids after.
    """
    kinds = layer_kinds(num_layers, period)
    locals_ = [l for l in range(num_layers) if not kinds[l]]
    globals_ = [l for l in range(num_layers) if kinds[l]]
    m = [-1] * num_layers
    cid = 0
    for i in range(0, len(locals_), 2):
        for l in locals_[i:i + 2]:
            m[l] = cid
        cid += 1
    for i in range(0, len(globals_), 2):
        for l in globals_[i:i + 2]:
            m[l] = cid
        cid += 1
    return m, cid


_MAP24, _NC24 = layer_to_cache_map(24)

CONFIGS: dict[str, Workload] = {
    # Tiny MQA decode: 4 sequences, 8 heads, d=64, page 16, identity table.
    "tiny": Workload(
        name="tiny", batch=4, num_q_heads=8, head_dim=64, page_size=16,
        len_kind="fixed", len_values=(17, 100, 250, 512),
        windows=(128, 0), num_caches=2, layer_map=(0, 1), shuffle=False, seed=0),
    # Single local layer: batch 64, ragged 1k-8k context, window 1024.
    "local_b64": Workload(
        name="local_b64", batch=64, num_q_heads=32, head_dim=128, page_size=64,
        len_kind="uniform", len_values=(1024, 8192),
        windows=(1024,), num_caches=1, layer_map=(0,), shuffle=True, seed=2),
    # Single global layer, long context: batch 8, 32k-128k, split-KV.
    "global_long_b8": Workload(
        name="global_long_b8", batch=8, num_q_heads=32, head_dim=128, page_size=64,
        len_kind="uniform", len_values=(32768, 131072),
        windows=(0,), num_caches=1, layer_map=(0,), shuffle=True, seed=3),
    # Full decode step of a 24-layer local/global stack with 12 shared caches.
    "stack24_b128": Workload(
        name="stack24_b128", batch=128, num_q_heads=32, head_dim=128, page_size=64,
        len_kind="lognormal", len_values=(4096, 1.0, 32768),
        windows=tuple(0 if g else 1024 for g in layer_kinds(24)),
        num_caches=_NC24, layer_map=tuple(_MAP24), shuffle=True, seed=4),
    # Prefix-reuse chunked prefill: 32 groups x 8 sequences share an 8k prefix,
    # each appends 512 tokens; run once local (1024) and once global.
    "prefix_prefill": Workload(
        name="prefix_prefill", batch=256, num_q_heads=32, head_dim=128, page_size=64,
        len_kind="prefix", len_values=(8192, 512),
        windows=(1024, 0), num_caches=1, layer_map=(0, 0), shuffle=True, seed=5,
        groups=32, new_tokens=512),
}
