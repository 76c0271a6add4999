"""Benchmark of the int8 paged MQA serving hot path on one (or N replica) GPUs.

Default workload (one "step"): a full decode step of a 24-layer local/global
stack -- 20 local layers (window 1024) and 4 global layers, 12 caches shared by
adjacent layers, batch 128, 32 query heads, d=128, context lengths lognormal
(median 4096, cap 32768), int8 paged KV with page 64.  A step appends the new
token of every sequence to each of the 12 caches (kv_quant_append) and runs
the 24 decode-attention calls in layer order (split-KV + combine where the
planner chooses it).  Other workloads (--workload) time a single local layer,
a single long-context global layer, or the prefix-reuse chunked prefill.

Prints ONE JSON line (rank 0): the step's decode tokens/s as `value`, the
decode kernel's HBM roofline (every call timed alone with L2 flushed before it),
the same step through the public Python API with host buffers (`e2e`), and the
CPU oracle's rate on a bounded sample of the workload (`cpu_baseline`).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402
from mqa_decode_attention_kv_gb300 import accounting as acc  # noqa: E402

METRIC = "decode-attention KV GB/s (frac of HBM peak) and decode tokens/s on 1 GB300"
L2_FLUSH_BYTES = 512 << 20  # > 2x the 129 MB L2


# ---------------------------------------------------------------- helpers
def rank_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def source_digest(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profile_traffic(name: str, digest: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/<name>,
    used only if the kernel sources still match the digest recorded there."""
    p = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(p):
        return None
    vals = {}
    for line in open(p):
        parts = line.split()
        if len(parts) >= 2 and not line.startswith("#"):
            vals[parts[0]] = parts[1]
    if vals.get("source_digest") != digest or "dram_bytes_per_launch" not in vals:
        return None
    return float(vals["dram_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU workloads
class DecodeStack:
    """Caches, inputs and pre-marshalled C-ABI arguments of a decode step.
    ring_local: caches read only by local layers are window-bounded rings of
    (W-1)/P + 2 pages per sequence (page p in table entry p % R); the global
    caches keep full tables."""

    def __init__(self, w: "synth.Workload", device, ring_local: bool = False):
        import ctypes
        import torch
        import mqa_decode_attention_kv_gb300 as mk
        self.w, self.mk, self.torch = w, mk, torch
        rng = np.random.default_rng(w.seed)
        self.lens = synth.seq_lens_for(w, rng)
        self.pb = synth.make_paged_batch(rng, self.lens, w.page_size, shuffle=w.shuffle)
        self.batch = mk.Batch.from_host(self.pb.block_table, self.lens, device=device)
        B, H, D, P = w.batch, w.num_q_heads, w.head_dim, w.page_size
        gen = torch.Generator(device=device)
        gen.manual_seed(1000 + w.seed)
        T = int(self.lens.sum())
        cu_all = torch.from_numpy(synth.cu_from_counts(self.lens)).to(device)
        # which caches are read by local layers only (candidates for rings)
        local_only = [all(w.windows[l] > 0 for l in range(w.num_layers) if w.layer_map[l] == c)
                      for c in range(w.num_caches)]
        self.ring = 0
        self.ring_batch = None
        self.cache_is_ring = [False] * w.num_caches
        if ring_local and any(local_only):
            wmax = max(w.windows[l] for l in range(w.num_layers) if local_only[w.layer_map[l]])
            self.ring = (wmax - 1) // P + 2
            table = rng.permutation(B * self.ring).astype(np.int32).reshape(B, self.ring)
            self.ring_batch = mk.Batch.from_host(table, self.lens, device=device, ring_blocks=self.ring)
            self.cache_is_ring = list(local_only)
            # the resident tokens of each sequence: its last pages, at most ring pages
            first_res = np.maximum(0, ((self.lens.astype(np.int64) - 1) // P - (self.ring - 1)) * P)
            res_counts = (self.lens - first_res).astype(np.int64)
            cu_res = torch.from_numpy(synth.cu_from_counts(res_counts)).to(device)
            T_res = int(res_counts.sum())
            cu_host = synth.cu_from_counts(self.lens)
            res_rows = torch.from_numpy(np.concatenate([np.arange(int(cu_host[b + 1]) - int(res_counts[b]),
                                                                  int(cu_host[b + 1])) for b in range(B)])).to(device)
        self.caches = []
        for c_i in range(w.num_caches):
            k = torch.randn((T, D), generator=gen, device=device).to(torch.bfloat16)
            v = torch.randn((T, D), generator=gen, device=device).to(torch.bfloat16)
            if self.cache_is_ring[c_i]:
                c = mk.KVCache.empty(B * self.ring, P, D, device=device)
                mk.kv_quant_append(c, self.ring_batch, cu_res, T_res, k[res_rows].contiguous(),
                                   v[res_rows].contiguous())
            else:
                c = mk.KVCache.empty(self.pb.num_blocks, P, D, device=device)
                mk.kv_quant_append(c, self.batch, cu_all, T, k, v)
            del k, v
            self.caches.append(c)
        self.pool_bytes = sum(c.k_codes.numel() * 2 + c.k_scale.numel() * 8 for c in self.caches)
        self.full_pool_bytes = w.num_caches * self.pb.num_blocks * P * 2 * (D + 4)
        L = w.num_layers
        self.q = torch.randn((L, B, H, D), generator=gen, device=device).to(torch.bfloat16)
        self.k_new = torch.randn((w.num_caches, B, D), generator=gen, device=device).to(torch.bfloat16)
        self.v_new = torch.randn((w.num_caches, B, D), generator=gen, device=device).to(torch.bfloat16)
        self.out = torch.empty_like(self.q)
        self.cu_step = torch.arange(B + 1, dtype=torch.int32, device=device)
        self.splits = [mk.mqa_decode_auto_splits(self.batch_of_layer(l), w.windows[l], H, D, P) for l in range(L)]
        ws = max(mk.mqa_decode_workspace_size(B, H, D, s) for s in self.splits)
        self.ws = torch.empty(max(ws, 16), dtype=torch.uint8, device=device)
        # device-side error bits of every call (bad inputs, a bounded wait that ran out)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        first = {}
        for l, c in enumerate(w.layer_map):
            first.setdefault(c, l)
        self.append_before = {l: c for c, l in first.items()}  # layer -> cache appended just before it
        # pre-marshalled arguments (same C ABI the binding uses, without per-call Python work)
        self._carr = mk._caches_array(self.caches)
        self._lmap = (ctypes.c_int32 * L)(*w.layer_map)
        self._bt = self.batch.c()
        self._bt_ring = self.ring_batch.c() if self.ring_batch is not None else None
        self._cptr = [ctypes.byref(self._carr[i]) for i in range(len(self.caches))]
        self.scale = 1.0 / math.sqrt(D)
        self.lib = mk.lib()
        self.bytes_per_layer = [acc.decode_kv_bytes(self.lens, w.windows[l], D) for l in range(L)]
        self.flops_per_layer = [acc.decode_flops(self.lens, w.windows[l], H, D) for l in range(L)]

    def batch_of_cache(self, c: int):
        return self.ring_batch if self.cache_is_ring[c] else self.batch

    def batch_of_layer(self, l: int):
        return self.batch_of_cache(self.w.layer_map[l])

    def _bt_of_cache(self, c: int):
        return self._bt_ring if self.cache_is_ring[c] else self._bt

    def launches_per_step(self) -> int:
        return len(self.append_before) + sum(2 if s > 1 else 1 for s in self.splits)

    def append(self, c: int, stream: int):
        B = self.w.batch
        import ctypes
        rc = self.lib.kv_quant_append(self._cptr[c], ctypes.byref(self._bt_of_cache(c)), self.cu_step.data_ptr(), B,
                                      self.k_new[c].data_ptr(), self.v_new[c].data_ptr(), None, stream)
        assert rc == 0, rc

    def attend(self, l: int, stream: int):
        import ctypes
        w = self.w
        rc = self.lib.mqa_decode_attn(self._carr, len(self.caches), self._lmap, w.num_layers, l, w.windows[l],
                                      ctypes.byref(self._bt_of_cache(w.layer_map[l])), self.q[l].data_ptr(),
                                      self.out[l].data_ptr(),
                                      w.num_q_heads, self.scale, self.splits[l], self.ws.data_ptr(),
                                      self.ws.numel(), ctypes.c_void_p(self.status.data_ptr()), stream)
        assert rc == 0, rc

    def step(self, stream: int):
        for l in range(self.w.num_layers):
            c = self.append_before.get(l)
            if c is not None:
                self.append(c, stream)
            self.attend(l, stream)


def flush_l2(buf):
    """Evict L2 by reading a buffer larger than it (a read leaves no dirty lines
    whose write-back would be charged to the next timed kernel)."""
    buf.sum(dtype=torch_int64())


def torch_int64():
    import torch
    return torch.int64


def time_steps(fn, steps, flush_buf, stream):
    """Per-step device time (ms) with CUDA events on `stream`, L2 flushed
    before every step (outside the timed intervals); flush_buf None = no flush
    (back-to-back steps: what fits in L2 stays there)."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            if flush_buf is not None:
                flush_l2(flush_buf)
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
    stream.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def cold_layer_times(stack: DecodeStack, reps, flush_buf, stream):
    """Every layer of the step as its own timed segment with L2 flushed before
    it: the append of the cache it is the first to read (if any), then its
    decode call.  Returns ({layer: [segment ms]}, {layer: [decode-call ms]}):
    the sum of the segments is a step whose every layer reads its KV from HBM;
    the decode-call times are the per-launch HBM roofline measurement."""
    import torch
    sptr = stream.cuda_stream
    seg = {l: [] for l in range(stack.w.num_layers)}
    call = {l: [] for l in range(stack.w.num_layers)}
    evs = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            for l in range(stack.w.num_layers):
                flush_l2(flush_buf)
                e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
                e0.record(stream)
                c = stack.append_before.get(l)
                if c is not None:
                    stack.append(c, sptr)
                e1.record(stream)
                stack.attend(l, sptr)
                e2.record(stream)
                evs.append((l, e0, e1, e2))
    stream.synchronize()
    for l, e0, e1, e2 in evs:
        seg[l].append(e0.elapsed_time(e2))
        call[l].append(e1.elapsed_time(e2))
    return seg, call


def e2e_steps(stack: DecodeStack, steps, stream, graph: bool):
    """End-to-end step through the public Python API with host buffers: H2D of
    the step's queries and new K/V from pinned memory, the appends and 24
    attention calls, D2H of all outputs.  graph=True captures that whole
    sequence (copies included) once into a CUDA graph and replays it, as a
    serving loop would; graph=False issues it eagerly every step (the host's
    call overhead then shows).  Returns (per-step ms, h2d, d2h bytes, the copy groups)."""
    import torch
    mk = stack.mk
    w = stack.w
    q_host = stack.q.cpu().pin_memory()
    kn_host = stack.k_new.cpu().pin_memory()
    vn_host = stack.v_new.cpu().pin_memory()
    out_host = torch.empty(stack.out.shape, dtype=stack.out.dtype, pin_memory=True)
    q_dev = torch.empty_like(stack.q)
    kn_dev = torch.empty_like(stack.k_new)
    vn_dev = torch.empty_like(stack.v_new)
    out_dev = torch.empty_like(stack.out)
    h2d = (q_host.numel() + kn_host.numel() + vn_host.numel()) * 2
    d2h = out_host.numel() * 2

    copy_stream = torch.cuda.Stream(device=stack.q.device)

    def one_step_plain(s):
        q_dev.copy_(q_host, non_blocking=True)
        kn_dev.copy_(kn_host, non_blocking=True)
        vn_dev.copy_(vn_host, non_blocking=True)
        for l in range(w.num_layers):
            c = stack.append_before.get(l)
            if c is not None:
                mk.kv_quant_append(stack.caches[c], stack.batch_of_cache(c), stack.cu_step, w.batch, kn_dev[c],
                                   vn_dev[c], stream=s)
            mk.mqa_decode_attn(stack.caches, list(w.layer_map), l, w.windows[l], stack.batch_of_layer(l), q_dev[l],
                               out=out_dev[l], num_splits=stack.splits[l], workspace=stack.ws, stream=s)
        out_host.copy_(out_dev, non_blocking=True)

    # copies on their own stream, overlapping the layers, in few large copies: the queries in
    # growing groups of layers (1, 2, 4, ...; the first with the new K/V), each group arriving
    # while earlier layers run; the outputs in shrinking groups (half the layers left, then
    # half of the rest, ...), each leaving once its last layer is done, so only the last
    # layer's output is copied after the step's last kernel
    L = w.num_layers
    in_groups, a, n = [], 0, 1
    while a < L:
        in_groups.append((a, min(L, a + n)))
        a, n = in_groups[-1][1], 2 * n
    out_groups, a = [], 0
    while a < L:
        out_groups.append((a, a + (L - a + 1) // 2))
        a = out_groups[-1][1]
    out_after = {b - 1: (a, b) for a, b in out_groups}

    def one_step(s):
        cs = copy_stream
        cs.wait_stream(s)
        arrived = {}
        with torch.cuda.stream(cs):
            for gi, (a, b) in enumerate(in_groups):
                if gi == 0:
                    kn_dev.copy_(kn_host, non_blocking=True)
                    vn_dev.copy_(vn_host, non_blocking=True)
                q_dev[a:b].copy_(q_host[a:b], non_blocking=True)
                arrived[a] = torch.cuda.Event()
                arrived[a].record(cs)
        for l in range(L):
            if l in arrived:
                s.wait_event(arrived[l])
            c = stack.append_before.get(l)
            if c is not None:
                mk.kv_quant_append(stack.caches[c], stack.batch_of_cache(c), stack.cu_step, w.batch, kn_dev[c],
                                   vn_dev[c], stream=s)
            mk.mqa_decode_attn(stack.caches, list(w.layer_map), l, w.windows[l], stack.batch_of_layer(l), q_dev[l],
                               out=out_dev[l], num_splits=stack.splits[l], workspace=stack.ws, stream=s)
            if l in out_after:
                a, b = out_after[l]
                done = torch.cuda.Event()
                done.record(s)
                cs.wait_event(done)
                with torch.cuda.stream(cs):
                    out_host[a:b].copy_(out_dev[a:b], non_blocking=True)
        s.wait_stream(cs)

    run = None
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            one_step(stream)  # warm-up outside the capture
        stream.synchronize()
        with torch.cuda.graph(g, stream=stream):
            one_step(torch.cuda.current_stream())
        run = g.replay
    else:
        run = lambda: one_step_plain(stream)
    times = []
    with torch.cuda.stream(stream):
        for _ in range(steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            run()
            e1.record(stream)
            times.append((e0, e1))
    stream.synchronize()
    # the outputs that reached the host are the device path's, bit for bit (the kernels are
    # deterministic and every step appends the same tokens): a copy that went wrong fails here
    if not torch.equal(out_host.view(torch.int16), stack.out.cpu().view(torch.int16)):
        raise SystemExit("end-to-end outputs differ from the device path's")
    groups = "queries in groups of %s layers, outputs in groups of %s" % (
        ", ".join(str(b - a) for a, b in in_groups), ", ".join(str(b - a) for a, b in out_groups))
    return [a.elapsed_time(b) for a, b in times], h2d, d2h, groups


# ---------------------------------------------------------------- CPU oracle baseline
class OracleStack:
    """The oracle (single-threaded C, fp64) set up on a bounded, seeded sample of
    the workload's sequences: caches filled with their tokens, one query per
    layer and one new K/V token per cache."""

    def __init__(self, w: "synth.Workload", n_seqs: int, seed: int = 123):
        import oracle
        oracle.build()
        self.oracle, self.w = oracle, w
        rng = np.random.default_rng(w.seed)
        lens_all = synth.seq_lens_for(w, rng)
        pick = synth.sample_rows(np.random.default_rng(seed), len(lens_all), n_seqs)
        self.lens = lens_all[pick]
        self.pb = synth.make_paged_batch(rng, self.lens, w.page_size, shuffle=w.shuffle)
        cu = synth.cu_from_counts(self.lens)
        T = int(cu[-1])
        d, H = w.head_dim, w.num_q_heads
        self.caches = []
        for _ in range(w.num_caches):
            c = oracle.Cache.empty(self.pb.num_blocks, w.page_size, d)
            oracle.quant_append(c, self.pb.block_table, self.lens, cu, synth.bf16_normal(rng, (T, d)),
                                synth.bf16_normal(rng, (T, d)))
            self.caches.append(c)
        n = len(self.lens)
        self.q = [synth.bf16_normal(rng, (n, H, d)) for _ in range(w.num_layers)]
        self.kn = [synth.bf16_normal(rng, (n, d)) for _ in range(w.num_caches)]
        self.vn = [synth.bf16_normal(rng, (n, d)) for _ in range(w.num_caches)]
        self.cu_step = synth.cu_from_counts(np.ones(n))
        first = {}
        for l, c in enumerate(w.layer_map):
            first.setdefault(c, l)
        self.before = {l: c for c, l in first.items()}
        self.scale = 1.0 / math.sqrt(d)
        self.desc = (f"{n} of {w.batch} sequences (seeded sample, mean context {self.lens.mean():.0f}) "
                     f"through all {w.num_layers} layers; one decode token each")

    def step(self) -> float:
        """One decode step of the sample (appends + every layer); returns seconds."""
        w = self.w
        t0 = time.perf_counter()
        for l in range(w.num_layers):
            c = self.before.get(l)
            if c is not None:
                self.oracle.quant_append(self.caches[c], self.pb.block_table, self.lens, self.cu_step, self.kn[c],
                                         self.vn[c])
            self.oracle.decode(self.caches[w.layer_map[l]], self.pb.block_table, self.lens, self.q[l], w.windows[l],
                               self.scale)
        return time.perf_counter() - t0


def oracle_decode_sample(w: "synth.Workload", n_seqs: int, seed: int = 123):
    """Time one oracle step on a bounded sample of the workload: n_seqs
    sequences through every layer.  Returns (tokens/s, seconds, description)."""
    st = OracleStack(w, n_seqs, seed)
    dt = st.step()
    return len(st.lens) / dt, dt, st.desc


class PrefillWorkload:
    """Prefix-reuse chunked prefill: groups of sequences share int8 prefixes;
    each sequence appends its new tokens (kv_quant_append over all of them) and
    runs causal prefill attention over prefix + chunk, once with the local
    window and once globally (two single-layer runs on the same cache)."""

    def __init__(self, w: "synth.Workload", device):
        import ctypes
        import torch
        import mqa_decode_attention_kv_gb300 as mk
        self.w, self.mk = w, mk
        rng = np.random.default_rng(w.seed)
        prefix, new = w.len_values
        per = w.batch // w.groups
        pbs = synth.make_prefix_shared_batch(rng, w.groups, per, prefix, new, w.page_size)
        self.pbs = pbs
        self.lens = pbs.seq_lens
        self.q_lens = np.full(w.batch, new, np.int64)
        D, H = w.head_dim, w.num_q_heads
        gen = torch.Generator(device=device)
        gen.manual_seed(2000 + w.seed)
        self.cache = mk.KVCache.empty(pbs.num_blocks, w.page_size, D, device=device)
        leaders = np.arange(w.groups) * per
        lead = mk.Batch.from_host(np.ascontiguousarray(pbs.block_table[leaders]),
                                  np.full(w.groups, prefix, np.int32), device=device)
        Tp = w.groups * prefix
        cu_p = torch.from_numpy(synth.cu_from_counts([prefix] * w.groups)).to(device)
        mk.kv_quant_append(self.cache, lead, cu_p, Tp,
                           torch.randn((Tp, D), generator=gen, device=device).to(torch.bfloat16),
                           torch.randn((Tp, D), generator=gen, device=device).to(torch.bfloat16))
        self.batch = mk.Batch.from_host(pbs.block_table, self.lens, device=device)
        self.T = w.batch * new
        self.cu_q = torch.from_numpy(synth.cu_from_counts(self.q_lens)).to(device)
        self.k_new = torch.randn((self.T, D), generator=gen, device=device).to(torch.bfloat16)
        self.v_new = torch.randn((self.T, D), generator=gen, device=device).to(torch.bfloat16)
        self.q = torch.randn((self.T, H, D), generator=gen, device=device).to(torch.bfloat16)
        self.out = [torch.empty_like(self.q) for _ in w.windows]
        self.max_q = new
        # one workspace for every layer (the largest: the global layer's tile images)
        self.ws = torch.empty(max(16, max(mk.mqa_prefill_workspace_size(w.batch, self.batch.max_seq_len, W, new, D)
                                          for W in w.windows)), dtype=torch.uint8, device=device)
        self.lib = mk.lib()
        self._c = self.cache.c()
        self._carr = (mk._Cache * 1)(self._c)
        self._lmap = (ctypes.c_int32 * len(w.windows))(*w.layer_map)
        self._bt = self.batch.c()
        self.scale = 1.0 / math.sqrt(D)
        self.flops = [acc.prefill_flops(self.lens, self.q_lens, W, H, D) for W in w.windows]

    def append(self, stream: int):
        import ctypes
        rc = self.lib.kv_quant_append(ctypes.byref(self._c), ctypes.byref(self._bt), self.cu_q.data_ptr(), self.T,
                                      self.k_new.data_ptr(), self.v_new.data_ptr(), None, stream)
        assert rc == 0, rc

    def attend(self, l: int, stream: int):
        import ctypes
        w = self.w
        rc = self.lib.mqa_prefill_attn(self._carr, 1, self._lmap, len(w.windows), l, w.windows[l],
                                       ctypes.byref(self._bt), self.cu_q.data_ptr(), self.T, self.max_q,
                                       self.q.data_ptr(), self.out[l].data_ptr(), w.num_q_heads, self.scale,
                                       self.ws.data_ptr(), self.ws.numel(), None, stream)
        assert rc == 0, rc

    def step(self, stream: int):
        self.append(stream)
        for l in range(len(self.w.windows)):
            self.attend(l, stream)


def dist_setup(world, local_rank):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
        return dist
    return None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def reduce_max(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- main
def describe(w: "synth.Workload", lens) -> str:
    if w.name == "prefix_prefill":
        return (f"{w.name}: {w.groups} groups x {w.batch // w.groups} sequences sharing {w.len_values[0]}-token int8 "
                f"prefixes (shared blocks), {w.len_values[1]} new tokens each; kv_quant_append of all new tokens, "
                f"then causal MQA prefill with window {w.windows[0]} and global; {w.num_q_heads} q heads, "
                f"d={w.head_dim}, page {w.page_size}")
    n_glob = sum(1 for x in w.windows if x == 0)
    return (f"{w.name}: {w.num_layers}-layer decode step ({w.num_layers - n_glob} local window "
            f"{max(w.windows)} + {n_glob} global), {w.num_caches} caches via layer->cache map, batch {w.batch}, "
            f"{w.num_q_heads} q heads, 1 int8 KV head, d={w.head_dim}, page {w.page_size}, "
            f"ctx {w.len_kind} {w.len_values} (mean {float(np.mean(lens)):.0f})")


def run_reference(args, w):
    """Reference arm: the CPU oracle, as it stands, on the host cores.  Each
    step is one decode step of a bounded sample of the workload (the same
    --ref-seqs sequences every step): W untimed warm-up steps, then K timed."""
    rank, world, _ = rank_info()
    if rank != 0:
        return
    st = OracleStack(w, args.ref_seqs)
    for _ in range(args.warmup):
        st.step()
    times = [st.step() for _ in range(args.steps)]
    dt = sum(times) / len(times)
    val = len(st.lens) / dt
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": describe(w, synth.seq_lens_for(w, np.random.default_rng(w.seed))),
                                            "sample_per_step": st.desc},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": st.desc},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_decode(args, w):
    import torch
    rank, world, local_rank = rank_info()
    dist = dist_setup(world, local_rank)
    device = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    hbm, bf16, bf16_sus, peak_kind = measured_peaks()
    stack = DecodeStack(w, device, ring_local=args.ring_local)
    stream = torch.cuda.Stream(device=device)
    sptr = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    B = w.batch
    # eager warm-up, then capture the whole step in a CUDA graph
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            stack.step(sptr)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        stack.step(torch.cuda.current_stream().cuda_stream)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            graph.replay()
    stream.synchronize()

    barrier(dist)
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk:
        times = time_steps(graph.replay, args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(dist)
    total_ms = reduce_max(dist, float(sum(times)))
    ms = total_ms / args.steps
    value = world * B * args.steps / (total_ms / 1000.0)
    kv_bytes = sum(stack.bytes_per_layer)

    # eager step (no graph) for reference
    eager = time_steps(lambda: stack.step(sptr), max(3, min(args.steps, 10)), flush, stream)
    # the L2-warm column: graph replays back to back, no flush (a working set under the
    # 129 MB L2 is then served from it; the appends still write every step)
    warm = time_steps(graph.replay, max(3, min(args.steps, 20)), None, stream)
    warm_ms = statistics.mean(warm)
    # every layer with L2 flushed before it: the step with all KV from HBM, and the
    # per-call roofline of the decode kernel (+ the kernel merging cut pairs)
    seg, cold = cold_layer_times(stack, args.roofline_reps, flush, stream)
    cold_ms = {l: statistics.mean(v) for l, v in cold.items()}
    seg_ms = sum(statistics.mean(v) for v in seg.values())
    achieved = sum(stack.bytes_per_layer) / (sum(cold_ms.values()) * 1e6)
    loc = [l for l in range(w.num_layers) if w.windows[l] > 0]
    glo = [l for l in range(w.num_layers) if w.windows[l] == 0]

    def part(ls):
        if not ls:
            return None
        t = sum(cold_ms[l] for l in ls)
        return {"layers": len(ls), "ms_per_call": t / len(ls),
                "gbps": sum(stack.bytes_per_layer[l] for l in ls) / (t * 1e6),
                "splits": sorted(set(stack.splits[l] for l in ls))}

    digest = source_digest(["mqa_decode_attention_kv_gb300/csrc/decode_tc.cu",
                            "mqa_decode_attention_kv_gb300/csrc/tc_pipe.cuh",
                            "mqa_decode_attention_kv_gb300/csrc/kv_stage.cuh",
                            "mqa_decode_attention_kv_gb300/csrc/common.cuh"])
    # the committed capture is of the full-table step
    traffic = None if args.ring_local else profile_traffic(f"decode_{w.name}_traffic.txt", digest)
    e2e = None
    if not args.no_e2e:
        n_e2e = max(3, min(args.steps, 10))
        et, h2d, d2h, groups = e2e_steps(stack, n_e2e, stream, graph=True)
        ee, _, _, _ = e2e_steps(stack, n_e2e, stream, graph=False)
        e2e = {"value": world * B / (statistics.mean(et) / 1000.0), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": statistics.mean(et),
               "how": "public Python API, pinned host buffers; the step (H2D copies of every query and new "
                      "K/V, 12 appends, 24 decode calls, D2H of every output; copies on a second stream "
                      "overlapping the layers: " + groups + ") captured once into a CUDA graph and replayed",
               "eager": {"value": world * B / (statistics.mean(ee) / 1000.0), "ms_per_step": statistics.mean(ee),
                         "how": "the same calls issued eagerly every step, copies in line with the layers "
                                "(three H2D copies before, one D2H after)"}}
    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline:
        val, dt, desc = oracle_decode_sample(w, args.cpu_seqs)
        cpu = {"value": val, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": desc, "seconds": dt}
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "i8kv-f16mma-f32acc", "data": "synthetic",
        "config": {"workload": describe(w, stack.lens), "global_batch": B * world,
                   "seq_len": f"{w.len_kind} {w.len_values}", "parallelism": f"replicas x{world}",
                   "l2": ("L2 flushed (512 MB read) before every timed step, outside the timed interval.  Inside "
                          "the step the second of two adjacent layers that share a cache finds part of it in L2 "
                          "(nothing runs between them), so kv_gbps is not an HBM figure; step_layers_cold and "
                          "roofline time every layer with L2 flushed before it"),
                   "timing": "CUDA graph of the whole step, replayed; CUDA events on the launching stream",
                   "kv_bytes_per_step": kv_bytes, "kv_gbps": kv_bytes / (ms * 1e6),
                   "local_caches": (f"window-bounded rings of {stack.ring} pages per sequence" if stack.ring
                                    else "full block tables"),
                   "kv_pool_bytes": stack.pool_bytes, "kv_pool_bytes_full_tables": stack.full_pool_bytes},
        "step_layers_cold": {"ms_per_step": seg_ms, "tokens_per_s": world * B / (seg_ms / 1000.0),
                             "kv_gbps": kv_bytes / (seg_ms * 1e6),
                             "how": "sum over the 24 layers of (append if any + decode call), each timed alone "
                                    "with L2 flushed before it (eager launches)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": "decode attention call (the decode kernel + the kernel merging pairs cut between "
                               "CTAs), each call timed alone with L2 flushed before it",
                     "local": part(loc), "global": part(glo)},
        "eager_ms_per_step": statistics.mean(eager),
        "l2_warm": {"ms_per_step": warm_ms, "tokens_per_s": world * B / (warm_ms / 1000.0),
                    "kv_gbps": kv_bytes / (warm_ms * 1e6),
                    "how": "the same graph replayed back to back without the L2 flush (not the headline: KV "
                           "that fits in L2 is read from it)"},
        "gpu_launches": stack.launches_per_step() * args.steps,
        "clocks": clk.summary(),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    dev_status = int(stack.status.item())
    if dev_status:
        # a call flagged bad input or a wait that ran out: the timings are not valid
        line["device_status"] = dev_status
    print(json.dumps(line), flush=True)
    if dev_status:
        raise SystemExit(f"decode calls reported device status {dev_status:#x}")


def run_prefill(args, w):
    import torch
    rank, world, local_rank = rank_info()
    dist = dist_setup(world, local_rank)
    device = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    hbm, bf16, bf16_sus, peak_kind = measured_peaks()
    wl = PrefillWorkload(w, device)
    stream = torch.cuda.Stream(device=device)
    sptr = stream.cuda_stream
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            wl.step(sptr)
    stream.synchronize()
    barrier(dist)
    with ClockSampler(local_rank) as clk:
        times = time_steps(lambda: wl.step(sptr), args.steps, flush, stream)
    barrier(dist)
    total_ms = reduce_max(dist, float(sum(times)))
    ms = total_ms / args.steps
    flops = sum(wl.flops)
    value = world * flops / (ms * 1e-3) / 1e12
    # per-call timing of the prefill kernel (the dominant kernel) and of the append
    per = {l: [] for l in range(len(w.windows))}
    app = []
    with torch.cuda.stream(stream):
        evs = []
        for _ in range(args.roofline_reps):
            flush_l2(flush)
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            wl.append(sptr)
            a1.record(stream)
            for l in range(len(w.windows)):
                flush_l2(flush)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                wl.attend(l, sptr)
                e1.record(stream)
                evs.append((l, e0, e1))
            app.append((a0, a1))
    stream.synchronize()
    for l, e0, e1 in evs:
        per[l].append(e0.elapsed_time(e1))
    per_ms = [statistics.mean(per[l]) for l in range(len(w.windows))]
    app_ms = statistics.mean(a.elapsed_time(b) for a, b in app)
    achieved = sum(wl.flops) / (sum(per_ms) * 1e-3) / 1e12
    append_bytes = wl.T * w.head_dim * 2 * 2 + wl.T * (2 * w.head_dim + 8)
    # the step before prefill: a cached 8192-token prefix (128 pages) uploaded from the
    # pinned host pool into device blocks (and offloaded once to fill the pool)
    import mqa_decode_attention_kv_gb300 as mk
    prefix = w.len_values[0]
    n_pages = prefix // w.page_size
    pc = mk.PrefixCache(w.page_size, w.head_dim, 1, host_pages=n_pages)
    _, slots = pc.insert(np.arange(prefix, dtype=np.int32))
    blocks = wl.pbs.block_table[0, :n_pages]
    pc.offload([wl.cache], blocks, slots, stream=stream)
    ups = []
    with torch.cuda.stream(stream):
        for _ in range(args.roofline_reps + 1):
            flush_l2(flush)
            u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            u0.record(stream)
            pc.upload([wl.cache], slots, blocks, stream=stream)
            u1.record(stream)
            ups.append((u0, u1))
    stream.synchronize()
    up_ms = statistics.mean(a.elapsed_time(b) for a, b in ups[1:])
    up_bytes = n_pages * pc.stats()["slot_bytes"]
    pc.close()
    if rank != 0:
        return
    line = {
        "metric": "prefix-reuse chunked prefill attention TFLOP/s on 1 GB300", "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "i8kv-f16mma-f32acc", "data": "synthetic",
        "config": {"workload": describe(w, wl.lens), "global_batch": w.batch * world,
                   "parallelism": f"replicas x{world}", "l2": "L2 flushed (512 MB read) before every timed step and call",
                   "prefill_flops_per_step": flops, "tokens_per_step": wl.T},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                     "frac": achieved / bf16, "traffic": None,
                     "peak_source": f"{peak_kind} bf16_tflops (fp16 dense rate = bf16 rate)",
                     "kernel": "mqa_prefill_attn kernel, each call timed alone",
                     "ms_per_call": dict(zip([f"window_{x}" for x in w.windows], per_ms))},
        "append": {"ms": app_ms, "gbps": append_bytes / (app_ms * 1e6), "tokens": wl.T},
        "prefix_upload": {"pages": n_pages, "bytes": up_bytes, "ms": up_ms, "gbps": up_bytes / (up_ms * 1e6),
                          "how": "mqa_pc_upload of one cached 8192-token prefix from pinned host memory"},
        "gpu_launches": (1 + len(w.windows)) * args.steps,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_mixed(args):
    """Continuous batching, one layer: 120 sequences decode one token while 8
    prefill a 512-token chunk (lognormal contexts as in the 24-layer stack).
    Times the whole batch as ONE mqa_prefill_attn launch (decode rows are
    sequences with q_len = 1) against the same work as two launches (the decode
    kernel over the 120 decode rows, the prefill kernel over the 8 chunks),
    local window 1024 and global, L2 flushed before each."""
    import torch
    import mqa_decode_attention_kv_gb300 as mk
    torch.cuda.set_device(0)
    device = "cuda:0"
    rng = np.random.default_rng(7)
    n_dec, n_ch, chunk, H, D, P = 120, 8, 512, 32, 128, 64
    ctx = np.clip(np.round(np.exp(rng.normal(np.log(4096.0), 1.0, n_dec + n_ch))), 1, 32768).astype(np.int64)
    q_lens = np.concatenate([np.ones(n_dec, np.int64), np.full(n_ch, chunk, np.int64)])
    lens = ctx.copy()
    lens[n_dec:] += chunk
    order = rng.permutation(n_dec + n_ch)
    lens, q_lens = lens[order].astype(np.int32), q_lens[order]
    pb = synth.make_paged_batch(rng, lens, P, shuffle=True)
    gen = torch.Generator(device=device)
    gen.manual_seed(77)
    cache = mk.KVCache.empty(pb.num_blocks, P, D, device=device)
    cu_all = torch.from_numpy(synth.cu_from_counts(lens)).to(device)
    T_all = int(lens.sum())
    batch = mk.Batch.from_host(pb.block_table, lens, device=device)
    mk.kv_quant_append(cache, batch, cu_all, T_all,
                       torch.randn((T_all, D), generator=gen, device=device).to(torch.bfloat16),
                       torch.randn((T_all, D), generator=gen, device=device).to(torch.bfloat16))
    cu_q = torch.from_numpy(synth.cu_from_counts(q_lens)).to(device)
    T = int(q_lens.sum())
    q = torch.randn((T, H, D), generator=gen, device=device).to(torch.bfloat16)
    dec = np.nonzero(q_lens == 1)[0]
    chs = np.nonzero(q_lens > 1)[0]
    b_dec = mk.Batch.from_host(np.ascontiguousarray(pb.block_table[dec]), lens[dec], device=device)
    b_ch = mk.Batch.from_host(np.ascontiguousarray(pb.block_table[chs]), lens[chs], device=device)
    cu_ch = torch.from_numpy(synth.cu_from_counts(q_lens[chs])).to(device)
    q_dec = q[torch.from_numpy(synth.cu_from_counts(q_lens)[dec]).to(device)].contiguous()
    rows_ch = np.concatenate([np.arange(synth.cu_from_counts(q_lens)[b], synth.cu_from_counts(q_lens)[b + 1])
                              for b in chs])
    q_ch = q[torch.from_numpy(rows_ch).to(device)].contiguous()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    stream = torch.cuda.Stream(device=device)
    res = {}
    with torch.cuda.stream(stream):
        for W in (1024, 0):
            ws = None
            splits = mk.mqa_decode_auto_splits(b_dec, W, H, D, P)
            if splits > 1:
                ws = torch.empty(mk.mqa_decode_workspace_size(len(dec), H, D, splits), dtype=torch.uint8,
                                 device=device)
            ws_one = torch.empty(max(16, mk.mqa_prefill_workspace_size(batch.batch, batch.max_seq_len, W, chunk, D)),
                                 dtype=torch.uint8, device=device)
            ws_ch = torch.empty(max(16, mk.mqa_prefill_workspace_size(b_ch.batch, b_ch.max_seq_len, W, chunk, D)),
                                dtype=torch.uint8, device=device)
            one = lambda: mk.mqa_prefill_attn([cache], [0], 0, W, batch, cu_q, q, chunk, workspace=ws_one,
                                              stream=stream)
            two = lambda: (mk.mqa_decode_attn([cache], [0], 0, W, b_dec, q_dec, num_splits=splits, workspace=ws,
                                              stream=stream),
                           mk.mqa_prefill_attn([cache], [0], 0, W, b_ch, cu_ch, q_ch, chunk, workspace=ws_ch,
                                               stream=stream))
            for name, fn in (("one_launch", one), ("two_launches", two)):
                for _ in range(max(args.warmup, 1)):
                    fn()
                ts = []
                for _ in range(args.steps):
                    flush_l2(flush)
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(stream)
                    fn()
                    e1.record(stream)
                    ts.append((e0, e1))
                stream.synchronize()
                res[f"window_{W}_{name}_ms"] = statistics.mean(a.elapsed_time(b) for a, b in ts)
    line = {"metric": "mixed decode + prefill-chunk batch attention ms per layer on 1 GB300",
            "value": res["window_1024_one_launch_ms"], "unit": "ms", "higher_is_better": False,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "dtype": "i8kv-f16mma-f32acc",
            "data": "synthetic",
            "config": {"workload": f"mixed_b128: {n_dec} decode rows + {n_ch} prefill chunks of {chunk} tokens, "
                                   f"32 q heads, d=128, page 64, ctx lognormal (4096, 1.0, 32768) "
                                   f"(mean {float(lens.mean()):.0f})", "tokens": T,
                       "l2": "L2 flushed (512 MB read) before every timed call"},
            "times": res}
    print(json.dumps(line), flush=True)


_MMA_RATE_SRC = r"""
// Warp-level MMA throughput: int8 m16n8k32 (s32 accumulate) against fp16 m16n8k16 (fp32
// accumulate), eight independent accumulators per warp, registers only.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
template <bool I8>
__global__ void __launch_bounds__(256) rate(long long *out, int iters) {
    uint32_t a[4] = {threadIdx.x, threadIdx.x * 3u, 7u, 9u}, b[2] = {5u, threadIdx.x};
    float f[8][4] = {};
    int s[8][4] = {};
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (I8)
                asm volatile("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                             : "+r"(s[k][0]), "+r"(s[k][1]), "+r"(s[k][2]), "+r"(s[k][3])
                             : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
            else
                asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                             : "+f"(f[k][0]), "+f"(f[k][1]), "+f"(f[k][2]), "+f"(f[k][3])
                             : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
        }
    }
    float acc = 0.f;
    for (int k = 0; k < 8; ++k) for (int q = 0; q < 4; ++q) acc += f[k][q] + (float)s[k][q];
    if (acc == 12345.f) out[0] = 1;
}
int main() {
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    long long *d;
    cudaMalloc(&d, 8);
    const int iters = 4096, blocks = sms * 4;
    for (int i8 = 0; i8 < 2; ++i8) {
        cudaEvent_t e0, e1;
        cudaEventCreate(&e0);
        cudaEventCreate(&e1);
        float ms = 0.f;
        for (int rep = 0; rep < 3; ++rep) {
            cudaEventRecord(e0);
            if (i8) rate<true><<<blocks, 256>>>(d, iters); else rate<false><<<blocks, 256>>>(d, iters);
            cudaEventRecord(e1);
            cudaEventSynchronize(e1);
            cudaEventElapsedTime(&ms, e0, e1);
        }
        const double ops = (double)blocks * 8 * iters * 8 * (i8 ? 8192.0 : 4096.0);
        printf("%s %.1f %s\n", i8 ? "int8_m16n8k32_tops" : "fp16_m16n8k16_tflops", ops / (ms * 1e9),
               cudaGetErrorString(cudaGetLastError()));
    }
    return 0;
}
"""

_KIND_I8_SRC = r"""
#include <cstdint>
__global__ void k(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
    asm volatile("{\n\t.reg .pred pa;\n\tsetp.ne.b32 pa, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::i8 [%0], %1, %2, %3, pa;\n\t}" ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(1u));
}
"""


def run_mma_rates(args):
    """The int8-MMA question (fully int8 attention only pays if int8 MMA beats
    fp16 here): whether ptxas accepts tcgen05.mma kind::i8 for sm_103a, and the
    measured warp-level int8 and fp16 MMA rates of this GPU."""
    import shutil
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    out = {"metric": "warp-level MMA rates (int8 vs fp16) and tcgen05 kind::i8 availability on 1 GB300"}
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "i8.cu")
        open(src, "w").write(_KIND_I8_SRC)
        r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-c", src, "-o",
                            os.path.join(tmp, "i8.o")], capture_output=True, text=True)
        msg = [l for l in (r.stdout + r.stderr).splitlines() if "error" in l]
        out["tcgen05_kind_i8_sm_103a"] = {"compiles": r.returncode == 0,
                                          "ptxas": msg[0].split("error")[-1].strip(" :") if msg else ""}
        src = os.path.join(tmp, "rate.cu")
        open(src, "w").write(_MMA_RATE_SRC)
        exe = os.path.join(tmp, "rate")
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", src, "-o", exe])
        res = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
        for line in res:
            parts = line.split()
            if len(parts) >= 3:
                out[parts[0]] = float(parts[1])
                assert parts[2] == "no", line
    print(json.dumps(out), flush=True)


def run_profile(args, w):
    """Set-up plus a few eager steps, nothing else: a short, bounded program
    for ncu (one GPU)."""
    import torch
    torch.cuda.set_device(0)
    wl = PrefillWorkload(w, "cuda:0") if w.name == "prefix_prefill" else DecodeStack(w, "cuda:0")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(args.steps):
            wl.step(stream.cuda_stream)
    stream.synchronize()
    print(f"profile run done: {args.steps} steps of {w.name}", flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stack24_b128", choices=sorted(synth.CONFIGS) + ["mixed_b128", "mma_rates"])
    ap.add_argument("--roofline-reps", type=int, default=3)
    ap.add_argument("--cpu-seqs", type=int, default=32, help="sequences in the cpu_baseline's timed sample")
    ap.add_argument("--ref-seqs", type=int, default=4,
                    help="sequences per step of the reference arm (the oracle on the host cores)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ring-local", action="store_true",
                    help="decode workloads: caches read only by local layers as window-bounded rings")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="set up the workload, run --steps eager steps and exit (for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3 and not args.profile:
        ap.error("--warmup must be >= 3")
    if args.workload == "mma_rates":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "a hardware-rate probe has no reference arm"}))
            return
        run_mma_rates(args)
        return
    if args.workload == "mixed_b128":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle baseline covers decode workloads only"}))
            return
        from mqa_decode_attention_kv_gb300 import build as _b
        _b.build()
        run_mixed(args)
        return
    w = synth.CONFIGS[args.workload]
    if args.impl == "reference":
        if w.name == "prefix_prefill":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle baseline covers decode workloads only"}))
            return
        run_reference(args, w)
        return
    from mqa_decode_attention_kv_gb300 import build as _b
    _b.build()
    if args.profile:
        run_profile(args, w)
    elif w.name == "prefix_prefill":
        run_prefill(args, w)
    else:
        run_decode(args, w)


if __name__ == "__main__":
    main()
