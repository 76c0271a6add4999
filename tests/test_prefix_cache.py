"""Host-side tests of the prefix cache (no GPU): the C++ tree against the plain
model in oracle/prefix_cache_model.py, on seeded conversation-like streams, and
its argument checks."""
import ctypes

import numpy as np
import pytest

import mqa_decode_attention_kv_gb300 as mk
from mqa_decode_attention_kv_gb300 import build as mkbuild
from oracle.prefix_cache_model import PrefixCacheModel


@pytest.fixture(scope="module", autouse=True)
def built():
    mkbuild.build()


def conversations(rng, n_convs, page, vocab=50):
    """Token streams shaped like chat sessions: a shared system prompt, then
    turns that grow each conversation (later turns extend earlier ones)."""
    system = rng.integers(0, vocab, 2 * page + 5).astype(np.int32)
    convs = []
    for _ in range(n_convs):
        toks = list(system)
        turns = []
        for _ in range(rng.integers(2, 5)):
            toks += list(rng.integers(0, vocab, int(rng.integers(1, 3 * page))))
            turns.append(np.array(toks, np.int32))
        convs.append(turns)
    return convs


@pytest.mark.parametrize("page,capacity,seed", [(16, 6, 0), (16, 40, 1), (64, 9, 2), (16, 3, 3)])
def test_tree_matches_the_model(page, capacity, seed):
    rng = np.random.default_rng(seed)
    pc = mk.PrefixCache(page, 64, 2, capacity, pinned=False)
    model = PrefixCacheModel(page, capacity)
    convs = conversations(rng, 6, page)
    ops = 0
    for step in range(60):
        turns = convs[int(rng.integers(0, len(convs)))]
        toks = turns[int(rng.integers(0, len(turns)))]
        if rng.random() < 0.3:
            # an edited message: one token changed somewhere in the stream
            toks = toks.copy()
            toks[int(rng.integers(0, len(toks)))] += 1000
        if rng.random() < 0.5:
            got = pc.match(toks).tolist()
            assert got == model.match(toks), f"step {step}: match"
        else:
            idx, slots = pc.insert(toks)
            assert list(zip(idx.tolist(), slots.tolist())) == model.insert(toks), f"step {step}: insert"
        ops += 1
    st = pc.stats()
    assert st["cached_pages"] == len(model.pages)
    assert st["free_slots"] == len(model.free)
    assert st["pages_evicted"] == model.evicted
    assert st["cached_pages"] + st["free_slots"] == capacity


def test_longest_prefix_and_partial_pages():
    pc = mk.PrefixCache(16, 128, 1, 16, pinned=False)
    a = np.arange(100, dtype=np.int32)           # 6 whole pages + 4 tokens
    idx, slots = pc.insert(a)
    assert idx.tolist() == list(range(6))         # the partial last page is not cached
    assert pc.match(a).tolist() == slots.tolist()
    assert len(pc.match(a[:95])) == 5             # a shorter query matches its whole pages
    b = a.copy()
    b[40] = -7                                    # differs inside page 2
    assert pc.match(b).tolist() == slots[:2].tolist()
    # inserting b shares pages 0-1 and adds its own pages 2-5
    idx_b, slots_b = pc.insert(b)
    assert idx_b.tolist() == [2, 3, 4, 5] and not set(slots_b) & set(slots)
    assert pc.match(b).tolist() == slots[:2].tolist() + slots_b.tolist()
    assert len(pc.match(np.arange(15, dtype=np.int32))) == 0


def test_lru_evicts_leaves_only_and_protects_the_inserted_path():
    pc = mk.PrefixCache(16, 64, 1, 4, pinned=False)
    a = np.arange(64, dtype=np.int32)             # 4 pages: fills the pool
    pc.insert(a)
    pc.match(a[:32])                              # pages 0, 1 most recent; page 3 is the only leaf
    c = np.concatenate([a[:32], np.full(32, 500, np.int32)])
    idx, slots = pc.insert(c)                     # needs 2 slots: evicts page 3, then page 2
    assert idx.tolist() == [2, 3]
    assert pc.match(a).tolist()[:2] == pc.match(c).tolist()[:2]
    assert len(pc.match(a)) == 2                  # a's pages 2, 3 are gone
    # a path longer than the pool: insertion stops once nothing is evictable
    d = np.arange(1000, 1000 + 16 * 6, dtype=np.int32)
    idx, _ = pc.insert(d)
    assert idx.tolist() == [0, 1, 2, 3]
    assert pc.stats()["free_slots"] == 0


def test_argument_checks():
    L = mk.lib()
    h = ctypes.c_void_p()
    assert L.mqa_pc_create(32, 128, 1, 4, 0, ctypes.byref(h)) == mk.MQA_ERR_UNSUPPORTED
    assert L.mqa_pc_create(64, 96, 1, 4, 0, ctypes.byref(h)) == mk.MQA_ERR_UNSUPPORTED
    assert L.mqa_pc_create(64, 128, 0, 4, 0, ctypes.byref(h)) == mk.MQA_ERR_INVALID_ARG
    assert L.mqa_pc_create(64, 128, 33, 4, 0, ctypes.byref(h)) == mk.MQA_ERR_INVALID_ARG
    assert L.mqa_pc_create(64, 128, 1, 0, 0, ctypes.byref(h)) == mk.MQA_ERR_INVALID_ARG
    assert L.mqa_pc_create(64, 128, 1, 4, 0, None) == mk.MQA_ERR_INVALID_ARG
    pc = mk.PrefixCache(64, 128, 1, 4, pinned=False)
    assert L.mqa_pc_match(pc._h, None, 64, None, 0) == mk.MQA_ERR_INVALID_ARG
    assert L.mqa_pc_match(pc._h, None, 0, None, 0) == 0
    assert L.mqa_pc_insert(pc._h, None, -1, None, None, 0) == mk.MQA_ERR_INVALID_ARG
    assert L.mqa_pc_match(None, None, 0, None, 0) == mk.MQA_ERR_INVALID_ARG
    # no pinned pool: the copies are refused before any CUDA call
    cache = (mk._Cache * 1)(mk._Cache(0x10000, 0x10000, 0x10000, 0x10000, 8, 64, 128))
    blocks = np.zeros(1, np.int32)
    slots = np.zeros(1, np.int64)
    assert L.mqa_pc_upload(pc._h, cache, 1, slots.ctypes.data, blocks.ctypes.data, 1, None) == mk.MQA_ERR_UNSUPPORTED
    assert L.mqa_pc_offload(pc._h, cache, 1, blocks.ctypes.data, slots.ctypes.data, 1, None) == \
        mk.MQA_ERR_UNSUPPORTED
    out = np.zeros(8, np.int64)
    assert L.mqa_pc_stats(pc._h, out.ctypes.data) == mk.MQA_OK and out[2] == 4 and out[7] == 64 * 264
    L.mqa_pc_destroy(None)
