"""Pins for the oracle's int8 quantise-and-append step (CPU only).

The quantiser is symmetric per token: scale = max|x|/127 in fp32, codes are
round-half-to-even of x/scale clamped to +-127.  These tests pin it with tie
cases whose answers follow from the rounding rule, exact power-of-two
round-trips, the zero vector, and the error bound |x - code*scale| <= scale/2
that any correct round-to-nearest quantiser satisfies.
"""
import numpy as np
import pytest

import oracle
from synth import bf16_bits_to_f32, bf16_normal, cu_from_counts, f32_to_bf16_bits, make_paged_batch


def _bits(vals, d=None):
    a = np.asarray(vals, np.float32)
    if d is not None and a.shape[-1] < d:
        a = np.concatenate([a, np.zeros(d - a.shape[-1], np.float32)])
    b = f32_to_bf16_bits(a)
    assert np.array_equal(bf16_bits_to_f32(b), a), "test values must be exact in bf16"
    return b


def test_ties_round_half_to_even():
    # amax = 127 makes the scale exactly 1, so codes are the rounded inputs.
    x = _bits([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 1.5, 126.5, -125.5, 0.25, -127.0, 7.0, 0.75])
    codes, scales = oracle.quantize_tokens(x[None, :])
    assert scales[0] == np.float32(1.0)
    assert codes[0].tolist() == [127, 2, 4, -2, -4, 0, 0, 2, 126, -126, 0, -127, 7, 1]


@pytest.mark.parametrize("k", [-30, -7, -1, 0, 3, 19])
def test_power_of_two_round_trip(k):
    rng = np.random.default_rng(100 + k)
    c = rng.integers(-127, 128, size=64).astype(np.int64)
    c[rng.integers(0, 64)] = 127 if rng.integers(0, 2) else -127
    x = _bits(np.ldexp(c.astype(np.float64), k).astype(np.float32))
    codes, scales = oracle.quantize_tokens(x[None, :])
    assert scales[0] == np.float32(2.0 ** k)
    assert np.array_equal(codes[0].astype(np.int64), c)


def test_zero_vector():
    codes, scales = oracle.quantize_tokens(np.zeros((3, 128), np.uint16))
    assert np.all(scales == 0) and np.all(codes == 0)


def test_negative_zero_and_single_spike():
    x = np.zeros(64, np.float32)
    x[5] = -3.0
    b = f32_to_bf16_bits(x)
    b[7] = 0x8000  # -0.0
    codes, scales = oracle.quantize_tokens(b[None, :])
    assert codes[0, 5] == -127 and codes[0, 7] == 0
    assert np.count_nonzero(codes[0]) == 1


def test_random_tokens_error_bound_and_range():
    rng = np.random.default_rng(7)
    x = bf16_normal(rng, (500, 128), scale=3.0)
    codes, scales = oracle.quantize_tokens(x)
    xf = bf16_bits_to_f32(x).astype(np.float64)
    amax = np.abs(xf).max(axis=1)
    s = scales.astype(np.float64)
    # the scale is amax/127 up to one fp32 rounding
    assert np.all(np.abs(s * 127.0 - amax) <= amax * 2.0 ** -23)
    # every token uses the full code range at its max element
    assert np.all(np.abs(codes.astype(np.int64)).max(axis=1) == 127)
    # round-to-nearest error bound; fl32(x/s) may itself move by half an ulp of
    # a value below 128, i.e. by at most 2^-17 of a code step
    err = np.abs(xf - codes.astype(np.float64) * s[:, None])
    assert np.all(err <= s[:, None] * (0.5 + 2.0 ** -17))


def test_append_scatters_to_paged_slots():
    rng = np.random.default_rng(3)
    d, P = 64, 16
    seq_lens = np.array([5, 33, 16, 1], np.int32)
    pb = make_paged_batch(rng, seq_lens, P, shuffle=True)
    cache = oracle.Cache.empty(pb.num_blocks, P, d)
    counts = seq_lens.copy()
    cu = cu_from_counts(counts)
    k = bf16_normal(rng, (int(cu[-1]), d))
    v = bf16_normal(rng, (int(cu[-1]), d))
    oracle.quant_append(cache, pb.block_table, seq_lens, cu, k, v)
    kc, ks = oracle.quantize_tokens(k)
    vc, vs = oracle.quantize_tokens(v)
    for b in range(len(seq_lens)):
        for pos in range(seq_lens[b]):
            blk = pb.block_table[b, pos // P]
            row = cu[b] + pos
            assert np.array_equal(cache.k_codes[blk, pos % P], kc[row])
            assert np.array_equal(cache.v_codes[blk, pos % P], vc[row])
            assert cache.k_scale[blk, pos % P] == ks[row]
            assert cache.v_scale[blk, pos % P] == vs[row]
    # untouched slots stay zero: exactly sum(L) slots were written
    assert np.count_nonzero(cache.k_scale) == int(seq_lens.sum())


def test_append_tail_only_and_bounds():
    rng = np.random.default_rng(4)
    d, P = 64, 16
    seq_lens = np.array([20, 40], np.int32)
    pb = make_paged_batch(rng, seq_lens, P)
    cache = oracle.Cache.empty(pb.num_blocks, P, d)
    cu = cu_from_counts([2, 1])  # append the last 2 tokens of seq 0, last 1 of seq 1
    k = bf16_normal(rng, (3, d))
    oracle.quant_append(cache, pb.block_table, seq_lens, cu, k, k)
    kc, _ = oracle.quantize_tokens(k)
    assert np.array_equal(cache.k_codes[pb.block_table[0, 18 // P], 18 % P], kc[0])
    assert np.array_equal(cache.k_codes[pb.block_table[0, 19 // P], 19 % P], kc[1])
    assert np.array_equal(cache.k_codes[pb.block_table[1, 39 // P], 39 % P], kc[2])
    assert np.count_nonzero(cache.k_scale) == 3
    bad = pb.block_table.copy()
    bad[1, 2] = pb.num_blocks  # out of the pool
    with pytest.raises(ValueError):
        oracle.quant_append(cache, bad, seq_lens, cu, k, k)
