"""Pins of the oracle's packed signed-byte dot (the pages' streaming example).

Loom pages, "Tune loop unrolling and pipelining", section "Apply the same
controls to a packed dot product": each lane unpacks four signed bytes per
record, scales them by the record's f16 scale and advances an ordered f32 dot
accumulation against four f32 activations of its stream.  The oracle is
pinned here against a library routine (numpy's binary16 decoding), exact
integer arithmetic on inputs where every step is exact, and hand-derived f32
results that fix the fused step, the record order and the element order.
"""
import numpy as np
import pytest

import oracle

F16_ONE = 0x3C00


def test_f16_decoding_matches_numpy_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), want[~nan].view(np.uint32))


def _case(P, R, L, S, seed):
    rng = np.random.default_rng(seed)
    fields = rng.integers(0, 1 << 32, size=(P, R, L), dtype=np.uint64).astype(np.uint32)
    return rng, fields


def test_exact_inputs_match_integer_arithmetic():
    # Scale 1/4 and small integer activations keep every product and partial
    # sum exact in f32, so the result is the exact sum, computed here with
    # int64 from a byte view of the packed words (not from shifts).
    P, R, L, S = 2, 9, 2048, 64
    rng, fields = _case(P, R, L, S, 7)
    scales = np.full((P, R, L), np.float16(0.25)).view(np.uint16)
    rhs = rng.integers(-4, 5, size=(P, R, S, 4)).astype(np.float32)
    counts = np.array([9, 5], np.int32)
    init = rng.integers(-100, 101, size=(P, L)).astype(np.float32)
    got = oracle.packed_dot(fields, scales, rhs, counts, init)
    b = fields.view("<i4").view(np.int8).reshape(P, R, L, 4).astype(np.int64)
    a = rhs.astype(np.int64)[:, :, np.arange(L) % S, :]            # lane l reads stream l mod S
    for p in range(P):
        c = counts[p]
        total = 4 * init[p].astype(np.int64) + (b[p, :c] * a[p, :c]).sum(axis=(0, 2))   # in quarters
        assert np.array_equal(got[p].astype(np.float64) * 4, total.astype(np.float64)), p


def test_empty_and_initial():
    rng, fields = _case(3, 4, 64, 64, 3)
    scales = np.full((3, 4, 64), F16_ONE, np.uint16)
    rhs = rng.standard_normal((3, 4, 64, 4)).astype(np.float32)
    init = rng.standard_normal((3, 64)).astype(np.float32)
    out = oracle.packed_dot(fields, scales, rhs, [0, 0, 0], init)
    assert np.array_equal(out.view(np.uint32), init.view(np.uint32))
    assert not oracle.packed_dot(fields, scales, rhs, [0, 0, 0]).any()


def _one(words, scale_bits, rhs_rows, initial=0.0):
    """One lane, one stream: records given as (word, f16 bits, four activations)."""
    R = len(words)
    fields = np.array(words, np.uint32).reshape(1, R, 1)
    scales = np.array(scale_bits, np.uint16).reshape(1, R, 1)
    rhs = np.array(rhs_rows, np.float32).reshape(1, R, 1, 4)
    init = np.array([[initial]], np.float32)
    return oracle.packed_dot(fields, scales, rhs, [R], init)[0, 0]


def test_each_element_is_one_fused_multiply_add():
    # scaled = 1 * (1 + 2^-10) (f16 0x3C01), activation 1 + 2^-14, sum -1:
    # the exact product is 1 + 2^-10 + 2^-14 + 2^-24.  A fused step keeps the
    # 2^-24 (the result is 2^-10 + 2^-14 + 2^-24, exact in f32); a rounded
    # product would lose it (a tie, rounded to even) and give 2^-10 + 2^-14.
    got = _one([0x00000001], [0x3C01], [[1 + 2.0 ** -14, 0, 0, 0]], initial=-1.0)
    assert got == np.float32(2.0 ** -10 + 2.0 ** -14 + 2.0 ** -24)


def test_records_accumulate_in_order():
    # products 2^24, then 1, then -2^24: in record order 2^24 + 1 rounds back
    # to 2^24 (a tie, to even) and the result is 0; the reverse order or
    # cancelling first keeps the 1.
    words = [0x00000040, 0x00000001, 0x000000C0]   # bytes 64, 1, -64
    rhs = [[2.0 ** 18, 0, 0, 0], [1, 0, 0, 0], [2.0 ** 18, 0, 0, 0]]
    assert _one(words, [F16_ONE] * 3, rhs) == 0.0
    assert _one(words[::-1], [F16_ONE] * 3, rhs[::-1]) == 1.0
    assert _one([words[0], words[2], words[1]], [F16_ONE] * 3, [rhs[0], rhs[2], rhs[1]]) == 1.0


def test_elements_accumulate_in_order():
    # the same cancellation across the four elements of one record
    word = 0x00C00140                                 # bytes 64, 1, -64, 0
    assert _one([word], [F16_ONE], [[2.0 ** 18, 1, 2.0 ** 18, 0]]) == 0.0
    word_b = 0x0040C001                               # bytes 1, -64, 64, 0
    assert _one([word_b], [F16_ONE], [[1, 2.0 ** 18, 2.0 ** 18, 0]]) == 1.0


def test_lane_reads_its_stream_and_its_scale():
    # only stream 5 is nonzero: lanes 5, 69, 133 ... get outputs, the rest 0;
    # per-lane scales 2^-(l mod 3) show up in each lane's result
    P, R, L, S = 1, 1, 256, 64
    fields = np.full((P, R, L), 0x00000002, np.uint32)           # byte 2, then zeros
    exps = np.arange(L) % 3
    scales = np.array([np.float16(2.0 ** -e) for e in exps], np.float16).view(np.uint16).reshape(P, R, L)
    rhs = np.zeros((P, R, S, 4), np.float32)
    rhs[0, 0, 5, 0] = 3.0
    out = oracle.packed_dot(fields, scales, rhs, [1])[0]
    want = np.where(np.arange(L) % S == 5, 6.0 * 2.0 ** -exps, 0.0)
    assert np.array_equal(out, want.astype(np.float32))


def test_count_range_is_checked():
    fields = np.zeros((1, 4, 8), np.uint32)
    scales = np.zeros((1, 4, 8), np.uint16)
    rhs = np.zeros((1, 4, 8, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.packed_dot(fields, scales, rhs, [5])
