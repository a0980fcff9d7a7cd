"""Pins of the oracle's per-lane f32 sums (the pages' sum_rows, sum_vector_rows
and sum_guarded_rows examples, batched over independent segments).

Loom pages, "Tune loop unrolling and pipelining": sections "Keep one checked
source for experiments" and "Complete correctness cases and benchmark"
(sum_rows and its printed check vectors), "Give each motif its own schedule"
(sum_vector_rows) and "Keep guards and inner loops in the source"
(sum_guarded_rows).  The sums are f32 recurrences in source order, so the
pins fix values (printed vectors, exact integer inputs against int64
arithmetic) and orders (cancellations that only one order leaves at 0).
"""
import os

import numpy as np
import pytest

import oracle
import synth

BIG = 2.0 ** 24


def _golden(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "sum_rows_iota.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(tuple(int(t) for t in line.split()))
    return rows


def test_sum_rows_reproduces_the_printed_vectors(golden_dir):
    values = synth.iota_case(rows=64, lanes=32, count=0)["values"]
    cases = _golden(golden_dir)
    seg = np.broadcast_to(values, (len(cases), 64, 32))
    got = oracle.lane_sums(seg, [c for c, _, _ in cases])
    for i, (count, offset, step) in enumerate(cases):
        want = (offset + step * np.arange(32)).astype(np.float32)
        assert np.array_equal(got[i], want), (count, got[i][:4])


def test_exact_inputs_match_integer_sums():
    rng = np.random.default_rng(5)
    S, R, L = 7, 64, 32
    counts = np.array([0, 1, 5, 31, 32, 63, 64], np.int32)
    for width in (1, 4):
        shape = (S, R, L) if width == 1 else (S, R, L, 4)
        ints = rng.integers(-1000, 1001, size=shape)
        got = oracle.lane_sums(ints.astype(np.float32), counts, width=width)
        for s in range(S):
            block = ints[s, :counts[s]]
            want = block.sum(axis=0) if width == 1 else block.sum(axis=(0, 2))
            assert np.array_equal(got[s], want.astype(np.float32)), (width, s)


def test_rows_add_in_order():
    v = np.zeros((2, 3, 1), np.float32)
    v[0, :, 0] = [BIG, 1, -BIG]          # BIG + 1 rounds back to BIG (a tie, to even)
    v[1, :, 0] = [-BIG, 1, BIG]          # -BIG + 1 is exact
    got = oracle.lane_sums(v, [3, 3])
    assert got[0, 0] == 0.0 and got[1, 0] == 1.0


def test_vector_elements_add_in_order_after_the_carried_sum():
    v = np.zeros((3, 2, 1, 4), np.float32)
    v[0, 0, 0] = [BIG, 1, -BIG, 0]
    v[1, 0, 0] = [BIG, -BIG, 1, 0]
    v[2, 0, 0] = [BIG, 0, 0, 0]          # then the next row adds to the carried BIG
    v[2, 1, 0] = [1, -BIG, 0, 0]
    got = oracle.lane_sums(v, [1, 1, 2], width=4)
    assert got[0, 0] == 0.0 and got[1, 0] == 1.0 and got[2, 0] == 0.0


def test_lanes_are_columns():
    v = np.zeros((1, 4, 32), np.float32)
    v[0, :, 7] = [1, 2, 3, 4]
    got = oracle.lane_sums(v, [3])[0]
    assert got[7] == 6.0 and not np.delete(got, 7).any()


def _guarded_case(rng, count, rows=63, lanes=32):
    ints = rng.integers(-500, 501, size=(1, rows, lanes, 4)).astype(np.float32)
    return ints


@pytest.mark.parametrize("count,columns,active", [(0, 4, 32), (1, 1, 32), (5, 3, 17), (8, 4, 32),
                                                  (63, 4, 32), (62, 2, 1), (13, 0, 32), (40, 4, 0)])
def test_guarded_rows_exact(count, columns, active):
    rng = np.random.default_rng(count * 100 + columns * 10 + active)
    v = _guarded_case(rng, count)
    want = np.zeros(32, np.float64)
    want[:active] = v[0, :count, :active, :columns].astype(np.float64).sum(axis=(0, 2))
    # what the guards exclude holds NaN: rows at or past the count, columns at or
    # past `columns`, lanes at or past `active`
    v[0, count:] = np.nan
    v[0, :, :, columns:] = np.nan
    v[0, :, active:, :] = np.nan
    got = oracle.guarded_rows(v, [count], columns, active)[0]
    assert np.array_equal(got, want.astype(np.float32))


def test_guarded_rows_orders():
    v = np.zeros((2, 8, 32, 4), np.float32)
    v[0, 0, 0, :3] = [BIG, 1, -BIG]                 # inside a row: column order
    v[1, 0, 0, 0], v[1, 1, 0, 0], v[1, 2, 0, 0] = BIG, 1, -BIG   # across rows: row order
    got = oracle.guarded_rows(v, [1, 3], 3, 32)
    assert got[0, 0] == 0.0 and got[1, 0] == 0.0
    v[0, 0, 0, :3] = [-BIG, 1, BIG]
    v[1, 0, 0, 0], v[1, 2, 0, 0] = -BIG, BIG
    got = oracle.guarded_rows(v, [1, 3], 3, 32)
    assert got[0, 0] == 1.0 and got[1, 0] == 1.0


def test_counts_are_checked():
    with pytest.raises(ValueError):
        oracle.lane_sums(np.zeros((1, 4, 32), np.float32), [5])
    with pytest.raises(ValueError):
        oracle.guarded_rows(np.zeros((1, 4, 32, 4), np.float32), [5], 4, 32)
    with pytest.raises(ValueError):
        oracle.guarded_rows(np.zeros((1, 4, 32, 4), np.float32), [2], 5, 32)
