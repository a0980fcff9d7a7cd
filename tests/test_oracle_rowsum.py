"""Pins for the row-sum oracle, independent of the oracle's own code.

Each check comes from the pages or from mathematics, never from the oracle
itself:
  * the full-tile split against its closed form  F = T*floor(c/T), t = c mod T
    (page "Tune loop unrolling and pipelining", "Derive full tiles from a
    ragged loop"), including the 63-row, count 61 worked case (56, 5);
  * the pages' printed per-lane check vectors for the iota input
    1 + 32*row + lane ("Complete correctness cases and benchmark");
  * closed forms of the iota row sums derived from that same input;
  * exact rational sums on random inputs drawn on the 2**-23 grid.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth


@pytest.mark.parametrize("tile", [1, 2, 3, 5, 8, 13, 64])
def test_split_closed_form(tile):
    for c in range(0, 200):
        assert oracle.full_tile_split(c, tile) == (tile * (c // tile), c % tile)


def test_split_worked_case():
    # 63-row segment, count 61, tile 8: eight-row tiles end at row 56, five rows remain.
    assert oracle.full_tile_split(61, 8) == (56, 5)


def test_split_rejects_bad_tile():
    with pytest.raises(ValueError):
        oracle.full_tile_split(5, 0)


def _golden_rows(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "sum_rows_iota.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(tuple(int(t) for t in line.split()))
    return rows


def test_sum_rows_page_vectors(golden_dir):
    values = synth.iota_case(rows=64, lanes=32, count=0)["values"]
    cases = _golden_rows(golden_dir)
    assert len(cases) == 8
    for count, offset, step in cases:
        got = oracle.sum_rows(values, count)
        want = offset + step * np.arange(32, dtype=np.float64)
        assert np.array_equal(got, want), (count, got[:4])


def test_page_vectors_match_stated_formula(golden_dir):
    # The pages also state the closed form N*(lane+1) + 16*N*(N-1); the printed
    # vectors must agree with it (guards the transcription of the fixture).
    for count, offset, step in _golden_rows(golden_dir):
        for lane in (0, 1, 31):
            assert offset + step * lane == count * (lane + 1) + 16 * count * (count - 1)


def _iota_row_sum(r, lanes=32):
    # sum over l of (1 + lanes*r + l)
    return lanes + lanes * lanes * r + lanes * (lanes - 1) // 2


@pytest.mark.parametrize("tile", [1, 3, 8, 64])
def test_full_tile_sum_iota_closed_form(tile):
    values = synth.iota_case(rows=63, lanes=32, count=0)["values"]
    for c in range(0, 64):
        F, t = tile * (c // tile), c % tile
        fr, tc, fs, ts = oracle.full_tile_sum(values, c, 0.5, tile)
        assert (fr, tc) == (F, t)
        assert fs == 0.5 + 528 * F + 512 * F * (F - 1)
        assert ts == 528 * t + 1024 * (t * F + t * (t - 1) // 2)
        assert fs - 0.5 == sum(_iota_row_sum(r) for r in range(F))


def test_full_tile_sum_iota_worked_case():
    values = synth.iota_case(rows=63, lanes=32, count=61, initial=0.5)["values"]
    assert oracle.full_tile_sum(values, 61, 0.5, 8) == (56, 5, 1606528.5, 299600.0)


def test_row_sum_agrees_with_page_vectors(golden_dir):
    # Summing the pages' per-lane column sums over the lanes must give the
    # row-reduction total: this ties the row-sum oracle's indexing to printed values.
    values = synth.iota_case(rows=64, lanes=32, count=0)["values"]
    for count, offset, step in _golden_rows(golden_dir):
        lane_total = sum(offset + step * lane for lane in range(32))
        for tile in (1, 8, 64):
            _, _, fs, ts = oracle.full_tile_sum(values, count, 0.0, tile)
            assert fs + ts == lane_total


def _exact_split(values, count, initial, tile):
    F = tile * (count // tile)
    full = Fraction(initial) + sum((Fraction(float(x)) for x in values[:F].ravel()), Fraction(0))
    tail = sum((Fraction(float(x)) for x in values[F:count].ravel()), Fraction(0))
    return F, count - F, full, tail


def test_brute_force_exact_rationals():
    rng_seed = synth.workload_seed(1) ^ 0x5A5A
    shapes = [(3, 2), (4, 5), (7, 1), (9, 32), (16, 3), (5, 32)]
    case = 0
    for rows, lanes in shapes:
        for tile in (1, 2, 3, 8):
            vals = synth.uniform_grid_f32(synth.stream_seed(rng_seed, case), rows * lanes)
            vals = vals.reshape(rows, lanes)
            init = float(synth.uniform_grid_f32(synth.stream_seed(rng_seed, 1000 + case), 1)[0])
            case += 1
            for c in range(rows + 1):
                F, t, full, tail = _exact_split(vals, c, init, tile)
                fr, tc, fs, ts = oracle.full_tile_sum(vals, c, init, tile)
                assert (fr, tc) == (F, t)
                # grid values: every fp64 partial sum is exact, so equality is exact
                assert Fraction(fs) == full and Fraction(ts) == tail


def test_normal_values_against_fsum():
    vals = synth.normal_f32(12345, 40 * 32).reshape(40, 32)
    for c in (0, 7, 8, 33, 40):
        F = 8 * (c // 8)
        fr, tc, fs, ts = oracle.full_tile_sum(vals, c, 1.25, 8)
        full = math.fsum([1.25] + [float(x) for x in vals[:F].ravel()])
        tail = math.fsum(float(x) for x in vals[F:c].ravel())
        bound = 2 * (vals.size + 1) * 2.0**-53 * (np.abs(vals[:c]).sum() + 1.25)
        assert abs(fs - full) <= bound and abs(ts - tail) <= bound


def test_batched_matches_single_segments():
    d = synth.batched_segments(num_segments=37, rows=63, lanes=32)
    out = oracle.row_sum_batched(d["values"], d["seg_stride"], 63, 32, d["counts"], d["initial"], 8,
                                 threads=4)
    for s in range(37):
        r = oracle.full_tile_sum(d["values"][s], int(d["counts"][s]), float(d["initial"][s]), 8)
        assert (out["final_row"][s], out["tail_count"][s], out["full_sum"][s], out["tail_sum"][s]) == r
    sel = oracle.row_sum_batched(d["values"], d["seg_stride"], 63, 32, d["counts"], d["initial"], 8,
                                 segments=[5, 0, 36])
    assert list(sel["full_sum"]) == [out["full_sum"][5], out["full_sum"][0], out["full_sum"][36]]


def test_empty_and_full_segments():
    vals = synth.full_tile_case()["values"]
    assert oracle.full_tile_sum(vals, 0, -2.5, 8) == (0, 0, -2.5, 0.0)
    fr, tc, fs, ts = oracle.full_tile_sum(vals, 63, 0.0, 8)
    assert (fr, tc) == (56, 7)
    with pytest.raises(ValueError):
        oracle.full_tile_sum(vals, 64, 0.0, 8)
    with pytest.raises(ValueError):
        oracle.full_tile_sum(vals, -1, 0.0, 8)


def test_config1_golden(golden_dir):
    # Stored by tests/golden/make_golden.py from the seeded generator and the oracle.
    path = os.path.join(golden_dir, "full_tile_case.txt")
    want = {}
    with open(path) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                want[k] = float.fromhex(v) if "x" in v else int(v)
    case = synth.full_tile_case()
    fr, tc, fs, ts = oracle.full_tile_sum(case["values"], case["count"], case["initial"], case["tile_size"])
    assert (fr, tc) == (want["final_row"], want["tail_count"]) == (56, 5)
    assert fs == want["full_sum"] and ts == want["tail_sum"]
    # grid values: the fp64 oracle is the exact sum
    _, _, full, tail = _exact_split(case["values"], 61, case["initial"], 8)
    assert Fraction(fs) == full and Fraction(ts) == tail
