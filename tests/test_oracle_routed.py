"""Pins of the oracle's routed row combine (a mixture-of-experts combine).

Loom pages, "Tune loop unrolling and pipelining", section "Separate route and
payload lookahead": per token, each route's row id selects a payload row;
missing ids suppress the weight and payload reads and leave the sum
unchanged; the weighted payload is accumulated in route order in f32.  Pins:
exact integer inputs against int64 arithmetic on a gather, NaN wherever a
missing route or an unreferenced row would be read, a cancellation that only
route order leaves at 0, and a product that only a separately rounded
multiply gives.
"""
import numpy as np
import pytest

import oracle

BIG = 2.0 ** 24


def test_exact_inputs_match_integer_gather():
    rng = np.random.default_rng(3)
    T, R, rows, W = 40, 8, 50, 96
    ids = rng.integers(-3, rows, size=(T, R)).astype(np.int32)   # about 6% missing
    weights = rng.integers(-4, 5, size=(T, R)).astype(np.float32)
    payload = rng.integers(-1000, 1001, size=(rows, W)).astype(np.float32)
    got = oracle.routed_combine(ids, weights, payload)
    valid = ids >= 0
    gathered = payload.astype(np.int64)[np.where(valid, ids, 0)]              # [T][R][W]
    want = (gathered * (weights.astype(np.int64) * valid)[:, :, None]).sum(axis=1)
    assert np.array_equal(got, want.astype(np.float32))


def test_missing_routes_read_nothing():
    T, R, rows, W = 6, 5, 10, 32
    rng = np.random.default_rng(4)
    ids = np.full((T, R), -1, np.int32)
    ids[:, 1] = rng.integers(0, 5, size=T)
    weights = np.full((T, R), np.nan, np.float32)
    weights[:, 1] = 2.0
    payload = np.full((rows, W), np.nan, np.float32)
    payload[:5] = rng.integers(-9, 10, size=(5, W))
    got = oracle.routed_combine(ids, weights, payload)
    assert np.array_equal(got, 2.0 * payload[ids[:, 1]])
    assert not oracle.routed_combine(np.full((2, 3), -1, np.int32), np.zeros((2, 3), np.float32), payload).any()


def test_routes_accumulate_in_order():
    payload = np.array([[BIG], [1.0], [-BIG]], np.float32)
    ones = np.ones((1, 3), np.float32)
    assert oracle.routed_combine(np.array([[0, 1, 2]], np.int32), ones, payload)[0, 0] == 0.0
    assert oracle.routed_combine(np.array([[2, 1, 0]], np.int32), ones, payload)[0, 0] == 1.0


def test_product_and_sum_round_separately():
    # route 0 adds -1; route 1 adds round((1 + 2^-12)^2) = 1 + 2^-11 (the 2^-24 is a
    # tie, rounded to even): the sum is 2^-11; a fused step would keep 2^-11 + 2^-24
    x = np.float32(1 + 2.0 ** -12)
    payload = np.array([[-1.0], [x]], np.float32)
    got = oracle.routed_combine(np.array([[0, 1]], np.int32), np.array([[1.0, x]], np.float32), payload)
    assert got[0, 0] == np.float32(2.0 ** -11)


def test_row_ids_are_checked():
    with pytest.raises(ValueError):
        oracle.routed_combine(np.array([[3]], np.int32), np.ones((1, 1), np.float32), np.zeros((3, 4), np.float32))
