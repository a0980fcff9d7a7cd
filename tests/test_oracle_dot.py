"""Pins for the packed-int8 oracle (unpack and dequantised dot product).

Checks come from mathematics and from independent library routines:
  * the unpack reading (element j = bits [8j, 8j+7], sign-extended) on a
    hand-worked word and on every byte value in every position, against
    Python's own signed little-endian decoding;
  * every signed-byte product through a one-word dot product;
  * closed-form extremes of a long dot product;
  * random dot products against numpy's int64 matrix product, and the
    scale epilogue against its definition.
"""
import numpy as np
import pytest

import oracle
import synth


def test_unpack_hand_worked_word():
    # 0x80FF017F: bytes from the low end are 0x7F, 0x01, 0xFF, 0x80.
    assert oracle.unpack_word(0x80FF017F) == [127, 1, -1, -128]


def test_unpack_every_byte_every_position():
    for pos in range(4):
        for b in range(256):
            word = b << (8 * pos)
            want = [0, 0, 0, 0]
            want[pos] = int.from_bytes(bytes([b]), "little", signed=True)
            assert oracle.unpack_word(word) == want


def test_unpack_matches_int8_view():
    words = synth.splitmix64(99, 0, 512).astype(np.uint32)
    as_bytes = words.astype("<u4").view(np.int8).reshape(-1, 4)
    for w, b in zip(words[:512], as_bytes):
        assert oracle.unpack_word(int(w)) == [int(t) for t in b]


def test_all_byte_products():
    vals = np.arange(-128, 128, dtype=np.int64)
    for pos in range(4):
        w = np.zeros((256, 4), np.int8)
        x = np.zeros((256, 4), np.int8)
        w[:, pos] = vals
        x[:, pos] = vals
        sw = np.ones(256, np.float32)
        sx = np.ones(256, np.float32)
        acc, y = oracle.i8_dequant_dot(w, sw, x, sx, threads=4)
        assert np.array_equal(acc, np.outer(vals, vals))
        assert np.array_equal(y, np.outer(vals, vals).astype(np.float64))


@pytest.mark.parametrize("k", [4, 16384])
def test_extremes(k):
    sw = np.array([1.0, 1.0, 1.0], np.float32)
    sx = np.array([1.0, 1.0], np.float32)
    w = np.empty((3, k), np.int8)
    w[0] = -128
    w[1] = 127
    w[2, 0::2] = 100
    w[2, 1::2] = -100
    x = np.empty((2, k), np.int8)
    x[0] = -128
    x[1] = 1
    acc, _ = oracle.i8_dequant_dot(w, sw, x, sx)
    assert acc[0, 0] == 128 * 128 * k          # 2**28 at k = 16384
    assert acc[1, 0] == -127 * 128 * k         # -266,338,304 at k = 16384
    assert acc[2, 0] == 0 and acc[2, 1] == 0   # alternating signs cancel
    assert acc[0, 1] == -128 * k


def test_random_against_numpy_matmul():
    d = synth.dequant_batched(n_rows=48, k=1000, batch=5, seed=777)
    acc, y = oracle.i8_dequant_dot(d["w"], d["scale_w"], d["x"], d["scale_x"], threads=3)
    ref = d["w"].astype(np.int64) @ d["x"].astype(np.int64).T
    assert np.array_equal(acc, ref)
    want = d["scale_w"].astype(np.float64)[:, None] * d["scale_x"].astype(np.float64)[None, :] * ref
    assert np.array_equal(y, want)


def test_selected_rows_match_full():
    d = synth.dequant_gemv(n_rows=64, k=256, seed=5)
    acc, y = oracle.i8_dequant_dot(d["w"], d["scale_w"], d["x"], d["scale_x"])
    acc_s, y_s = oracle.i8_dequant_dot(d["w"], d["scale_w"], d["x"], d["scale_x"], rows=[63, 0, 17])
    assert np.array_equal(acc_s, acc[[63, 0, 17]]) and np.array_equal(y_s, y[[63, 0, 17]])


def test_empty_dims():
    acc, y = oracle.i8_dequant_dot(np.zeros((0, 8), np.int8), np.zeros(0, np.float32),
                                   np.zeros((2, 8), np.int8), np.ones(2, np.float32))
    assert acc.shape == (0, 2)
    acc, y = oracle.i8_dequant_dot(np.ones((3, 0), np.int8), np.ones(3, np.float32),
                                   np.ones((2, 0), np.int8), np.ones(2, np.float32))
    assert np.array_equal(acc, np.zeros((3, 2), np.int64))


def test_workgroups_page_example():
    # 1009 elements in 256-wide workgroups need four workgroups
    # (page "Kernels and launch configuration", "Workload is not workgroup count").
    assert oracle.workgroups(1009, 256) == 4
    assert [oracle.workgroups(n, 256) for n in (0, 1, 256, 257, 512)] == [0, 1, 1, 2, 2]
