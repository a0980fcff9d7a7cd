"""The seeded generators: published SplitMix64 outputs, determinism, ranges."""
import numpy as np

import synth


def test_splitmix64_published_outputs():
    # First outputs of SplitMix64 started from state 0 (the sequence printed with
    # the reference C implementation, splitmix64.c).
    got = [int(v) for v in synth.splitmix64(0, 0, 3)]
    assert got == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_counter_form_slices_agree():
    whole = synth.splitmix64(1234, 0, 5000)
    assert np.array_equal(synth.splitmix64(1234, 1700, 300), whole[1700:2000])


def test_chunked_generation_is_deterministic():
    n = (1 << 21) + 77   # several chunks
    a = synth.uniform_grid_f32(42, n)
    b = synth.uniform_grid_f32(42, n)
    assert np.array_equal(a, b)
    assert np.array_equal(synth.uniform_grid_f32(42, 1000), a[:1000])


def test_distribution_ranges():
    g = synth.uniform_grid_f32(1, 100000)
    assert g.min() >= -1.0 and g.max() < 1.0
    assert np.all(g.astype(np.float64) * 2**23 == np.round(g.astype(np.float64) * 2**23))
    c = synth.uniform_int(2, 100000, 0, 63)
    assert c.min() == 0 and c.max() == 63
    f = synth.uniform_f32(3, 100000, 1e-3, 1e-2)
    assert f.min() >= np.float32(1e-3) and f.max() <= np.float32(1e-2)
    b = synth.int8_bytes(4, 100003)
    assert b.dtype == np.int8 and b.size == 100003 and b.min() == -128 and b.max() == 127
    n = synth.normal_f32(5, 200001)
    assert n.size == 200001 and abs(float(n.mean())) < 0.01 and abs(float(n.std()) - 1) < 0.01


def test_workload_shapes_small():
    d = synth.batched_segments(num_segments=10)
    assert d["values"].shape == (10, 63, 32) and d["counts"].dtype == np.int32
    w = synth.wide_rows(n_rows=4, n_cols=100)
    assert w["values"].shape == (4, 100) and w["counts"].max() <= 100
    g = synth.dequant_gemv(n_rows=8, k=64)
    bt = synth.dequant_batched(n_rows=8, k=64, batch=3)
    assert np.array_equal(g["w"], bt["w"])          # the same weights
    assert g["x"].shape == (1, 64) and bt["x"].shape == (3, 64)
    assert not np.array_equal(bt["x"][0], bt["w"][0])
