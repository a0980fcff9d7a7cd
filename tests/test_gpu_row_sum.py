"""GPU parity of the ragged full-tile row sum against the CPU oracle.

Indices (final_row, tail_count) must match bit for bit; sums must be within
a relative 1e-5 of the fp64 oracle.  The kernel's sums are error-free double
words rounded once, so they are in fact within one f32 rounding (2**-24
relative) of the exact sum plus the rounding of the small lo parts (below
1e-9 absolute at these sizes); the tests also check that tighter bound.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (REL_TOL, assert_rel, check_guard, guarded, injected_stall, loom_module, loom_test_module,
                      require_gpu, to_dev)

pytestmark = pytest.mark.gpu
ULP_REL = 2.0**-23   # within one f32 rounding of the exact sum, with margin
ULP_ATOL = 1e-9      # rounding of the lo parts (error terms of size u * |partial sums|)


@pytest.fixture(scope="module")
def env():
    torch = require_gpu()
    return torch, loom_module()


def run_batched(loom, torch, values_dev, S, stride, rows, lanes, counts_dev, init_dev, tile,
                tuning=None, error=None):
    if tuning is None:
        out = loom.loom_row_sum_batched(values_dev, S, stride, rows, lanes, counts_dev, init_dev,
                                        tile, error=error)
    else:
        out = loom.loom_row_sum_batched_ex(values_dev, S, stride, rows, lanes, counts_dev, init_dev,
                                           tile, tuning=tuning, error=error)
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


def compare(got, want, what, exact_sums=False, rel=REL_TOL):
    atol = ULP_ATOL if rel == ULP_REL else 0.0
    fr, tc, fs, ts = got
    assert np.array_equal(fr.astype(np.int64), want["final_row"]), what + " final_row"
    assert np.array_equal(tc.astype(np.int64), want["tail_count"]), what + " tail_count"
    if exact_sums:
        assert np.array_equal(fs.astype(np.float64), want["full_sum"]), what + " full_sum"
        assert np.array_equal(ts.astype(np.float64), want["tail_sum"]), what + " tail_sum"
    else:
        assert_rel(fs, want["full_sum"], rel, what + " full_sum", atol)
        assert_rel(ts, want["tail_sum"], rel, what + " tail_sum", atol)
    # empty sums are exact
    empty_tail = want["tail_count"] == 0
    assert np.all(ts[empty_tail] == 0.0)


def test_full_tile_sum_worked_case(env):
    torch, loom = env
    case = synth.full_tile_case()
    want = oracle.full_tile_sum(case["values"], 61, 0.5, 8)
    fr, tc, fs, ts = loom.loom_full_tile_sum(to_dev(case["values"], torch), 61, 0.5, 8)
    torch.cuda.synchronize()
    assert (int(fr.item()), int(tc.item())) == (56, 5) == want[:2]
    assert abs(fs.item() - want[2]) <= ULP_REL * abs(want[2]) + ULP_ATOL
    assert abs(ts.item() - want[3]) <= ULP_REL * abs(want[3]) + ULP_ATOL


def test_full_tile_sum_iota_bit_exact(env):
    # iota input 1 + 32*row + lane: every partial sum is an integer below 2**24,
    # so the result is exact in any order: 1,606,528.5 and 299,600.
    torch, loom = env
    case = synth.iota_case(rows=63, lanes=32, count=61, initial=0.5)
    fr, tc, fs, ts = loom.loom_full_tile_sum(to_dev(case["values"], torch), 61, 0.5, 8)
    torch.cuda.synchronize()
    assert (fr.item(), tc.item(), fs.item(), ts.item()) == (56, 5, 1606528.5, 299600.0)


@pytest.mark.parametrize("tile", [1, 3, 8, 64])
def test_full_tile_sum_every_count(env, tile):
    torch, loom = env
    case = synth.full_tile_case()
    v = to_dev(case["values"], torch)
    iota = to_dev(synth.iota_case(rows=63, lanes=32)["values"], torch)
    for c in range(64):
        want = oracle.full_tile_sum(case["values"], c, -1.25, tile)
        fr, tc, fs, ts = loom.loom_full_tile_sum(v, c, -1.25, tile)
        got = (fr.item(), tc.item(), fs.item(), ts.item())
        assert got[:2] == want[:2], (c, got, want)
        assert abs(got[2] - want[2]) <= ULP_REL * abs(want[2]) + ULP_ATOL, (c, got, want)
        assert abs(got[3] - want[3]) <= ULP_REL * abs(want[3]) + ULP_ATOL, (c, got, want)
        F = tile * (c // tile)
        fr, tc, fs, ts = loom.loom_full_tile_sum(iota, c, 0.5, tile)
        assert fs.item() == 0.5 + 528 * F + 512 * F * (F - 1)
        t = c - F
        assert ts.item() == 528 * t + 1024 * (t * F + t * (t - 1) // 2)


@pytest.mark.parametrize("lanes", [32, 1])
def test_full_tile_sum_one_lane_and_tiny(env, lanes):
    torch, loom = env
    for rows in (0, 1, 2, 5, 37):
        vals = synth.uniform_grid_f32(1000 + rows, max(rows, 1) * lanes)[: rows * lanes]
        vals = vals.reshape(rows, lanes)
        dv = to_dev(vals if rows else np.zeros((1, lanes), np.float32), torch)
        for c in range(rows + 1):
            want = oracle.full_tile_sum(vals, c, 2.0, 3) if rows else (0, 0, 2.0, 0.0)
            fr, tc, fs, ts = loom.loom_full_tile_sum(dv, c, 2.0, 3, rows=rows, lanes=lanes)
            got = (fr.item(), tc.item(), fs.item(), ts.item())
            assert got[:2] == want[:2]
            assert abs(got[2] - want[2]) <= ULP_REL * abs(want[2]) + ULP_ATOL and \
                abs(got[3] - want[3]) <= ULP_REL * abs(want[3]) + ULP_ATOL, (rows, c, got, want)


def _batched_case(S, rows=63, lanes=32, seed=None):
    return synth.batched_segments(num_segments=S, rows=rows, lanes=lanes, seed=seed)


@pytest.mark.parametrize("S", [1, 15, 16, 17, 1000, 4099])
def test_batched_small_ragged(env, S):
    torch, loom = env
    d = _batched_case(S, seed=0xBEEF + S)
    d["counts"][: min(S, 3)] = [0, 63, 8][: min(S, 3)]   # empty, full and exact-tile segments
    want = oracle.row_sum_batched(d["values"], 2016, 63, 32, d["counts"], d["initial"], 8)
    got = run_batched(loom, torch, to_dev(d["values"], torch), S, 2016, 63, 32,
                      to_dev(d["counts"], torch), to_dev(d["initial"], torch), 8)
    compare(got, want, f"S={S}", rel=ULP_REL)


@pytest.fixture(scope="module")
def config2(env):
    torch, _ = env
    d = _batched_case(65536)
    dev = dict(values=to_dev(d["values"], torch), counts=to_dev(d["counts"], torch),
               initial=to_dev(d["initial"], torch))
    want = oracle.row_sum_batched(d["values"], 2016, 63, 32, d["counts"], d["initial"], 8, threads=8)
    return d, dev, want


def test_batched_full_workload(env, config2):
    torch, loom = env
    d, dev, want = config2
    got = run_batched(loom, torch, dev["values"], 65536, 2016, 63, 32, dev["counts"], dev["initial"], 8)
    compare(got, want, "65536 segments")
    compare(got, want, "65536 segments, one rounding", rel=ULP_REL)


def test_batched_depth_and_path_invariance(env, config2):
    # Read-ahead depth, segments per warp and the load path change the schedule
    # only: every setting must return identical bits.
    torch, loom = env
    d, dev, want = config2
    ref = run_batched(loom, torch, dev["values"], 65536, 2016, 63, 32, dev["counts"], dev["initial"], 8)
    for depth in (1, 2, 3, 4):
        for upw, warps, chunk in ((1, 1, 4096), (4, 2, 8192), (32, 4, 512), (7, 1, 2048)):
            t = loom.make_tuning(depth=depth, path=loom.LOOM_PATH_STAGED, units_per_warp=upw,
                                 warps_per_cta=warps, chunk_bytes=chunk)
            got = run_batched(loom, torch, dev["values"], 65536, 2016, 63, 32, dev["counts"],
                              dev["initial"], 8, tuning=t)
            for a, b in zip(got, ref):
                assert np.array_equal(a.view(np.int32), b.view(np.int32)), (depth, upw, warps, chunk)
    t = loom.make_tuning(path=loom.LOOM_PATH_DIRECT)
    got = run_batched(loom, torch, dev["values"], 65536, 2016, 63, 32, dev["counts"], dev["initial"], 8,
                      tuning=t)
    for a, b in zip(got, ref):
        assert np.array_equal(a.view(np.int32), b.view(np.int32)), "direct path"
    again = run_batched(loom, torch, dev["values"], 65536, 2016, 63, 32, dev["counts"], dev["initial"], 8)
    for a, b in zip(again, ref):
        assert np.array_equal(a.view(np.int32), b.view(np.int32)), "run to run"


@pytest.mark.parametrize("rows,chunk", [(64, 8192), (100, 16384), (127, 16384), (20, 2560)])
def test_segment_ring_sizes(env, rows, chunk):
    # Segments that fill the one-copy-per-segment ring exactly (64 x 32 lanes in 8 KiB),
    # larger segments under a larger ring (100 and 127 rows in 16 KiB: one segment in
    # flight beside part of the next), and a ring that is not a power of two.  Same bits
    # as the chunked kernel and the direct path, and the oracle's sums.
    torch, loom = env
    S = 3001
    d = _batched_case(S, rows=rows, seed=rows * 7 + chunk)
    vals, counts, init = to_dev(d["values"], torch), to_dev(d["counts"], torch), to_dev(d["initial"], torch)
    stride = rows * 32
    want = oracle.row_sum_batched(d["values"], stride, rows, 32, d["counts"], d["initial"], 8, threads=8)
    L = loom.loom_launch_config(loom.LOOM_OP_ROW_SUM_BATCHED, [S, rows, 32, 1, 0, 0, 0, chunk])
    assert L["kernel"] == loom.LOOM_KERNEL_ROWSUM_SEGMENTS
    ref = None
    for depth in (1, 2, 4):
        t = loom.make_tuning(depth=depth, path=loom.LOOM_PATH_STAGED, chunk_bytes=chunk)
        got = run_batched(loom, torch, vals, S, stride, rows, 32, counts, init, 8, tuning=t)
        compare(got, want, f"rows {rows} ring {chunk} depth {depth}", rel=ULP_REL)
        if ref is None:
            ref = got
        for a, b in zip(got, ref):
            assert np.array_equal(a.view(np.int32), b.view(np.int32)), depth
    for t in (loom.make_tuning(path=loom.LOOM_PATH_STAGED, chunk_bytes=2048),
              loom.make_tuning(path=loom.LOOM_PATH_DIRECT)):
        got = run_batched(loom, torch, vals, S, stride, rows, 32, counts, init, 8, tuning=t)
        for a, b in zip(got, ref):
            assert np.array_equal(a.view(np.int32), b.view(np.int32)), "chunked / direct"


def test_unaligned_input_takes_direct_path_with_same_bits(env):
    torch, loom = env
    S = 300
    d = _batched_case(S, seed=99)
    flat = d["values"].reshape(-1)
    buf = torch.zeros(flat.size + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(flat).cuda()
    counts, init = to_dev(d["counts"], torch), to_dev(d["initial"], torch)
    staged = run_batched(loom, torch, buf[1:].clone(), S, 2016, 63, 32, counts, init, 8)
    direct = run_batched(loom, torch, buf[1:], S, 2016, 63, 32, counts, init, 8)  # 4-byte aligned only
    for a, b in zip(staged, direct):
        assert np.array_equal(a.view(np.int32), b.view(np.int32))
    want = oracle.row_sum_batched(d["values"], 2016, 63, 32, d["counts"], d["initial"], 8)
    compare(direct, want, "unaligned", rel=ULP_REL)


def test_strided_segments_and_null_initial(env):
    torch, loom = env
    S, rows, lanes, stride = 97, 20, 32, 20 * 32 + 36   # padded segments, stride % 4 == 0
    vals = synth.uniform_grid_f32(4242, S * stride)
    counts = synth.uniform_int(4343, S, 0, rows).astype(np.int32)
    want = oracle.row_sum_batched(vals, stride, rows, lanes, counts, None, 5)
    got = run_batched(loom, torch, to_dev(vals, torch), S, stride, rows, lanes, to_dev(counts, torch),
                      None, 5)
    compare(got, want, "strided", rel=ULP_REL)


def test_guard_bands_and_over_dispatch(env):
    torch, loom = env
    S = 37   # three CTAs of 16 segments: the last one over-dispatched by 11
    d = _batched_case(S, seed=7)
    bufs = [guarded(torch, S, dt) for dt in (torch.int32, torch.int32, torch.float32, torch.float32)]
    loom.loom_row_sum_batched(to_dev(d["values"], torch), S, 2016, 63, 32, to_dev(d["counts"], torch),
                              to_dev(d["initial"], torch), 8, out=tuple(v for _, v in bufs))
    torch.cuda.synchronize()
    for buf, _ in bufs:
        check_guard(buf, S)
    want = oracle.row_sum_batched(d["values"], 2016, 63, 32, d["counts"], d["initial"], 8)
    compare([v.cpu().numpy() for _, v in bufs], want, "guarded", rel=ULP_REL)


def test_out_of_range_counts_are_clamped_and_flagged(env):
    torch, loom = env
    S = 40
    d = _batched_case(S, seed=11)
    bad = d["counts"].copy()
    bad[3], bad[17], bad[39] = -5, 64, 1000
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_batched(loom, torch, to_dev(d["values"], torch), S, 2016, 63, 32, to_dev(bad, torch),
                      to_dev(d["initial"], torch), 8, error=err)
    assert int(err.item()) & loom.LOOM_DEVERR_COUNT_RANGE
    clamped = np.clip(bad, 0, 63).astype(np.int32)
    want = oracle.row_sum_batched(d["values"], 2016, 63, 32, clamped, d["initial"], 8)
    compare(got, want, "clamped", rel=ULP_REL)


def test_injected_stall_times_out_and_device_stays_usable(env):
    torch, loom = env
    S = 64
    d = _batched_case(S, seed=12)
    dv, dc, di = to_dev(d["values"], torch), to_dev(d["counts"], torch), to_dev(d["initial"], torch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hooks = loom_test_module()
    t = hooks.make_tuning(wait_ns=2_000_000, path=loom.LOOM_PATH_STAGED)
    with injected_stall(hooks):
        fr, tc, fs, ts = run_batched(hooks, torch, dv, S, 2016, 63, 32, dc, di, 8, tuning=t, error=err)
    assert int(err.item()) & loom.LOOM_DEVERR_TIMEOUT
    has_data = d["counts"] > 0
    assert np.isnan(fs[has_data]).all()
    want = oracle.row_sum_batched(d["values"], 2016, 63, 32, d["counts"], d["initial"], 8)
    assert np.array_equal(fr.astype(np.int64), want["final_row"])   # indices need no data
    got = run_batched(loom, torch, dv, S, 2016, 63, 32, dc, di, 8)     # the context still works
    compare(got, want, "after timeout", rel=ULP_REL)


def test_non_default_stream(env):
    torch, loom = env
    S = 500
    d = _batched_case(S, seed=13)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dv, dc, di = to_dev(d["values"], torch), to_dev(d["counts"], torch), to_dev(d["initial"], torch)
        out = loom.loom_row_sum_batched(dv, S, 2016, 63, 32, dc, di, 8)
    s.synchronize()
    want = oracle.row_sum_batched(d["values"], 2016, 63, 32, d["counts"], d["initial"], 8)
    compare([t.cpu().numpy() for t in out], want, "stream", rel=ULP_REL)


@pytest.mark.parametrize("n_rows,n_cols,tile", [(257, 1000, 8), (64, 4099, 3), (5, 16, 8)])
def test_wide_rows_small(env, n_rows, n_cols, tile):
    torch, loom = env
    d = synth.wide_rows(n_rows=n_rows, n_cols=n_cols, tile_size=tile, seed=n_rows * 31 + n_cols)
    counts = d["counts"].copy()
    counts[:3] = [0, n_cols, min(n_cols, 7)][:3]
    want = oracle.row_sum_batched(d["values"], n_cols, n_cols, 1, counts, None, tile)
    got = run_batched(loom, torch, to_dev(d["values"], torch), n_rows, n_cols, n_cols, 1,
                      to_dev(counts, torch), None, tile)
    compare(got, want, "wide", rel=ULP_REL)


def test_wide_rows_full_workload(env):
    torch, loom = env
    d = synth.wide_rows()
    want = oracle.row_sum_batched(d["values"], 16384, 16384, 1, d["counts"], None, 8, threads=8)
    got = run_batched(loom, torch, to_dev(d["values"], torch), 16384, 16384, 16384, 1,
                      to_dev(d["counts"], torch), None, 8)
    compare(got, want, "16384 x 16384")
    compare(got, want, "16384 x 16384, one rounding", rel=ULP_REL)


@pytest.mark.parametrize("path", [0, 2])   # staged ring, plain loads
def test_nan_past_the_active_rows_is_never_read(env, path):
    # every value past a segment's count (or a wide row's length) is NaN: a
    # stray read would turn its sum into NaN
    torch, loom = env
    d = _batched_case(2000, seed=0xACE)
    v = d["values"].reshape(2000, 63, 32).copy()
    for s, c in enumerate(d["counts"]):
        v[s, c:] = np.nan
    want = oracle.row_sum_batched(v, 2016, 63, 32, d["counts"], d["initial"], 8)
    t = loom.make_tuning(path=path)
    got = run_batched(loom, torch, to_dev(v, torch), 2000, 2016, 63, 32, to_dev(d["counts"], torch),
                      to_dev(d["initial"], torch), 8, tuning=t)
    assert np.isfinite(got[2]).all() and np.isfinite(got[3]).all()
    compare(got, want, f"poisoned segments path {path}", rel=ULP_REL)
    w = synth.wide_rows(n_rows=300, n_cols=5000, seed=0xACF)
    vals = w["values"].copy()
    for r, L in enumerate(w["counts"]):
        vals[r, L:] = np.nan
    want = oracle.row_sum_batched(vals, 5000, 5000, 1, w["counts"], None, 8)
    got = run_batched(loom, torch, to_dev(vals, torch), 300, 5000, 5000, 1, to_dev(w["counts"], torch), None, 8,
                      tuning=t)
    assert np.isfinite(got[2]).all() and np.isfinite(got[3]).all()
    compare(got, want, f"poisoned wide rows path {path}", rel=ULP_REL)


@pytest.mark.parametrize("path", [0, 2])
def test_infinities_and_nan_follow_ieee(env, path):
    # +inf, -inf, both, and NaN in the full-tile rows or in the tail rows:
    # the sums are what IEEE addition gives (the oracle's double sums, rounded)
    torch, loom = env
    S = 64
    d = _batched_case(S, seed=0xF00)
    v = d["values"].reshape(S, 63, 32).copy()
    c = np.full(S, 61, np.int32)                       # full-tile rows 0..55, tail rows 56..60
    specials = [(1, 3, 5, np.inf), (2, 10, 0, -np.inf), (3, 4, 1, np.inf), (3, 50, 7, -np.inf),
                (4, 20, 20, np.nan), (5, 58, 3, np.inf), (6, 57, 1, np.nan), (7, 62, 9, np.inf)]
    for s, r, l, x in specials:                        # (row 62 of segment 7 is past its count)
        v[s, r, l] = x
    want = oracle.row_sum_batched(v, 2016, 63, 32, c, d["initial"], 8)
    got = run_batched(loom, torch, to_dev(v, torch), S, 2016, 63, 32, to_dev(c, torch),
                      to_dev(d["initial"], torch), 8, tuning=loom.make_tuning(path=path))
    for g, w in ((got[2], want["full_sum"]), (got[3], want["tail_sum"])):
        w32 = w.astype(np.float32)
        assert np.array_equal(np.isnan(g), np.isnan(w32))
        inf = np.isinf(w32)
        assert np.array_equal(g[inf], w32[inf])
        fin = np.isfinite(w32)
        assert np.all(np.abs(g[fin] - w[fin]) <= ULP_REL * np.abs(w[fin]) + ULP_ATOL)
    assert np.isinf(got[2][1]) and got[2][1] > 0 and np.isnan(got[2][3]) and np.isnan(got[2][4])
    assert np.isinf(got[3][5]) and np.isnan(got[3][6]) and np.isfinite(got[2][7]) and np.isfinite(got[3][7])
