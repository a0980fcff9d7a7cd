"""GPU parity of the per-lane f32 sums (the pages' sum_rows, sum_vector_rows and
guarded ragged rows).  Each result is a fixed sequence of f32 additions, so the
kernels must give the oracle's bits exactly, for every schedule."""
import itertools

import numpy as np
import pytest

import oracle
import synth
from gpu_util import check_guard, guarded, injected_stall, loom_module, loom_test_module, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = require_gpu()
    return torch, loom_module()


def same_bits(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.int32), np.asarray(b, np.float32).view(np.int32))


def run_rows(loom, torch, v, counts, width, tuning=None, error=None, device_counts=True, offset=0):
    S, R, L = v.shape[:3]
    flat = np.zeros(v.size + offset, np.float32)
    flat[offset:] = v.reshape(-1)
    dv = to_dev(flat, torch)[offset:]
    buf, out = guarded(torch, S * L, torch.float32)
    c = to_dev(np.asarray(counts, np.int32), torch) if device_counts else None
    loom.loom_sum_rows(dv, S, R * L * width, R, L, width, c, int(counts[0]), out=out, tuning=tuning, error=error)
    torch.cuda.synchronize()
    check_guard(buf, S * L)
    return out.cpu().numpy().reshape(S, L)


def run_guarded(loom, torch, v, counts, columns, active, tuning=None, error=None):
    S, R, L = v.shape[:3]
    buf, out = guarded(torch, S * L, torch.float32)
    loom.loom_sum_guarded_rows(to_dev(v, torch), S, R * L * 4, R, L, to_dev(np.asarray(counts, np.int32), torch),
                               0, columns, active, out=out, tuning=tuning, error=error)
    torch.cuda.synchronize()
    check_guard(buf, S * L)
    return out.cpu().numpy().reshape(S, L)


def test_sum_rows_page_check_cases(env, golden_dir):
    # the pages' input 1 + 32 row + lane and their printed expectations, counts 0..5, 63, 64
    torch, loom = env
    values = synth.iota_case(rows=64, lanes=32, count=0)["values"]
    cases = []
    with open(f"{golden_dir}/sum_rows_iota.txt") as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                cases.append(tuple(int(t) for t in line.split()))
    seg = np.ascontiguousarray(np.broadcast_to(values, (len(cases), 64, 32)))
    got = run_rows(loom, torch, seg, [c for c, _, _ in cases], 1)
    for i, (count, offset, step) in enumerate(cases):
        assert np.array_equal(got[i], (offset + step * np.arange(32)).astype(np.float32)), count


@pytest.mark.parametrize("width", [1, 4])
def test_random_segments_bitwise(env, width):
    torch, loom = env
    d = synth.lane_segments(num_segments=1000, rows=64, lanes=32, width=width, seed=31 + width)
    got = run_rows(loom, torch, d["values"], d["counts"], width)
    assert same_bits(got, oracle.lane_sums(d["values"], d["counts"], width=width, threads=8))


@pytest.mark.parametrize("width", [1, 4])
@pytest.mark.parametrize("depth,warps,upw,chunk,path", [(1, 1, 1, 512, 0), (2, 2, 3, 4096, 0), (4, 4, 8, 1024, 0),
                                                        (8, 1, 2, 2048, 0), (3, 2, 1, 16384, 0), (0, 0, 0, 0, 2)])
def test_schedule_invariance(env, width, depth, warps, upw, chunk, path):
    torch, loom = env
    d = synth.lane_segments(num_segments=333, rows=40, lanes=32, width=width, seed=41)
    t = loom.make_tuning(depth=depth, warps_per_cta=warps, units_per_warp=upw, chunk_bytes=chunk, path=path)
    got = run_rows(loom, torch, d["values"], d["counts"], width, tuning=t)
    assert same_bits(got, oracle.lane_sums(d["values"], d["counts"], width=width))


@pytest.mark.parametrize("lanes,width,offset", [(7, 1, 0), (12, 1, 0), (32, 1, 1), (3, 4, 0), (32, 4, 2), (1, 1, 0)])
def test_narrow_and_unaligned(env, lanes, width, offset):
    torch, loom = env
    d = synth.lane_segments(num_segments=50, rows=17, lanes=lanes, width=width, seed=51 + lanes)
    got = run_rows(loom, torch, d["values"], d["counts"], width, offset=offset)
    assert same_bits(got, oracle.lane_sums(d["values"], d["counts"], width=width))


def test_host_count_and_clamped_device_counts(env):
    torch, loom = env
    d = synth.lane_segments(num_segments=9, rows=20, lanes=32, width=1, seed=61)
    got = run_rows(loom, torch, d["values"], np.full(9, 13, np.int32), 1, device_counts=False)
    assert same_bits(got, oracle.lane_sums(d["values"], np.full(9, 13, np.int32)))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    counts = np.array([-5, 0, 20, 21, 7, 99, 3, 1, 2], np.int32)
    got = run_rows(loom, torch, d["values"], counts, 1, error=err, tuning=loom.make_tuning())
    assert same_bits(got, oracle.lane_sums(d["values"], np.clip(counts, 0, 20)))
    assert int(err.item()) & loom.LOOM_DEVERR_COUNT_RANGE


def test_injected_stall(env):
    torch, loom = env
    d = synth.lane_segments(num_segments=40, rows=64, lanes=32, width=4, seed=71)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    counts = np.maximum(d["counts"], 1)
    hooks = loom_test_module()
    with injected_stall(hooks):
        got = run_rows(hooks, torch, d["values"], counts, 4, error=err, tuning=hooks.make_tuning(wait_ns=2_000_000))
    assert np.isnan(got).all() and int(err.item()) & loom.LOOM_DEVERR_TIMEOUT
    assert same_bits(run_rows(loom, torch, d["values"], counts, 4), oracle.lane_sums(d["values"], counts, width=4))


def test_guarded_rows_combinations(env):
    # row counts x inner extents x active lanes x seeds, bit for bit (360 combinations)
    torch, loom = env
    counts = [0, 1, 3, 4, 5, 17, 62, 63, 31, 8]
    combos = list(itertools.product(counts, [0, 1, 2, 3, 4], [0, 1, 31, 32], [0, 1]))
    assert len(combos) == 400
    combos = [c for c in combos if not (c[1] == 0 and c[2] in (1, 31))][:360]
    for columns, active in sorted({(c[1], c[2]) for c in combos}):
        group = [c for c in combos if c[1] == columns and c[2] == active]
        seg_counts = np.array([c[0] for c in group], np.int32)
        v = np.concatenate([synth.lane_segments(num_segments=1, rows=63, lanes=32, width=4,
                                                seed=1000 + 10 * c[0] + c[3])["values"] for c in group])
        got = run_guarded(loom, torch, v, seg_counts, columns, active)
        assert same_bits(got, oracle.guarded_rows(v, seg_counts, columns, active)), (columns, active)


def test_guarded_rows_schedules(env):
    torch, loom = env
    d = synth.lane_segments(num_segments=200, rows=63, lanes=32, width=4, seed=81)
    want = oracle.guarded_rows(d["values"], d["counts"], 3, 29)
    for t in (None, loom.make_tuning(depth=1), loom.make_tuning(depth=4, units_per_warp=3, chunk_bytes=2048),
              loom.make_tuning(path=loom.LOOM_PATH_DIRECT)):
        assert same_bits(run_guarded(loom, torch, d["values"], d["counts"], 3, 29, tuning=t), want)


@pytest.mark.slow
@pytest.mark.parametrize("width", [1, 4])
def test_full_workloads_bitwise(env, width):
    torch, loom = env
    S = 65536 if width == 1 else 16384
    d = synth.lane_segments(num_segments=S, rows=64, lanes=32, width=width)
    got = run_rows(loom, torch, d["values"], d["counts"], width)
    assert same_bits(got, oracle.lane_sums(d["values"], d["counts"], width=width, threads=16))


@pytest.mark.slow
def test_guarded_full_workload_bitwise(env):
    torch, loom = env
    d = synth.lane_segments(num_segments=16384, rows=63, lanes=32, width=4)
    got = run_guarded(loom, torch, d["values"], d["counts"], 4, 32)
    assert same_bits(got, oracle.guarded_rows(d["values"], d["counts"], 4, 32, threads=16))


@pytest.mark.parametrize("width,path", [(1, 0), (4, 0), (1, 2), (4, 2)])
def test_nan_past_the_active_rows_is_never_read(env, width, path):
    torch, loom = env
    d = synth.lane_segments(num_segments=500, rows=63, lanes=32, width=width, seed=91 + width)
    v = d["values"].copy()
    for s, c in enumerate(d["counts"]):
        v[s, c:] = np.nan
    t = loom.make_tuning(path=path)
    got = run_rows(loom, torch, v, d["counts"], width, tuning=t)
    assert np.isfinite(got).all()
    assert same_bits(got, oracle.lane_sums(v, d["counts"], width=width))
    if width == 4:   # the guarded rows also never read past the count
        got = run_guarded(loom, torch, v, d["counts"], 4, 32, tuning=t)
        assert np.isfinite(got).all()
        assert same_bits(got, oracle.guarded_rows(v, d["counts"], 4, 32))
