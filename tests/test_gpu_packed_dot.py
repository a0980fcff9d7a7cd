"""GPU parity of the pages' packed signed-byte dot (f16 scales, f32 activations,
ordered f32 accumulation).

The sum is a defined sequence of f32 fused multiply-adds, so the kernel must
give the oracle's bits exactly, for every schedule.
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import check_guard, guarded, injected_stall, loom_module, loom_test_module, require_gpu, to_dev

pytestmark = pytest.mark.gpu

# the 14 record counts of the check: empty, short loops, partial and full stages
LENGTHS = [0, 1, 2, 3, 4, 5, 7, 8, 9, 15, 16, 17, 127, 128]


@pytest.fixture(scope="module")
def env():
    torch = require_gpu()
    return torch, loom_module()


def run(loom, torch, d, tuning=None, error=None, with_initial=True, device_counts=True, offset=0):
    """Runs the call on device copies of d (inputs shifted by `offset` elements
    inside larger buffers when asked); returns the host output."""
    def dev(a, dtype=None):
        a = np.ascontiguousarray(a)
        if offset == 0:
            return to_dev(a, torch)
        flat = np.zeros(a.size + offset, a.dtype)
        flat[offset:] = a.reshape(-1)
        return to_dev(flat, torch)[offset:]
    P, R, L, S = d["problems"], d["records"], d["lanes"], d["streams"]
    f = dev(d["fields"])
    sc = dev(d["scales"].view(np.int16))
    rhs = dev(d["rhs"])
    init = dev(d["initial"]) if with_initial else None
    counts = to_dev(d["counts"], torch) if device_counts else None
    count = int(d["counts"][0])
    buf, out = guarded(torch, P * L, torch.float32)
    if tuning is None and error is None:
        loom.loom_packed_dot(f, sc, rhs, counts, count, init, problems=P, records=R, lanes=L, streams=S,
                             out=out)
    else:
        loom.loom_packed_dot_ex(f, sc, rhs, counts, count, init, problems=P, records=R, lanes=L,
                                streams=S, out=out, tuning=tuning, error=error)
    torch.cuda.synchronize()
    check_guard(buf, P * L)
    return out.cpu().numpy().reshape(P, L)


def want(d, with_initial=True):
    return oracle.packed_dot(d["fields"], d["scales"], d["rhs"], d["counts"],
                             d["initial"] if with_initial else None, threads=8)


def same_bits(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.int32), np.asarray(b, np.float32).view(np.int32))


def test_fourteen_lengths_bitwise(env):
    torch, loom = env
    d = synth.packed_dot_case(problems=len(LENGTHS), records=128, lanes=2048, streams=64, counts=LENGTHS,
                              seed=101)
    got = run(loom, torch, d)
    assert same_bits(got, want(d))
    assert same_bits(got[0], d["initial"][0])   # count 0: the initial sums, untouched


@pytest.mark.parametrize("depth,rps,path", [(1, 1, 0), (1, 8, 0), (2, 3, 0), (3, 8, 0), (4, 2, 0),
                                            (8, 4, 0), (5, 7, 0), (1, 32, 0), (0, 0, 2), (3, 5, 2)])
def test_schedule_invariance(env, depth, rps, path):
    # the read-ahead depth, records per stage and the load path never change a bit
    torch, loom = env
    d = synth.packed_dot_case(problems=6, records=40, lanes=512, streams=64, counts=[0, 1, 9, 17, 33, 40],
                              seed=202)
    t = loom.make_tuning(depth=depth, units_per_warp=rps, path=path)
    assert same_bits(run(loom, torch, d, tuning=t), want(d))


@pytest.mark.parametrize("P,R,L,S,counts", [
    (3, 5, 264, 7, [5, 0, 3]),        # a partial lane block, streams not a power of two (staged)
    (2, 9, 1000, 64, [9, 4]),         # lanes not a multiple of 8: plain loads
    (2, 6, 256, 128, [6, 6]),         # more streams than one copy row holds: plain loads
    (1, 3, 8, 1, [3]),                # one stream shared by every lane
    (4, 200, 40, 3, [200, 199, 1, 0]),
])
def test_ragged_shapes(env, P, R, L, S, counts):
    torch, loom = env
    d = synth.packed_dot_case(problems=P, records=R, lanes=L, streams=S, counts=counts, seed=303 + L)
    assert same_bits(run(loom, torch, d), want(d))
    assert same_bits(run(loom, torch, d, with_initial=False), want(d, with_initial=False))
    if len(set(counts)) == 1:
        assert same_bits(run(loom, torch, d, device_counts=False), want(d))


@pytest.mark.parametrize("streams,tuning_kw", [(64, None), (48, None), (64, {"depth": 3, "units_per_warp": 24})])
def test_ctas_run_on_across_tiles(env, streams, tuning_kw):
    # 1344 tiles of 256 lanes, more than the grid holds CTAs (at most seven per SM with the
    # default stages, one with 24-record stages): each CTA's ring runs on from one tile into
    # the next, across instances of different lengths; 48 streams do not divide 128, so the
    # two lanes of a thread read different activations
    torch, loom = env
    P = 168
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert P * 2048 // 256 > 7 * sms
    d = synth.packed_dot_case(problems=P, records=24, lanes=2048, streams=streams,
                              counts=[(7 * i) % 25 for i in range(P)], seed=707 + streams)
    t = loom.make_tuning(**tuning_kw) if tuning_kw else None
    assert same_bits(run(loom, torch, d, tuning=t), want(d))


def test_unaligned_inputs_take_plain_loads(env):
    torch, loom = env
    d = synth.packed_dot_case(problems=2, records=16, lanes=256, streams=64, counts=[16, 11], seed=404)
    assert same_bits(run(loom, torch, d, offset=1), want(d))   # 4-byte (2-byte for scales) offsets
    t = loom.make_tuning(path=loom.LOOM_PATH_STAGED)
    with pytest.raises(loom.LoomError) as e:
        run(loom, torch, d, tuning=t, offset=1)
    assert e.value.status == loom.LOOM_ERR_ALIGN


def test_device_counts_out_of_range_are_clamped(env):
    torch, loom = env
    d = synth.packed_dot_case(problems=3, records=12, lanes=64, streams=8, counts=[-3, 12, 40], seed=505)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run(loom, torch, d, error=err, tuning=loom.make_tuning())
    clamped = dict(d, counts=np.array([0, 12, 12], np.int32))
    assert same_bits(got, want(clamped))
    assert int(err.item()) & loom.LOOM_DEVERR_COUNT_RANGE


def test_injected_stall_reports_and_recovers(env):
    torch, loom = env
    d = synth.packed_dot_case(problems=2, records=32, lanes=512, streams=64, counts=[32, 20], seed=606)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hooks = loom_test_module()
    with injected_stall(hooks):
        got = run(hooks, torch, d, tuning=hooks.make_tuning(wait_ns=2_000_000), error=err)
    assert np.isnan(got).all()
    assert int(err.item()) & loom.LOOM_DEVERR_TIMEOUT
    assert same_bits(run(loom, torch, d), want(d))   # the context is still usable


@pytest.mark.slow
def test_full_workload_bitwise(env):
    # 128 instances x 128 records x 2048 lanes x 64 streams, the launch the benchmark times
    torch, loom = env
    d = synth.packed_dot_case()
    assert same_bits(run(loom, torch, d), want(d))
