"""GPU parity of the routed row combine (a mixture-of-experts combine): the
weighted payload rows are added in route order with separately rounded f32
products and sums, so the kernels must give the oracle's bits exactly."""
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


def run(loom, torch, d, tuning=None, error=None, offset=0):
    T, W = d["tokens"], d["width"]
    pl = np.ascontiguousarray(d["payload"]).reshape(-1)
    flat = np.zeros(pl.size + offset, np.float32)
    flat[offset:] = pl
    payload = to_dev(flat, torch)[offset:]
    buf, out = guarded(torch, T * W, torch.float32)
    loom.loom_routed_combine(to_dev(d["ids"], torch), to_dev(d["weights"], torch), payload, tokens=T,
                             routes=d["routes"], rows=d["rows"], width=W, out=out, tuning=tuning, error=error)
    torch.cuda.synchronize()
    check_guard(buf, T * W)
    return out.cpu().numpy().reshape(T, W)


def want(d):
    return oracle.routed_combine(d["ids"], d["weights"], d["payload"], threads=8)


# the pages' shapes: 1, 16 and 256 tokens with 8 routes, and 32-route recurrences
@pytest.mark.parametrize("T,R,W", [(1, 8, 2048), (16, 8, 2048), (256, 8, 2048), (16, 32, 1024), (256, 32, 512),
                                   (33, 8, 1540), (5, 1, 4), (7, 3, 100), (9, 0, 64)])
def test_shapes_bitwise(env, T, R, W):
    torch, loom = env
    d = synth.routed_case(tokens=T, routes=R, width=W, seed=17 + T + R + W)
    assert same_bits(run(loom, torch, d), want(d))


@pytest.mark.parametrize("depth,warps,path", [(1, 1, 0), (2, 2, 0), (4, 4, 0), (8, 8, 0), (3, 1, 0), (0, 0, 2)])
def test_schedule_invariance(env, depth, warps, path):
    torch, loom = env
    d = synth.routed_case(tokens=100, routes=8, width=1536, seed=23)
    t = loom.make_tuning(depth=depth, warps_per_cta=warps, path=path)
    assert same_bits(run(loom, torch, d, tuning=t), want(d))


def test_missing_routes_and_cancellation(env):
    # every route missing, every route present, and large values that cancel
    torch, loom = env
    d = synth.routed_case(tokens=12, routes=8, width=512, missing_every=0, seed=29)
    d["ids"][0, :] = -1
    d["ids"][1, ::2] = -1
    d["payload"][d["ids"][2, 0]] *= 2.0 ** 24
    d["payload"][d["ids"][2, 2]] = -d["payload"][d["ids"][2, 0]]
    d["weights"][2, [0, 2]] = 1.0
    got = run(loom, torch, d)
    assert same_bits(got, want(d))
    assert not got[0].any()


def test_many_routes_and_unaligned_take_plain_loads(env):
    torch, loom = env
    d = synth.routed_case(tokens=20, routes=40, width=256, seed=31)   # more than 32 routes
    assert same_bits(run(loom, torch, d), want(d))
    d = synth.routed_case(tokens=20, routes=8, width=256, seed=37)
    assert same_bits(run(loom, torch, d, offset=1), want(d))
    with pytest.raises(loom.LoomError) as e:
        run(loom, torch, d, offset=1, tuning=loom.make_tuning(path=loom.LOOM_PATH_STAGED))
    assert e.value.status == loom.LOOM_ERR_ALIGN


def test_ids_past_the_last_row_are_flagged_and_skipped(env):
    torch, loom = env
    d = synth.routed_case(tokens=10, routes=8, width=128, seed=41)
    d["ids"][3, 5] = d["rows"] + 7
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run(loom, torch, d, error=err, tuning=loom.make_tuning())
    fixed = dict(d, ids=np.where(d["ids"] >= d["rows"], -1, d["ids"]).astype(np.int32))
    assert same_bits(got, want(fixed))
    assert int(err.item()) & loom.LOOM_DEVERR_COUNT_RANGE


def test_injected_stall(env):
    torch, loom = env
    d = synth.routed_case(tokens=16, routes=8, width=1024, missing_every=0, seed=43)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hooks = loom_test_module()
    with injected_stall(hooks):
        got = run(hooks, torch, d, error=err, tuning=hooks.make_tuning(wait_ns=2_000_000))
    assert np.isnan(got).all() and int(err.item()) & loom.LOOM_DEVERR_TIMEOUT
    assert same_bits(run(loom, torch, d), want(d))


@pytest.mark.slow
def test_full_workload_bitwise(env):
    torch, loom = env
    d = synth.routed_case()
    assert same_bits(run(loom, torch, d), want(d))
