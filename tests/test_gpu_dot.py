"""GPU parity of the packed-int8 dequantised dot product and the unpack kernel.

Integer accumulators must match the oracle bit for bit; y must be within a
relative 1e-5 of the fp64 oracle (the kernel's three f32 roundings give at
most about 2e-7).
"""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import (assert_rel, check_guard, guarded, injected_stall, loom_module, loom_test_module, require_gpu,
                      to_dev)

pytestmark = pytest.mark.gpu
Y_REL = 1e-5
Y_TIGHT = 4 * 2.0**-24   # three roundings: sw*sx, (float)acc, the product


@pytest.fixture(scope="module")
def env():
    torch = require_gpu()
    return torch, loom_module()


def packed(a: np.ndarray) -> np.ndarray:
    """int8 [r][k] -> int32 [r][k/4]: the same bytes read as little-endian words."""
    a = np.ascontiguousarray(a, dtype=np.int8)
    if a.shape[1] == 0:
        return np.zeros((a.shape[0], 0), np.int32)
    return np.ascontiguousarray(a.view("<i4"), dtype=np.int32)


def run_dot(loom, torch, d, tuning=None, error=None, want_acc=True, workspace="auto"):
    w = to_dev(packed(d["w"]), torch)
    x = to_dev(packed(d["x"]), torch)
    sw, sx = to_dev(d["scale_w"], torch), to_dev(d["scale_x"], torch)
    n, k = d["w"].shape
    b = d["x"].shape[0]
    # NaN / sentinel outputs: a row the kernel failed to write cannot pass
    y = torch.full((n, b), float("nan"), dtype=torch.float32, device="cuda")
    acc = torch.full((n, b), -7777, dtype=torch.int32, device="cuda") if want_acc else None
    if tuning is None and error is None:
        loom.loom_i8_dequant_dot(w, sw, n, k, x, sx, b, y=y, acc=acc, workspace=workspace)
    else:
        loom.loom_i8_dequant_dot_ex(w, sw, n, k, x, sx, b, y=y, acc=acc, workspace=workspace,
                                    tuning=tuning, error=error)
    torch.cuda.synchronize()
    return y.cpu().numpy(), (acc.cpu().numpy() if acc is not None else None)


def same_bits(a, b):
    return np.array_equal(np.asarray(a).view(np.int32), np.asarray(b).view(np.int32))


def check(d, y, acc, what, rows=None):
    want_acc, want_y = oracle.i8_dequant_dot(d["w"], d["scale_w"], d["x"], d["scale_x"], threads=8)
    assert np.array_equal(acc.astype(np.int64), want_acc), what + ": acc"
    assert_rel(y, want_y, Y_REL, what + ": y")
    assert_rel(y, want_y, Y_TIGHT, what + ": y (three roundings)")


def small(n, k, b, seed):
    return synth.dequant_batched(n_rows=n, k=k, batch=b, seed=seed)


@pytest.mark.parametrize("n,k,b", [(1, 16, 1), (37, 1040, 1), (37, 1040, 2), (37, 1040, 3),
                                   (64, 4096, 4), (37, 1040, 5), (33, 4112, 16), (9, 512, 17),
                                   (70, 2048, 33), (37, 0, 3), (5, 16, 16)])
def test_dot_small(env, n, k, b):
    torch, loom = env
    d = small(n, k, b, seed=n * 1000 + k + b)
    y, acc = run_dot(loom, torch, d)
    check(d, y, acc, f"{n}x{k}x{b}")


@pytest.mark.parametrize("k", [4, 12, 20, 1044])
def test_dot_k_not_multiple_of_16_takes_direct(env, k):
    torch, loom = env
    for b in (1, 4, 16):
        d = small(19, k, b, seed=k * 7 + b)
        y, acc = run_dot(loom, torch, d)
        check(d, y, acc, f"k={k} b={b}")


def test_dot_extremes(env):
    torch, loom = env
    k = 16384
    w = np.empty((4, k), np.int8)
    w[0], w[1], w[2] = -128, 127, 0
    w[3, 0::2], w[3, 1::2] = 100, -100
    x = np.empty((2, k), np.int8)
    x[0], x[1] = -128, 127
    d = dict(w=w, x=x, scale_w=np.ones(4, np.float32), scale_x=np.array([1.0, 0.5], np.float32))
    y, acc = run_dot(loom, torch, d)
    assert acc[0, 0] == 2**28 and acc[1, 0] == -127 * 128 * k and acc[0, 1] == -128 * 127 * k
    assert acc[2].tolist() == [0, 0] and acc[3].tolist() == [0, 0]
    check(d, y, acc, "extremes")


@pytest.mark.parametrize("k,b", [(131068, 16), (131068, 1), (131056, 16), (131056, 2), (131056, 3)])
def test_dot_at_the_largest_k(env, k, b):
    # |acc| <= 128 * 128 * k stays below 2^31 up to k = 131068, the largest k the
    # call accepts: -128 x -128 over all of k sums to 2,147,418,112 there (plain
    # loads: its rows are not 16-byte aligned).  131056, the largest multiple of 16,
    # also goes through the staged dp4a kernels and the tensor-core kernels (whole
    # rows, split bands, band clusters, whole bands) with 1024 units of k.
    torch, loom = env
    n = 40
    d = small(n, k, b, seed=k + b)
    w, x = d["w"].copy(), d["x"].copy()
    w[0], w[1] = -128, 127
    w[2, 0::2], w[2, 1::2] = -128, 127
    x[0] = -128
    if b > 1:
        x[1] = 127
    d = dict(w=w, x=x, scale_w=d["scale_w"], scale_x=d["scale_x"])
    runs = [("auto", None), ("direct", loom.make_tuning(path=loom.LOOM_PATH_DIRECT))]
    if k % 16 != 0:
        # rows of 131068 bytes are not 16-byte aligned: the staged kernels cannot take them
        with pytest.raises(loom.LoomError) as e:
            run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_STAGED))
        assert e.value.status == loom.LOOM_ERR_ALIGN
    else:
        runs.append(("staged", loom.make_tuning(path=loom.LOOM_PATH_STAGED)))
    if k % 16 == 0 and b >= 3:
        runs += [(f"tensor schedule {sc}", loom.make_tuning(path=loom.LOOM_PATH_TENSOR, tc_schedule=sc))
                 for sc in (4, 2, 3, 1)]
    ref = None
    for what, tu in runs:
        y, acc = run_dot(loom, torch, d, tuning=tu)
        assert acc[0, 0] == 16384 * k and acc[1, 0] == -127 * 128 * k, what
        assert acc[2, 0] == -128 * (-128 + 127) * (k // 2), what
        if b > 1:
            assert acc[0, 1] == -128 * 127 * k and acc[1, 1] == 127 * 127 * k, what
        if ref is None:
            check(d, y, acc, f"k={k} b={b} {what}")
            ref = (y, acc)
        else:
            assert np.array_equal(acc, ref[1]) and same_bits(y, ref[0]), what


def test_dot_path_and_depth_invariance(env):
    torch, loom = env
    for b in (1, 16):
        d = small(129, 8192, b, seed=31 + b)
        ref_y, ref_acc = run_dot(loom, torch, d)
        check(d, ref_y, ref_acc, f"b={b}")
        for depth in (1, 2, 3, 4):
            t = loom.make_tuning(depth=depth, path=loom.LOOM_PATH_STAGED)
            y, acc = run_dot(loom, torch, d, tuning=t)
            assert np.array_equal(acc, ref_acc) and np.array_equal(y.view(np.int32), ref_y.view(np.int32))
        y, acc = run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_DIRECT))
        assert np.array_equal(acc, ref_acc) and np.array_equal(y.view(np.int32), ref_y.view(np.int32))


@pytest.mark.parametrize("n,k,b", [(37, 16400, 1), (300, 8192, 2), (5, 48, 1), (1000, 4096, 1), (2, 32784, 2)])
def test_lanes_across_k_schedule_invariance(env, n, k, b):
    # Blocks of rows per CTA whose 8 KiB pieces the warps share out (rows split between
    # warps, ragged last pieces, fewer pieces than warps): any warps per CTA, CTAs per SM
    # and ring depth give the default's bits and the oracle's integers.
    torch, loom = env
    d = small(n, k, b, seed=5 * n + k + b)
    ref_y, ref_acc = run_dot(loom, torch, d)
    check(d, ref_y, ref_acc, f"lanes across k {n}x{k}x{b}")
    for warps, ctas, depth in ((1, 1, 1), (2, 3, 2), (4, 1, 4), (8, 2, 2), (4, 7, 3), (8, 32, 1), (1, 16, 8)):
        t = loom.make_tuning(depth=depth, warps_per_cta=warps, units_per_warp=ctas, path=loom.LOOM_PATH_STAGED)
        y, acc = run_dot(loom, torch, d, tuning=t)
        assert np.array_equal(acc, ref_acc) and same_bits(y, ref_y), (warps, ctas, depth)


@pytest.mark.parametrize("n,k,b", [(128, 1024, 16), (129, 1040, 3), (300, 2064, 7), (5, 16, 16),
                                   (257, 16384, 16), (64, 131056, 16), (130, 128, 4), (2049, 4112, 16)])
def test_tensor_core_matches_dp4a_bitwise(env, n, k, b):
    # Row tails (n % 128), k tails (k % 128), one-unit k, the longest k the
    # library accepts, partial batches and a unit list split unevenly over the
    # whole grid: the tensor-core kernel must give the dp4a kernels' bits and
    # the oracle's integers.
    torch, loom = env
    d = small(n, k, b, seed=n + 7 * k + 31 * b)
    y_tc, acc_tc = run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_TENSOR))
    y_dp, acc_dp = run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_STAGED))
    assert np.array_equal(acc_tc, acc_dp)
    assert same_bits(y_tc, y_dp)
    check(d, y_tc, acc_tc, f"tensor {n}x{k}x{b}")


def test_tensor_core_exact_at_group_bound(env):
    # 1024 products of -128 * -128 per accumulator reach 2**24 exactly.
    torch, loom = env
    k = 4096
    w = np.full((256, k), -128, np.int8)
    w[1::2] = 127
    x = np.full((16, k), -128, np.int8)
    x[3] = 127
    d = dict(w=w, x=x, scale_w=np.ones(256, np.float32), scale_x=np.ones(16, np.float32))
    y, acc = run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_TENSOR))
    assert acc[0, 0] == 128 * 128 * k and acc[1, 0] == -127 * 128 * k and acc[1, 3] == 127 * 127 * k
    check(d, y, acc, "group bound")


# (stages, units per stage, A buffers, pipelines per CTA, band schedule); 0 = default
TC_SCHEDULES = [(0, 0, 0, 0, 0), (1, 2, 0, 0, 0), (1, 1, 0, 0, 0), (2, 1, 0, 0, 0), (4, 1, 0, 0, 0),
                (0, 0, 0, 1, 0), (3, 2, 7, 1, 0), (1, 4, 0, 1, 0), (8, 1, 7, 1, 0), (3, 3, 0, 1, 0),
                (0, 0, 0, 0, 1), (0, 0, 0, 0, 2), (0, 0, 0, 0, 3), (4, 1, 0, 0, 3), (0, 0, 0, 1, 3),
                (1, 2, 0, 1, 2), (0, 0, 0, 1, 1),
                (0, 0, 0, 0, 4), (2, 0, 0, 0, 4), (4, 1, 3, 2, 4), (8, 0, 2, 0, 4), (6, 0, 3, 0, 4)]


@pytest.mark.parametrize("n,k,b", [(384, 8192, 16), (2049, 4112, 16), (128, 1024, 5), (3, 256, 9),
                                   (1024, 16384, 16), (128, 16384, 16), (200, 65536, 16)])
def test_tensor_core_schedule_invariance(env, n, k, b):
    # Every schedule -- a cluster per band, split or whole bands, stage depth
    # and width, A buffers, one or two pipelines per CTA -- gives the same bits.
    torch, loom = env
    d = small(n, k, b, seed=99 + n + k)
    ref_y, ref_acc = run_dot(loom, torch, d)
    check(d, ref_y, ref_acc, "tensor default")
    for ws in ("auto", None):
        for depth, ups, na, pipes, sched in TC_SCHEDULES:
            if sched == 2 and ws is None:
                continue   # the split schedule needs the workspace
            t = loom.make_tuning(depth=depth, path=loom.LOOM_PATH_TENSOR, tc_units_per_stage=ups,
                                 tc_a_buffers=na, tc_pipelines=pipes, tc_schedule=sched)
            y, acc = run_dot(loom, torch, d, tuning=t, workspace=ws)
            what = f"ws={ws} schedule={(depth, ups, na, pipes, sched)}"
            assert np.array_equal(acc, ref_acc), what
            assert same_bits(y, ref_y), what


@pytest.mark.parametrize("n,k,b", [(9729, 2048, 16), (9729, 2048, 5), (10000, 4112, 16), (4864, 2048, 3),
                                   (1, 16384, 16), (153, 1152, 16), (50000, 2064, 16)])
def test_tensor_core_whole_rows(env, n, k, b):
    # CTAs owning whole rows: two blocks per CTA (9729 rows: 65 per CTA, blocks of 33),
    # six blocks per CTA (50000 rows: 329 per CTA, blocks of 55, with a k tail),
    # a short last CTA, k tails and k quarters that end past k (zero-filled units), one
    # row, one row per CTA; the bits of the dp4a kernels and the oracle's integers.
    torch, loom = env
    d = small(n, k, b, seed=7 * n + k + b)
    y, acc = run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_TENSOR, tc_schedule=4))
    check(d, y, acc, f"rows {n}x{k}x{b}")
    y2, acc2 = run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_STAGED))
    assert np.array_equal(acc2, acc) and same_bits(y2, y)


def test_tensor_core_whole_rows_batches_over_16(env):
    # Passes of 16, 16 and 1 vectors through the row-block kernel (y rows 33 wide).
    torch, loom = env
    d = small(4864, 2048, 33, seed=333)
    y, acc = run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_TENSOR, tc_schedule=4))
    check(d, y, acc, "rows b=33")


def test_tensor_core_schedules_that_do_not_fit(env):
    torch, loom = env
    d = small(128, 1024, 16, seed=5)
    for depth, ups, na, pipes, sched in [(3, 2, 0, 0, 0), (0, 0, 4, 0, 0), (0, 0, 8, 1, 0), (2, 2, 2, 0, 0),
                                         (8, 2, 0, 1, 0), (0, 0, 6, 1, 0), (0, 3, 0, 0, 0), (3, 0, 0, 0, 4),
                                         (0, 0, 4, 0, 4), (0, 2, 0, 0, 4), (0, 0, 0, 1, 4)]:
        t = loom.make_tuning(depth=depth, path=loom.LOOM_PATH_TENSOR, tc_units_per_stage=ups,
                             tc_a_buffers=na, tc_pipelines=pipes, tc_schedule=sched)
        with pytest.raises(loom.LoomError) as e:
            run_dot(loom, torch, d, tuning=t)
        assert e.value.status == loom.LOOM_ERR_ARG
    with pytest.raises(loom.LoomError) as e:   # split schedule, no workspace
        run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_TENSOR, tc_schedule=2),
                workspace=None)
    assert e.value.status == loom.LOOM_ERR_ARG


def test_tensor_core_workspace_reuse_and_size(env):
    # One explicit workspace (garbage to start with) through many calls of
    # different shapes, then one too short.
    torch, loom = env
    shapes = [(2049, 4112, 16), (300, 2064, 7), (8192 // 8, 16384, 16), (129, 1040, 3)]
    need = max(loom.loom_i8_dequant_dot_workspace_bytes(n, k, b) for n, k, b in shapes)
    assert need > 0
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device="cuda")
    for rep in range(2):
        for i, (n, k, b) in enumerate(shapes):
            d = small(n, k, b, seed=11 * i + rep)
            y, acc = run_dot(loom, torch, d, workspace=ws)
            check(d, y, acc, f"reuse {rep} {n}x{k}x{b}")
    n, k, b = shapes[0]
    short = loom.loom_i8_dequant_dot_workspace_bytes(n, k, b) - 256
    with pytest.raises(loom.LoomError) as e:
        run_dot(loom, torch, small(n, k, b, seed=1), workspace=(ws.data_ptr(), short))
    assert e.value.status == loom.LOOM_ERR_ARG
    assert loom.loom_i8_dequant_dot_workspace_bytes(n, k, 2) == 0   # dp4a path: none


def test_tensor_core_injected_stall(env):
    # The stalled call reports a timeout and NaN outputs (its split bands'
    # records are marked invalid); the next call through the same workspace is exact.
    torch, loom = env
    for n, k, sched in ((256, 4096, 0), (2049, 4112, 0), (9729, 2048, 4)):
        d = small(n, k, 16, seed=41 + n)
        ws = loom.dot_workspace(n, k, 16)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        hooks = loom_test_module()
        t = hooks.make_tuning(wait_ns=2_000_000, path=loom.LOOM_PATH_TENSOR, tc_schedule=sched)
        with injected_stall(hooks):
            y, acc = run_dot(hooks, torch, d, tuning=t, error=err, workspace=ws)
        assert int(err.item()) & loom.LOOM_DEVERR_TIMEOUT
        assert np.isnan(y).all() and (acc == np.iinfo(np.int32).min).all()
        y, acc = run_dot(loom, torch, d, workspace=ws)
        check(d, y, acc, "after tensor-core timeout")


def test_tensor_core_batches_over_16(env):
    # Passes of 16 vectors reuse the workspace one after another.
    torch, loom = env
    for b in (19, 32, 35):
        d = small(700, 2048, b, seed=b)
        y, acc = run_dot(loom, torch, d)
        check(d, y, acc, f"b={b}")


def test_dot_guard_bands(env):
    torch, loom = env
    n, k, b = 35, 2048, 5
    d = small(n, k, b, seed=77)
    ybuf, y = guarded(torch, n * b, torch.float32)
    abuf, acc = guarded(torch, n * b, torch.int32)
    loom.loom_i8_dequant_dot(to_dev(packed(d["w"]), torch), to_dev(d["scale_w"], torch), n, k,
                             to_dev(packed(d["x"]), torch), to_dev(d["scale_x"], torch), b,
                             y=y, acc=acc)
    torch.cuda.synchronize()
    check_guard(ybuf, n * b)
    check_guard(abuf, n * b)
    check(d, y.cpu().numpy().reshape(n, b), acc.cpu().numpy().reshape(n, b), "guarded")


def test_dot_without_acc_output(env):
    torch, loom = env
    d = small(40, 1024, 16, seed=3)
    y, acc = run_dot(loom, torch, d, want_acc=False)
    assert acc is None
    _, want_y = oracle.i8_dequant_dot(d["w"], d["scale_w"], d["x"], d["scale_x"])
    assert_rel(y, want_y, Y_REL, "y only")


def test_dot_injected_stall(env):
    torch, loom = env
    for b in (1, 16):
        d = small(64, 4096, b, seed=5 + b)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        hooks = loom_test_module()
        t = hooks.make_tuning(wait_ns=2_000_000, path=loom.LOOM_PATH_STAGED)
        with injected_stall(hooks):
            y, acc = run_dot(hooks, torch, d, tuning=t, error=err)
        assert int(err.item()) & loom.LOOM_DEVERR_TIMEOUT
        assert np.isnan(y).all()
        y, acc = run_dot(loom, torch, d)
        check(d, y, acc, "after timeout")


@pytest.fixture(scope="module")
def weights():
    return synth.dequant_weights()


def test_gemv_full_workload(env, weights):
    torch, loom = env
    d = synth.dequant_gemv()
    y, acc = run_dot(loom, torch, d)
    check(d, y, acc, "8192 x 16384 x 1")


def test_batched_full_workload(env, weights):
    torch, loom = env
    d = synth.dequant_batched()
    y, acc = run_dot(loom, torch, d)
    check(d, y, acc, "8192 x 16384 x 16")
    # the same bits through the split schedule and through whole bands
    for sched in (2, 1, 3):
        y2, acc2 = run_dot(loom, torch, d, tuning=loom.make_tuning(path=loom.LOOM_PATH_TENSOR, tc_schedule=sched))
        assert np.array_equal(acc2, acc) and same_bits(y2, y), sched


def test_unpack_every_byte_and_over_dispatch(env):
    torch, loom = env
    n = 1009  # four CTAs of 256; the last runs 15 idle invocations
    words = synth.splitmix64(2024, 0, n).astype(np.uint32)
    words[:256] = np.arange(256, dtype=np.uint32) * 0x01010101  # every byte in every position
    buf, out = guarded(torch, 4 * n, torch.float32)
    loom.loom_i8_unpack(to_dev(words.view(np.int32), torch), n, out)
    torch.cuda.synchronize()
    check_guard(buf, 4 * n)
    got = out.cpu().numpy()
    want = np.array([oracle.unpack_word(int(w)) for w in words], dtype=np.float32).reshape(-1)
    assert np.array_equal(got, want)
    # unaligned output (4-byte only) uses scalar stores, same values
    ubuf = torch.full((4 * n + 1,), float("nan"), device="cuda")
    loom.loom_i8_unpack(to_dev(words.view(np.int32), torch), n, ubuf[1:])
    torch.cuda.synchronize()
    assert np.array_equal(ubuf[1:].cpu().numpy(), want) and np.isnan(ubuf[0].item())
