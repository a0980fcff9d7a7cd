"""The benchmark's step at full size: the four workloads run as two concurrent
lanes (CUDA streams forked and joined by events) return the same bits as the
same kernels run one at a time on one stream, step after step, and sampled
outputs agree with the oracle.  The end-to-end step (uploads from pinned host
memory, the kernels, read-back, per lane) returns the same bits to the host."""
import numpy as np
import pytest

import oracle
from gpu_util import assert_rel, loom_module, require_gpu

pytestmark = pytest.mark.gpu

SUM_REL, SUM_ATOL = 2.0**-23, 1e-9   # one f32 rounding of the exact sum (with margin)
Y_REL = 4 * 2.0**-24                # three roundings: sw*sx, (float)acc, the product


def outputs(work):
    o = work.o
    return [t.cpu().numpy().copy() for t in list(o["seg"]) + list(o["wide"]) + [o["y1"], o["y16"]]]


def poison(work, torch):
    o = work.o
    for t in list(o["seg"]) + list(o["wide"]) + [o["y1"], o["y16"]]:
        t.fill_(-1 if not t.dtype.is_floating_point else float("nan"))
    torch.cuda.synchronize()   # the fills run on torch's current stream, the step on its own


def same_bits(a, b):
    return a.dtype == b.dtype and np.array_equal(a.view(np.int32), b.view(np.int32))


def test_two_lane_step_matches_serial_kernels_and_oracle():
    torch = require_gpu()
    loom = loom_module()
    import bench
    inp = bench.make_inputs()
    s = torch.cuda.Stream()
    work = bench.DeviceWorkload(inp, torch, loom, s)
    step = bench.Step(torch, work)
    assert sorted(n for lane in bench.STEP_LANES for n in lane) == sorted(bench.ORDER)
    # the batched dot reads a weight array of its own
    assert work.d["wb"].data_ptr() != work.d["w"].data_ptr()

    poison(work, torch)
    with torch.cuda.stream(s):
        for name in bench.ORDER:
            work.launch(name)
    s.synchronize()
    serial = outputs(work)

    for rep in range(3):
        poison(work, torch)
        with torch.cuda.stream(s):
            for _ in range(2):          # back-to-back steps: no host sync between them
                step.run(s)
        s.synchronize()
        for i, (a, b) in enumerate(zip(outputs(work), serial)):
            assert same_bits(a, b), (rep, i)

    # the two-lane step captured as a CUDA graph (fork and join become graph edges)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step.run(s)
    poison(work, torch)
    g.replay()
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(zip(outputs(work), serial)):
        assert same_bits(a, b), ("graph", i)
    del g

    # the one-stream schedule (bench.py --lanes 1) through the same Step
    one = bench.Step(torch, work, bench.ONE_LANE)
    poison(work, torch)
    with torch.cuda.stream(s):
        one.run(s)
        one.run(s)
    s.synchronize()
    for i, (a, b) in enumerate(zip(outputs(work), serial)):
        assert same_bits(a, b), ("one lane", i)

    # sampled outputs against the oracle
    rng = np.random.default_rng(12)
    seg = inp["segments"]
    pick = np.sort(rng.choice(seg["num_segments"], 256, replace=False))
    want = oracle.row_sum_batched(seg["values"], 2016, 63, 32, seg["counts"], seg["initial"], 8, segments=pick)
    fr, tc, fs, ts = serial[0:4]
    assert np.array_equal(fr[pick].astype(np.int64), want["final_row"])
    assert np.array_equal(tc[pick].astype(np.int64), want["tail_count"])
    assert_rel(fs[pick], want["full_sum"], SUM_REL, "segments full_sum", SUM_ATOL)
    assert_rel(ts[pick], want["tail_sum"], SUM_REL, "segments tail_sum", SUM_ATOL)
    bat = inp["batched"]
    rows = np.sort(rng.choice(8192, 64, replace=False))
    acc, y = oracle.i8_dequant_dot(bat["w"], bat["scale_w"], bat["x"], bat["scale_x"], rows=rows)
    assert_rel(serial[9][rows], y, Y_REL, "batched y")
    g = inp["gemv"]
    acc, y = oracle.i8_dequant_dot(g["w"], g["scale_w"], g["x"], g["scale_x"], rows=rows)
    assert_rel(serial[8][rows], y, Y_REL, "gemv y")

    # end to end: with every device input poisoned first, one step must upload the
    # inputs (the ragged arrays' active rows only), run and read back the same bits
    for t in work.d.values():
        t.fill_(float("nan") if t.dtype.is_floating_point else -1)
    poison(work, torch)   # (synchronises the fills above too)
    e2e = bench.E2EStep(inp, torch, loom, work)
    with torch.cuda.stream(s):
        e2e.run(s)
    s.synchronize()
    host = [t.numpy() for k in ("seg", "wide", "y1", "y16") for t in e2e.host_out[k]]
    for i, (a, b) in enumerate(zip(host, serial)):
        assert same_bits(a, b), ("e2e", i)
