"""Upload of ragged row-sum inputs: only each segment's active rows are copied,
from pinned host memory (read in place by the GPU) or from device memory."""
import numpy as np
import pytest

import synth
from gpu_util import loom_module, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = require_gpu()
    return torch, loom_module()


@pytest.mark.parametrize("S,R,L,offset,source", [(4096, 63, 32, 0, "host"), (300, 1000, 1, 0, "host"),
                                                  (77, 9, 32, 1, "host"), (50, 37, 3, 0, "host"),
                                                  (200, 63, 32, 0, "device"), (1, 5000, 1, 3, "device")])
def test_only_active_rows_are_copied(env, S, R, L, offset, source):
    torch, loom = env
    rng = np.random.default_rng(S + R)
    vals = rng.standard_normal(S * R * L + offset).astype(np.float32)
    counts = rng.integers(0, R + 1, size=S).astype(np.int32)
    src_full = torch.from_numpy(vals)
    src_full = src_full.pin_memory() if source == "host" else src_full.cuda()
    src = src_full[offset:]
    dst_full = torch.full((S * R * L + offset,), -7.0, dtype=torch.float32, device="cuda")
    dst = dst_full[offset:]
    dc = to_dev(counts, torch)
    loom.loom_stage_rows(src, dst, S, R * L, R, L, dc)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().reshape(S, R * L)
    host = vals[offset:].reshape(S, R * L)
    for s in range(S):
        a = counts[s] * L
        assert np.array_equal(got[s, :a].view(np.int32), host[s, :a].view(np.int32)), s
        assert (got[s, a:] == -7.0).all(), s


def test_scalar_count_and_clamped_device_counts(env):
    torch, loom = env
    S, R, L = 10, 8, 32
    vals = torch.arange(S * R * L, dtype=torch.float32).pin_memory()
    dst = torch.zeros(S * R * L, dtype=torch.float32, device="cuda")
    loom.loom_stage_rows(vals, dst, S, R * L, R, L, None, 3)
    torch.cuda.synchronize()
    g = dst.cpu().numpy().reshape(S, R * L)
    assert np.array_equal(g[:, :96], vals.numpy().reshape(S, R * L)[:, :96]) and not g[:, 96:].any()
    dst.zero_()
    dc = to_dev(np.array([-2, 99, 0, 8, 1, 2, 3, 4, 5, 6], np.int32), torch)
    loom.loom_stage_rows(vals, dst, S, R * L, R, L, dc)
    torch.cuda.synchronize()
    g = dst.cpu().numpy().reshape(S, R * L)
    assert not g[0].any() and np.array_equal(g[1], vals.numpy().reshape(S, R * L)[1])


def test_row_sums_of_uploaded_rows_match(env):
    # the upload then the row sum, back to back on one stream
    torch, loom = env
    seg = synth.batched_segments(num_segments=2048)
    host = torch.from_numpy(seg["values"].reshape(-1)).pin_memory()
    dev = torch.full((host.numel(),), float("nan"), dtype=torch.float32, device="cuda")
    counts = to_dev(seg["counts"], torch)
    init = to_dev(seg["initial"], torch)
    loom.loom_stage_rows(host, dev, 2048, 2016, 63, 32, counts)
    a = loom.loom_row_sum_batched(dev, 2048, 2016, 63, 32, counts, init, 8)
    full = to_dev(seg["values"], torch)
    b = loom.loom_row_sum_batched(full, 2048, 2016, 63, 32, counts, init, 8)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
