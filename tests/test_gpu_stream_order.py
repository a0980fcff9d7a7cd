"""Stream order across library calls.  Every kernel is launched so that it may be
scheduled while the previous kernel on the stream drains, and waits for that
kernel before touching memory; these chains check read-after-write and
write-after-read between back-to-back calls with no host synchronisation."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import loom_module, require_gpu, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = require_gpu()
    return torch, loom_module()


def same_bits(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.int32), np.asarray(b, np.float32).view(np.int32))


def test_read_after_write_chains(env):
    # unpack writes floats that sum_rows reads at once; the dot writes y that
    # sum_rows reads at once; 40 rounds with fresh inputs each time
    torch, loom = env
    S, R, L = 64, 16, 32
    n_words = S * R * L // 4
    s = torch.cuda.Stream()
    d = synth.dequant_batched(n_rows=256, k=1024, batch=16, seed=5)
    w = to_dev(d["w"].view("<i4"), torch)
    x = to_dev(d["x"].view("<i4"), torch)
    sw, sx = to_dev(d["scale_w"], torch), to_dev(d["scale_x"], torch)
    counts = to_dev(np.full(S, R, np.int32), torch)
    floats = torch.empty(S * R * L, dtype=torch.float32, device="cuda")
    y = torch.empty((256, 16), dtype=torch.float32, device="cuda")
    sums1, sums2 = [], []
    words_host = []
    with torch.cuda.stream(s):
        for i in range(40):
            words = synth.int8_bytes(1000 + i, 4 * n_words).view("<i4")
            words_host.append(words)
            packed = to_dev(words, torch)
            loom.loom_i8_unpack(packed, n_words, out=floats, stream=s)
            sums1.append(loom.loom_sum_rows(floats, S, R * L, R, L, 1, counts, 0, stream=s))
            loom.loom_i8_dequant_dot(w, sw, 256, 1024, x, sx, 16, y=y, stream=s)
            sums2.append(loom.loom_sum_rows(y, 32, 8 * 16, 8, 16, 1, None, 8, stream=s))
    s.synchronize()
    y_host = y.cpu().numpy()
    want2 = oracle.lane_sums(y_host.reshape(32, 8, 16), np.full(32, 8, np.int32))
    for i in range(40):
        vals = words_host[i].view(np.int8).astype(np.float32).reshape(S, R, L)
        assert same_bits(sums1[i].cpu().numpy(), oracle.lane_sums(vals, np.full(S, R, np.int32))), i
        assert same_bits(sums2[i].cpu().numpy(), want2), i


def test_write_after_read(env):
    # sum_rows reads a buffer that the very next call overwrites
    torch, loom = env
    S, R, L = 512, 64, 32
    s = torch.cuda.Stream()
    a = synth.lane_segments(num_segments=S, rows=R, lanes=L, width=1, seed=7)
    vals = to_dev(a["values"], torch)
    counts = to_dev(np.full(S, R, np.int32), torch)
    n_words = S * R * L // 4
    junk = to_dev(synth.int8_bytes(9, 4 * n_words).view("<i4"), torch)
    with torch.cuda.stream(s):
        out = loom.loom_sum_rows(vals, S, R * L, R, L, 1, counts, 0, stream=s)
        loom.loom_i8_unpack(junk, n_words, out=vals, stream=s)     # overwrites what sum_rows read
    s.synchronize()
    assert same_bits(out.cpu().numpy(), oracle.lane_sums(a["values"], np.full(S, R, np.int32)))
