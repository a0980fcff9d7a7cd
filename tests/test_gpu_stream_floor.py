"""The read-only streaming probe (loom_stream_floor) reads every byte of its range.

The probe folds the words it loads into a per-thread checksum and writes the
sink only when a checksum equals a fixed constant.  A zero buffer with that
constant planted in one word therefore writes the sink exactly when the probe
read that word: planted in a middle stage, and in the short last stage of a
range that is not a whole number of 8 KiB stages, for every schedule.
"""
import pytest

from gpu_util import loom_module, require_gpu

MAGIC = 0x9E3779B9
SCHEDULES = [(0, 4, 4), (0, 8, 2), (1, 4, 4), (1, 8, 8), (2, 1, 3), (2, 2, 12), (2, 4, 6), (2, 8, 1)]

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = require_gpu()
    return torch, loom_module()


@pytest.mark.parametrize("kind,depth,cps", SCHEDULES)
def test_probe_reads_every_planted_word(env, kind, depth, cps):
    torch, loom = env
    nbytes = 5 * 8192 + 48
    for word in (3 * 8192 // 4 + 5, 5 * 8192 // 4 + 2, 0):
        buf = torch.zeros(nbytes // 4, dtype=torch.int32, device="cuda")
        buf[word] = MAGIC - (1 << 32)
        sink = torch.zeros(1, dtype=torch.int64, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        loom.loom_stream_floor(buf, nbytes, kind, depth, cps, sink, error=err)
        torch.cuda.synchronize()
        assert int(sink.item()) == MAGIC, (kind, depth, cps, word)
        assert int(err.item()) == 0
    # nothing planted: nothing written
    buf = torch.zeros(nbytes // 4, dtype=torch.int32, device="cuda")
    sink = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    loom.loom_stream_floor(buf, nbytes, kind, depth, cps, sink)
    torch.cuda.synchronize()
    assert int(sink.item()) == -1
