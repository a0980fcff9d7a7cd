"""The largest units the calls accept: a row-sum unit of 2^31 - 1 (lanes 1) or
2^31 - 32 (lanes 32) elements, and routed rows 2^31 - 4 (staged) or 2^31 - 1
(plain loads) floats wide.  Index arithmetic near INT32_MAX must neither wrap
nor drop data.

Inputs follow v[i] = 0.25 * ((i mod 7) - 3): every partial sum is a small
multiple of 0.25, so every f32 addition is exact and the expected sums have a
closed form, S(n) = sum over i < n of ((i mod 7) - 3) = sum over j < n mod 7 of
(j - 3), since each period of seven sums to zero.  (About 24 GB of device
memory.)"""
import numpy as np
import pytest

from gpu_util import loom_module, require_gpu

pytestmark = pytest.mark.gpu

N = 2**31 - 1


def S(n: int) -> int:
    return sum(j - 3 for j in range(n % 7))


@pytest.fixture(scope="module")
def big():
    torch = require_gpu()
    loom = loom_module()
    buf = torch.empty(N + 4, dtype=torch.float32, device="cuda")
    step = 1 << 27
    for a in range(0, N + 4, step):
        b = min(N + 4, a + step)
        i = torch.arange(a, b, dtype=torch.int64, device="cuda")
        buf[a:b] = ((i % 7) - 3).to(torch.float32) * 0.25
        del i
    torch.cuda.synchronize()
    yield torch, loom, buf
    del buf
    torch.cuda.empty_cache()


def test_row_sum_unit_of_2_31_minus_1_elements(big):
    torch, loom, buf = big
    # counts that leave the 16-byte-block count within one chunk of INT32_MAX and a tail
    for lanes, rows, c in ((1, N, N - 3), (32, N // 32, N // 32 - 1)):
        F = (c // 8) * 8
        want_full, want_tail = 0.25 * S(F * lanes), 0.25 * (S(c * lanes) - S(F * lanes))
        assert want_full != 0 and want_tail != 0 and c * lanes > 2**31 - 2048
        counts = torch.tensor([c], dtype=torch.int32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        fr, tc, fs, ts = loom.loom_row_sum_batched(buf, 1, rows * lanes, rows, lanes, counts, None, 8,
                                                   error=err)
        torch.cuda.synchronize()
        assert int(fr.item()) == F and int(tc.item()) == c - F, lanes
        assert fs.item() == want_full, (lanes, fs.item(), want_full)
        assert ts.item() == want_tail, (lanes, ts.item(), want_tail)
        assert int(err.item()) == 0


def test_routed_row_of_2_31_minus_4_floats(big):
    torch, loom, buf = big
    W = 2**31 - 4                       # a multiple of 4: bulk copies
    payload = buf[:W].view(1, W)
    ids = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    wts = torch.full((1, 1), 0.5, dtype=torch.float32, device="cuda")
    out = torch.full((1, W), float("nan"), dtype=torch.float32, device="cuda")
    loom.loom_routed_combine(ids, wts, payload, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, payload * 0.5)    # 0 + 0.5 * x: one exact rounding
    del out


def test_routed_plain_loads_row_of_2_31_minus_1_floats(big):
    # width not a multiple of 4: plain loads; a missing route leaves the zero sum
    torch, loom, buf = big
    W = N
    payload = buf[:W].view(1, W)
    ids = torch.full((1, 1), -1, dtype=torch.int32, device="cuda")
    wts = torch.full((1, 1), 0.5, dtype=torch.float32, device="cuda")
    out = torch.full((1, W), float("nan"), dtype=torch.float32, device="cuda")
    loom.loom_routed_combine(ids, wts, payload, out=out)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(out).item()) == 0
    del out


def test_packed_dot_instance_of_2_31_words():
    # One instance of 2^20 records x 2048 lanes: 2^31 words, so element offsets pass
    # INT32_MAX (8 GiB of words, 4 GiB of scales, 1 GiB of activations).  Every byte is
    # 1, every scale 1.0 and every activation of record r is 0.25 ((r mod 7) - 3): each
    # record adds (r mod 7) - 3 to every lane in four exact quarter steps, so a lane
    # ends at initial + S(count) exactly.  Full and ragged counts; the TMA-staged and
    # the plain-load paths.
    torch = require_gpu()
    loom = loom_module()
    R, L, ST = 2**20, 2048, 64
    fields = torch.full((1, R, L), 0x01010101, dtype=torch.int32, device="cuda")
    scales = torch.full((1, R, L), 0x3C00, dtype=torch.int16, device="cuda")
    r = torch.arange(R, device="cuda")
    rhs = ((r % 7) - 3).to(torch.float32).mul_(0.25).view(1, R, 1, 1).expand(1, R, ST, 4).contiguous()
    del r
    initial = torch.arange(L, dtype=torch.float32, device="cuda").view(1, L) * 0.5
    for count in (R, R - 5):
        want = initial + float(S(count))
        for what, tu in (("staged", loom.make_tuning(path=loom.LOOM_PATH_STAGED)),
                         ("direct", loom.make_tuning(path=loom.LOOM_PATH_DIRECT))):
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            out = torch.full((1, L), float("nan"), dtype=torch.float32, device="cuda")
            loom.loom_packed_dot_ex(fields, scales, rhs, None, count, initial, out=out, error=err, tuning=tu)
            torch.cuda.synchronize()
            assert torch.equal(out, want), (what, count)
            assert int(err.item()) == 0, what
    del fields, scales, rhs
    torch.cuda.empty_cache()
