"""loom_i8_dequant_dot_noalloc: the tensor-core dot with the library's fixed
device scratch instead of a caller workspace.

On the GPU its results must be the bits of loom_i8_dequant_dot (given a
workspace) on consecutive calls that reuse the same scratch; on the CPU its
argument checks run before any device access.
"""
import numpy as np
import pytest

import oracle
import synth

A = 1 << 20   # an aligned fake device address (never dereferenced on the CPU)


@pytest.fixture(scope="module")
def loom():
    import __graft_entry__
    __graft_entry__.build()
    import int8_dequant_dot_gb300 as loom
    return loom


def test_noalloc_argument_checks(loom):
    lib = loom.library()
    d = lambda w, n, k, x, b, y=A: lib.loom_i8_dequant_dot_noalloc(w, A, n, k, x, A, b, y, None, None)
    assert d(None, 0, 64, None, 4) == loom.LOOM_OK        # no rows: nothing to do
    assert d(None, 4, 64, A, 4) == loom.LOOM_ERR_NULL
    assert d(A, 4, 64, A, 4, None) == loom.LOOM_ERR_NULL
    assert d(A, 4, 62, A, 4) == loom.LOOM_ERR_SHAPE
    assert d(A, -1, 64, A, 4) == loom.LOOM_ERR_SHAPE
    assert d(A + 2, 4, 64, A, 4) == loom.LOOM_ERR_ALIGN


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_on_two_calls(loom):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    # calls through the same scratch: a grid of uneven band splits; 33 vectors
    # (three passes, the last of one vector below the tensor-core threshold, each
    # pass's streaming kernel following the previous pass's finishing kernel);
    # then the full 8192 x 16384 x 16 workload
    for n, k, b, seed in ((2049, 4112, 16, 7), (1500, 2048, 33, 8), (8192, 16384, 16, None)):
        d = synth.dequant_batched() if seed is None else synth.dequant_batched(n_rows=n, k=k, batch=b, seed=seed)
        need = loom.loom_i8_dequant_dot_workspace_bytes(n, k, b)
        assert 0 < need <= 8 << 20
        w, x = t(d["w"].view("<i4")), t(d["x"].view("<i4"))
        sw, sx = t(d["scale_w"]), t(d["scale_x"])
        y0 = torch.full((n, b), float("nan"), device="cuda")
        a0 = torch.full((n, b), -7777, dtype=torch.int32, device="cuda")
        loom.loom_i8_dequant_dot(w, sw, n, k, x, sx, b, y=y0, acc=a0, workspace=loom.dot_workspace(n, k, b))
        y1 = torch.full((n, b), float("nan"), device="cuda")
        a1 = torch.full((n, b), -7777, dtype=torch.int32, device="cuda")
        loom.loom_i8_dequant_dot_noalloc(w, sw, n, k, x, sx, b, y=y1, acc=a1)
        torch.cuda.synchronize()
        assert torch.equal(a0, a1)
        assert torch.equal(y0.view(torch.int32), y1.view(torch.int32))
        if seed is not None:
            want_acc, _ = oracle.i8_dequant_dot(d["w"], d["scale_w"], d["x"], d["scale_x"], threads=8)
            assert np.array_equal(a1.cpu().numpy().astype(np.int64), want_acc)
