"""Helpers shared by the GPU parity tests (no test functions here)."""
import numpy as np
import pytest

#: relative tolerance for f32 results against the fp64 oracle
REL_TOL = 1e-5


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def loom_module():
    import __graft_entry__
    __graft_entry__.build()
    import int8_dequant_dot_gb300 as loom
    return loom


def to_dev(a: np.ndarray, torch):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def guarded(torch, n, dtype, guard=64, fill=None):
    """A device buffer with `guard` canary elements on each side; returns (buffer, view)."""
    buf = torch.empty(n + 2 * guard, dtype=dtype, device="cuda")
    if fill is None:
        fill = -7777 if not dtype.is_floating_point else float("nan")
    buf.fill_(fill)
    return buf, buf[guard:guard + n]


def check_guard(buf, n, guard=64):
    import torch
    head = buf[:guard]
    tail = buf[guard + n:]
    if buf.dtype.is_floating_point:
        ok = bool(torch.isnan(head).all()) and bool(torch.isnan(tail).all())
    else:
        ok = bool((head == -7777).all()) and bool((tail == -7777).all())
    assert ok, "a kernel wrote outside its output range"


def assert_rel(got: np.ndarray, want: np.ndarray, rel=REL_TOL, what="", atol=0.0):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    bad = ~(err <= rel * np.abs(want) + atol)
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside rel {rel}; first at "
                             f"{i}: got {got.flat[i]!r} want {want.flat[i]!r}")
