"""Helpers shared by the GPU parity tests (no test functions here)."""
import ctypes

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


_test_binding = None


def loom_test_module():
    """A second instance of the binding, bound to libloom_test.so: the library
    built with the fault-test hook (the same kernels; its host layer also exports
    loom_test_inject_stall).  The shipping libloom.so cannot stall on purpose."""
    global _test_binding
    if _test_binding is None:
        import importlib.util
        import os
        import __graft_entry__
        __graft_entry__.build()
        pkg = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "int8_dequant_dot_gb300")
        spec = importlib.util.spec_from_file_location("loom_with_test_hooks", os.path.join(pkg, "__init__.py"))
        mod = importlib.util.module_from_spec(spec)
        mod.LIB_PATH = os.path.join(pkg, "libloom_test.so")
        spec.loader.exec_module(mod)
        lib = mod.library()
        lib.loom_test_inject_stall.argtypes = [ctypes.c_int32]
        lib.loom_test_inject_stall.restype = None
        _test_binding = mod
    return _test_binding


class injected_stall:
    """Context manager: the staged kernels that the test binding launches inside it
    issue no copies, so every wait of theirs runs out after the tuning's wait limit."""

    def __init__(self, mod):
        self.lib = mod.library()

    def __enter__(self):
        self.lib.loom_test_inject_stall(1)
        return self

    def __exit__(self, *exc):
        self.lib.loom_test_inject_stall(0)
        return False


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
