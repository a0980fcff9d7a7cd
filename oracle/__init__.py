"""Python access to the plain CPU oracle in ``oracle.c``.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product path
(the CUDA library and its binding) never imports it, and this package imports
nothing from the product.

The functions take numpy arrays and call the C oracle through ctypes (which
releases the GIL), optionally splitting independent segments or output rows
across threads.  Splitting never changes any unit's arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = ctypes.c_int64
_ptr = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (plain gcc -O2)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB lets the planted-mistake test load a mutated build of oracle.c.
        lib = ctypes.CDLL(os.environ.get("ORACLE_LIB") or build())
        lib.oracle_full_tile_split.argtypes = [_i64, _i64, _ptr, _ptr]
        lib.oracle_full_tile_sum.argtypes = [_ptr, _i64, _i64, _i64, ctypes.c_double, _i64,
                                             _ptr, _ptr, _ptr, _ptr]
        lib.oracle_row_sum_batched.argtypes = [_ptr, _i64, _i64, _i64, _ptr, _ptr, _i64, _i64, _i64,
                                               _ptr, _ptr, _ptr, _ptr]
        lib.oracle_sum_rows.argtypes = [_ptr, _i64, _i64, _i64, _ptr]
        lib.oracle_unpack_word.argtypes = [ctypes.c_uint32, _ptr]
        lib.oracle_unpack_word.restype = None
        lib.oracle_i8_dequant_dot.argtypes = [_ptr, _ptr, _i64, _i64, _ptr, _ptr, _i64, _i64, _i64,
                                              _ptr, _ptr]
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f32.restype = ctypes.c_float
        lib.oracle_packed_dot.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _i64, _i64, _ptr, _ptr, _i64,
                                          _i64, _ptr]
        lib.oracle_lane_sums_f32.argtypes = [_ptr, _i64, _i64, _i64, _i64, _ptr, _i64, _i64, _ptr]
        lib.oracle_guarded_rows_f32.argtypes = [_ptr, _i64, _i64, _i64, _ptr, _i64, _i64, _i64, _i64, _ptr]
        lib.oracle_routed_combine.argtypes = [_ptr, _ptr, _ptr, _i64, _i64, _i64, _i64, _i64, _i64, _ptr]
        lib.oracle_workgroups.argtypes = [_i64, _i64]
        lib.oracle_workgroups.restype = _i64
        _lib = lib
    return _lib


def _p(a: np.ndarray | None):
    if a is None:
        return None
    if not a.flags.c_contiguous:
        raise ValueError("oracle inputs must be C-contiguous")
    return a.ctypes.data


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def _spans(n: int, threads: int):
    threads = max(1, min(threads, n)) if n else 1
    step = -(-n // threads) if n else 0
    return [(a, min(n, a + step)) for a in range(0, n, step)] if n else []


def _run_spans(fn, n: int, threads: int):
    spans = _spans(n, threads)
    if len(spans) <= 1:
        for a, b in spans:
            fn(a, b)
        return
    with ThreadPoolExecutor(len(spans)) as ex:
        list(ex.map(lambda sp: fn(*sp), spans))


def full_tile_split(count: int, tile_size: int) -> tuple[int, int]:
    fr, tc = _i64(), _i64()
    _check(_load().oracle_full_tile_split(count, tile_size, ctypes.byref(fr), ctypes.byref(tc)),
           "full_tile_split")
    return fr.value, tc.value


def full_tile_sum(values: np.ndarray, count: int, initial: float, tile_size: int):
    """``(final_row, tail_count, full_sum, tail_sum)`` of one segment ``values[rows][lanes]``."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    rows, lanes = v.shape
    fr, tc = _i64(), _i64()
    fs, ts = ctypes.c_double(), ctypes.c_double()
    _check(_load().oracle_full_tile_sum(_p(v), rows, lanes, count, float(initial), tile_size,
                                        ctypes.byref(fr), ctypes.byref(tc),
                                        ctypes.byref(fs), ctypes.byref(ts)), "full_tile_sum")
    return fr.value, tc.value, fs.value, ts.value


def row_sum_batched(values: np.ndarray, seg_stride: int, rows: int, lanes: int,
                    counts: np.ndarray, initial: np.ndarray | None, tile_size: int,
                    segments: np.ndarray | None = None, threads: int = 1) -> dict:
    """Every segment (or only the listed ``segments``) of a batch.

    Returns int64 ``final_row``/``tail_count`` and float64 ``full_sum``/``tail_sum``
    arrays indexed like ``segments`` (all segments when it is None).
    """
    v = values.reshape(-1)
    if v.dtype != np.float32 or not v.flags.c_contiguous:
        raise ValueError("values must be contiguous float32")
    c = np.ascontiguousarray(counts, dtype=np.int32)
    init = None if initial is None else np.ascontiguousarray(initial, dtype=np.float32)
    lib = _load()
    if segments is None:
        n = c.shape[0]
        out = {k: np.zeros(n, dt) for k, dt in (("final_row", np.int64), ("tail_count", np.int64),
                                                ("full_sum", np.float64), ("tail_sum", np.float64))}

        def run(a, b):
            _check(lib.oracle_row_sum_batched(_p(v), seg_stride, rows, lanes, _p(c), _p(init),
                                              tile_size, a, b, _p(out["final_row"]),
                                              _p(out["tail_count"]), _p(out["full_sum"]),
                                              _p(out["tail_sum"])), "row_sum_batched")

        _run_spans(run, n, threads)
        return out
    seg = np.asarray(segments, dtype=np.int64)
    res = {"final_row": np.zeros(seg.size, np.int64), "tail_count": np.zeros(seg.size, np.int64),
           "full_sum": np.zeros(seg.size, np.float64), "tail_sum": np.zeros(seg.size, np.float64)}

    def run_sel(a, b):
        for i in range(a, b):
            s = int(seg[i])
            base = v[s * seg_stride: s * seg_stride + rows * lanes].reshape(rows, lanes)
            r = full_tile_sum(base, int(c[s]), 0.0 if init is None else float(init[s]), tile_size)
            res["final_row"][i], res["tail_count"][i], res["full_sum"][i], res["tail_sum"][i] = r

    _run_spans(run_sel, seg.size, threads)
    return res


def sum_rows(values: np.ndarray, count: int) -> np.ndarray:
    v = np.ascontiguousarray(values, dtype=np.float32)
    rows, lanes = v.shape
    out = np.zeros(lanes, np.float64)
    _check(_load().oracle_sum_rows(_p(v), rows, lanes, count, _p(out)), "sum_rows")
    return out


def unpack_word(word: int) -> list[int]:
    out = np.zeros(4, np.int32)
    _load().oracle_unpack_word(ctypes.c_uint32(word & 0xFFFFFFFF), _p(out))
    return [int(t) for t in out]


def i8_dequant_dot(w: np.ndarray, scale_w: np.ndarray, x: np.ndarray, scale_x: np.ndarray,
                   rows: np.ndarray | None = None, threads: int = 1):
    """``(acc int64[N][B], y float64[N][B])``; with ``rows`` only those output rows
    are computed and the results are ``[len(rows)][B]``."""
    w = np.ascontiguousarray(w, dtype=np.int8)
    x = np.ascontiguousarray(x, dtype=np.int8)
    sw = np.ascontiguousarray(scale_w, dtype=np.float32)
    sx = np.ascontiguousarray(scale_x, dtype=np.float32)
    n_rows, k = w.shape
    batch = x.shape[0]
    if x.shape[1] != k:
        raise ValueError("w and x disagree on k")
    lib = _load()
    if rows is None:
        acc = np.zeros((n_rows, batch), np.int64)
        y = np.zeros((n_rows, batch), np.float64)

        def run(a, b):
            _check(lib.oracle_i8_dequant_dot(_p(w), _p(sw), n_rows, k, _p(x), _p(sx), batch, a, b,
                                             _p(acc), _p(y)), "i8_dequant_dot")

        _run_spans(run, n_rows, threads)
        return acc, y
    sel = np.asarray(rows, dtype=np.int64)
    acc = np.zeros((sel.size, batch), np.int64)
    y = np.zeros((sel.size, batch), np.float64)

    def run_sel(a, b):
        for i in range(a, b):
            r = int(sel[i])
            wr = np.ascontiguousarray(w[r:r + 1])
            swr = np.ascontiguousarray(sw[r:r + 1])
            _check(lib.oracle_i8_dequant_dot(_p(wr), _p(swr), 1, k, _p(x), _p(sx), batch, 0, 1,
                                             _p(acc[i]), _p(y[i])), "i8_dequant_dot")

    _run_spans(run_sel, sel.size, threads)
    return acc, y


def workgroups(element_count: int, workgroup_size: int) -> int:
    return int(_load().oracle_workgroups(element_count, workgroup_size))


def f16_to_f32(bits: int) -> float:
    """Value of an IEEE binary16 bit pattern."""
    return float(_load().oracle_f16_to_f32(ctypes.c_uint16(bits & 0xFFFF)))


def packed_dot(fields: np.ndarray, scales: np.ndarray, rhs: np.ndarray, counts,
               initial: np.ndarray | None = None, threads: int = 1) -> np.ndarray:
    """The pages' packed signed-byte dot for every instance: ``out float32[P][lanes]``.

    fields uint32/int32 [P][records][lanes]; scales f16 bit patterns (uint16) or
    float16 [P][records][lanes]; rhs float32 [P][records][streams][4]; counts int [P];
    initial float32 [P][lanes] or None.
    """
    f = np.ascontiguousarray(fields).view(np.uint32)
    sc = np.ascontiguousarray(scales).view(np.uint16)
    a = np.ascontiguousarray(rhs, dtype=np.float32)
    P, R, L = f.shape
    S = a.shape[2]
    if sc.shape != f.shape or a.shape != (P, R, S, 4):
        raise ValueError("packed_dot: shapes disagree")
    c = np.ascontiguousarray(np.broadcast_to(np.asarray(counts, dtype=np.int32), (P,)))
    init = None if initial is None else np.ascontiguousarray(initial, dtype=np.float32).reshape(P, L)
    out = np.zeros((P, L), np.float32)
    lib = _load()

    def run(p0, p1):
        _check(lib.oracle_packed_dot(_p(f), _p(sc), _p(a), P, R, L, S, _p(c), _p(init), p0, p1,
                                     _p(out)), "packed_dot")

    _run_spans(run, P, threads)
    return out


def lane_sums(values: np.ndarray, counts, width: int = 1, threads: int = 1) -> np.ndarray:
    """Per-lane f32 sums of segments ``values[S][rows][lanes]`` (width 1) or
    ``values[S][rows][lanes][4]`` (width 4) over each segment's first ``counts[s]``
    rows: ``float32[S][lanes]``."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    S, rows, lanes = v.shape[:3]
    if (width == 1 and v.ndim != 3) or (width == 4 and (v.ndim != 4 or v.shape[3] != 4)):
        raise ValueError("lane_sums: values do not match the width")
    c = np.ascontiguousarray(np.broadcast_to(np.asarray(counts, np.int32), (S,)))
    out = np.zeros((S, lanes), np.float32)
    lib = _load()

    def run(a, b):
        _check(lib.oracle_lane_sums_f32(_p(v), rows * lanes * width, rows, lanes, width, _p(c), a, b, _p(out)),
               "lane_sums")

    _run_spans(run, S, threads)
    return out


def guarded_rows(values: np.ndarray, counts, columns: int, active_lanes: int, threads: int = 1) -> np.ndarray:
    """The pages' guarded ragged rows over segments ``values[S][rows][lanes][4]``:
    ``float32[S][lanes]``."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    S, rows, lanes = v.shape[:3]
    if v.ndim != 4 or v.shape[3] != 4:
        raise ValueError("guarded_rows: values must be [S][rows][lanes][4]")
    c = np.ascontiguousarray(np.broadcast_to(np.asarray(counts, np.int32), (S,)))
    out = np.zeros((S, lanes), np.float32)
    lib = _load()

    def run(a, b):
        _check(lib.oracle_guarded_rows_f32(_p(v), rows * lanes * 4, rows, lanes, _p(c), columns, active_lanes,
                                           a, b, _p(out)), "guarded_rows")

    _run_spans(run, S, threads)
    return out


def routed_combine(ids: np.ndarray, weights: np.ndarray, payload: np.ndarray, threads: int = 1) -> np.ndarray:
    """Routed row combine: ``out float32[tokens][width]``; ``ids`` int32 ``[tokens][routes]``
    (negative = missing), ``weights`` float32 ``[tokens][routes]``, ``payload`` float32
    ``[rows][width]``."""
    i = np.ascontiguousarray(ids, dtype=np.int32)
    w = np.ascontiguousarray(weights, dtype=np.float32)
    pl = np.ascontiguousarray(payload, dtype=np.float32)
    T, R = i.shape
    rows, width = pl.shape
    out = np.zeros((T, width), np.float32)
    lib = _load()

    def run(a, b):
        _check(lib.oracle_routed_combine(_p(i), _p(w), _p(pl), T, R, rows, width, a, b, _p(out)),
               "routed_combine")

    _run_spans(run, T, threads)
    return out
