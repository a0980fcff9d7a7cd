"""Seeded synthetic inputs for the streaming-reduction workloads.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark.  It holds none of the method's arithmetic: only a counter-based
random-number generator and the value distributions drawn from it, so the
arrays it returns are plain inputs that both sides consume unchanged.

Generator.  SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; the 64-bit finaliser constants are the ones
published with Vigna's splitmix64.c).  It is used in counter form: output
number ``i`` (0-based) of seed ``s`` is ``mix64(s + (i + 1) * GAMMA)`` with
wrap-around 64-bit arithmetic, so any slice of a stream can be produced
independently and in parallel.

Streams.  A workload draws each of its arrays from its own stream: stream
``t`` of base seed ``s`` is seeded with output number ``t`` of ``s``.

Distributions (every recipe is exact integer arithmetic except the normal
draw, which goes through numpy's ``log``/``cos`` and may differ in the last
bit between machines; no stored expected value depends on a normal draw):

* ``uniform_grid_f32``: uniform on [-1, 1) restricted to the 2**-23 grid,
  ``(k - 2**23) * 2**-23`` with ``k`` the top 24 bits of a draw.  Every value
  is exact in f32 and any sum of up to 2**29 of them is exact in f64.
* ``uniform_int``: integer in [lo, hi] from the top 32 bits of a draw by
  multiply-shift (Lemire), ``lo + ((z >> 32) * (hi - lo + 1) >> 32)``.
* ``normal_f32``: Box-Muller from two draws per pair of values:
  ``u1 = ((z0 >> 11) + 1) * 2**-53`` in (0, 1], ``u2 = (z1 >> 11) * 2**-53``;
  value ``2j`` is ``sqrt(-2 ln u1) * cos(2 pi u2)`` and value ``2j+1`` the
  same with ``sin``, in f64, rounded to f32.
* ``uniform_f32``: ``lo + (hi - lo) * u`` in f64 with ``u = (z >> 11) * 2**-53``,
  rounded to f32.
* ``int8_bytes``: the little-endian bytes of successive draws, read as int8
  (uniform on [-128, 127]).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 20

#: base seed of workload ``cfg`` (1-based, in the order the workloads are listed)
SEED_BASE = 0x100D0000


def workload_seed(cfg: int) -> int:
    return SEED_BASE + int(cfg)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _draws(seed: int, start: int, n: int) -> np.ndarray:
    idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * GAMMA)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def _chunked(n: int, out_dtype, fill) -> np.ndarray:
    """Fill an array of ``n`` values chunk by chunk on a thread pool.

    ``fill(start, stop)`` returns the values for positions [start, stop);
    numpy releases the GIL inside its kernels, so chunks run in parallel.
    """
    out = np.empty(n, dtype=out_dtype)
    spans = [(a, min(n, a + _CHUNK)) for a in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for a, b in spans:
            out[a:b] = fill(a, b)
        return out

    def work(span):
        a, b = span
        out[a:b] = fill(a, b)

    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(work, spans))
    return out


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Outputs ``start .. start+n-1`` of the SplitMix64 stream of ``seed``."""
    return _chunked(n, np.uint64, lambda a, b: _draws(seed, start + a, b - a))


def stream_seed(seed: int, stream: int) -> int:
    """Seed of sub-stream ``stream`` of ``seed`` (its output number ``stream``)."""
    return int(_draws(seed, int(stream), 1)[0])


def uniform_grid_f32(seed: int, n: int) -> np.ndarray:
    two23 = np.int64(1 << 23)

    def fill(a, b):
        k = (_draws(seed, a, b - a) >> np.uint64(40)).astype(np.int64)
        return ((k - two23).astype(np.float64) * 2.0**-23).astype(np.float32)

    return _chunked(n, np.float32, fill)


def uniform_int(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    span = np.uint64(int(hi) - int(lo) + 1)
    if int(hi) < int(lo) or int(span) > (1 << 32):
        raise ValueError("uniform_int needs lo <= hi and a span of at most 2**32")

    def fill(a, b):
        z = _draws(seed, a, b - a) >> np.uint64(32)
        return ((z * span) >> np.uint64(32)).astype(np.int64) + int(lo)

    return _chunked(n, np.int64, fill)


def uniform_f32(seed: int, n: int, lo: float, hi: float) -> np.ndarray:
    def fill(a, b):
        u = (_draws(seed, a, b - a) >> np.uint64(11)).astype(np.float64) * 2.0**-53
        return (lo + (hi - lo) * u).astype(np.float32)

    return _chunked(n, np.float32, fill)


def normal_f32(seed: int, n: int) -> np.ndarray:
    pairs = (n + 1) // 2

    def fill(a, b):
        z = _draws(seed, 2 * a, 2 * (b - a))
        u1 = ((z[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * 2.0**-53
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        out = np.empty(2 * (b - a), dtype=np.float32)
        out[0::2] = r * np.cos(t)
        out[1::2] = r * np.sin(t)
        return out

    both = _chunked_pairs(pairs, fill)
    return both[:n].copy() if both.size != n else both


def _chunked_pairs(pairs: int, fill) -> np.ndarray:
    out = np.empty(2 * pairs, dtype=np.float32)
    spans = [(a, min(pairs, a + _CHUNK)) for a in range(0, pairs, _CHUNK)]

    def work(span):
        a, b = span
        out[2 * a:2 * b] = fill(a, b)

    if len(spans) <= 1:
        for sp in spans:
            work(sp)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, spans))
    return out


def int8_bytes(seed: int, n: int) -> np.ndarray:
    words = (n + 7) // 8
    z = splitmix64(seed, 0, words).astype("<u8", copy=False)
    return z.view(np.int8)[:n].copy()


# --------------------------------------------------------------------------
# Workload recipes.  Each returns a dict of numpy arrays and scalars; the
# default sizes are the full workloads, smaller sizes keep the same recipe.
# --------------------------------------------------------------------------

def full_tile_case(rows: int = 63, lanes: int = 32, count: int = 61,
                   initial: float = 0.5, tile_size: int = 8, seed: int | None = None) -> dict:
    """One ``rows x lanes`` f32 segment, uniform on the 2**-23 grid."""
    s = workload_seed(1) if seed is None else seed
    values = uniform_grid_f32(stream_seed(s, 0), rows * lanes).reshape(rows, lanes)
    return dict(values=values, rows=rows, lanes=lanes, count=int(count),
                initial=float(np.float32(initial)), tile_size=int(tile_size))


def iota_case(rows: int = 63, lanes: int = 32, count: int = 61,
              initial: float = 0.5, tile_size: int = 8) -> dict:
    """Segment filled with ``1 + lanes*row + lane`` (the pages' check input)."""
    r = np.arange(rows, dtype=np.float64)[:, None]
    l = np.arange(lanes, dtype=np.float64)[None, :]
    values = (1.0 + lanes * r + l).astype(np.float32)
    return dict(values=values, rows=rows, lanes=lanes, count=int(count),
                initial=float(np.float32(initial)), tile_size=int(tile_size))


def batched_segments(num_segments: int = 65536, rows: int = 63, lanes: int = 32,
                     tile_size: int = 8, seed: int | None = None) -> dict:
    """Independent ``rows x lanes`` segments, ragged counts in [0, rows]."""
    s = workload_seed(2) if seed is None else seed
    values = uniform_grid_f32(stream_seed(s, 0), num_segments * rows * lanes)
    counts = uniform_int(stream_seed(s, 1), num_segments, 0, rows).astype(np.int32)
    initial = normal_f32(stream_seed(s, 2), num_segments)
    return dict(values=values.reshape(num_segments, rows, lanes), counts=counts,
                initial=initial, rows=rows, lanes=lanes, tile_size=int(tile_size),
                num_segments=num_segments, seg_stride=rows * lanes)


def wide_rows(n_rows: int = 16384, n_cols: int = 16384, tile_size: int = 8,
              seed: int | None = None) -> dict:
    """f32 matrix of N(0,1) values with ragged active lengths in [0, n_cols]."""
    s = workload_seed(3) if seed is None else seed
    values = normal_f32(stream_seed(s, 0), n_rows * n_cols).reshape(n_rows, n_cols)
    lengths = uniform_int(stream_seed(s, 1), n_rows, 0, n_cols).astype(np.int32)
    return dict(values=values, counts=lengths, initial=None, rows=n_cols, lanes=1,
                tile_size=int(tile_size), num_segments=n_rows, seg_stride=n_cols)


def dequant_weights(n_rows: int = 8192, k: int = 16384, seed: int | None = None) -> dict:
    """int8 weights ``[n_rows][k]`` and per-row f32 scales in [1e-3, 1e-2]."""
    s = workload_seed(4) if seed is None else seed
    w = int8_bytes(stream_seed(s, 0), n_rows * k).reshape(n_rows, k)
    scale_w = uniform_f32(stream_seed(s, 1), n_rows, 1e-3, 1e-2)
    return dict(w=w, scale_w=scale_w, n_rows=n_rows, k=k)


def dequant_gemv(n_rows: int = 8192, k: int = 16384, seed: int | None = None) -> dict:
    """The weights above against one int8 vector with scale 0.01."""
    d = dequant_weights(n_rows, k, seed)
    s = workload_seed(4) if seed is None else seed
    d["x"] = int8_bytes(stream_seed(s, 2), k).reshape(1, k)
    d["scale_x"] = np.array([0.01], dtype=np.float32)
    d["batch"] = 1
    return d


def dequant_batched(n_rows: int = 8192, k: int = 16384, batch: int = 16,
                    seed: int | None = None) -> dict:
    """The same weights against ``batch`` int8 vectors, scales in [1e-3, 1e-2]."""
    d = dequant_weights(n_rows, k, seed)
    s = workload_seed(5) if seed is None else seed
    d["x"] = int8_bytes(stream_seed(s, 3), batch * k).reshape(batch, k)
    d["scale_x"] = uniform_f32(stream_seed(s, 4), batch, 1e-3, 1e-2)
    d["batch"] = batch
    return d


def packed_dot_case(problems: int = 128, records: int = 128, lanes: int = 2048, streams: int = 64,
                    counts=None, seed: int | None = None) -> dict:
    """Instances of the pages' packed-dot example: packed signed bytes ``[P][R][L]``
    (int32 words of uniform bytes), f16 scales ``[P][R][L]`` uniform on
    [2**-8, 2**-4) rounded to binary16 (returned as their bit patterns),
    activations ``[P][R][S][4]`` N(0,1), initial sums ``[P][L]`` N(0,1) and one
    record count per instance (all ``records`` unless given)."""
    s = workload_seed(6) if seed is None else seed
    n = problems * records * lanes
    fields = int8_bytes(stream_seed(s, 0), 4 * n).view("<i4").reshape(problems, records, lanes)
    scales = uniform_f32(stream_seed(s, 1), n, 2.0 ** -8, 2.0 ** -4).astype(np.float16)
    rhs = normal_f32(stream_seed(s, 2), problems * records * streams * 4).reshape(problems, records, streams, 4)
    initial = normal_f32(stream_seed(s, 3), problems * lanes).reshape(problems, lanes)
    if counts is None:
        counts = np.full(problems, records, np.int32)
    counts = np.ascontiguousarray(np.broadcast_to(np.asarray(counts, np.int32), (problems,)))
    return dict(fields=fields, scales=scales.view(np.uint16).reshape(problems, records, lanes), rhs=rhs,
                initial=initial, counts=counts, problems=problems, records=records, lanes=lanes,
                streams=streams)


def lane_segments(num_segments: int = 65536, rows: int = 64, lanes: int = 32, width: int = 1,
                  count_max: int | None = None, seed: int | None = None) -> dict:
    """Segments ``[S][rows][lanes]`` (width 1) or ``[S][rows][lanes][4]`` (width 4) of
    values uniform on the 2**-23 grid in [-1, 1), with counts uniform in [0, count_max]
    (``rows`` unless given)."""
    s = workload_seed(7 if width == 1 else 8) if seed is None else seed
    shape = (num_segments, rows, lanes) if width == 1 else (num_segments, rows, lanes, 4)
    values = uniform_grid_f32(stream_seed(s, 0), int(np.prod(shape))).reshape(shape)
    hi = rows if count_max is None else count_max
    counts = uniform_int(stream_seed(s, 1), num_segments, 0, hi).astype(np.int32)
    return dict(values=values, counts=counts, num_segments=num_segments, rows=rows, lanes=lanes, width=width,
                seg_stride=rows * lanes * width)


def routed_case(tokens: int = 4096, routes: int = 8, width: int = 2048, missing_every: int = 16,
                seed: int | None = None) -> dict:
    """A routed row combine: ``tokens x routes`` row ids that visit every payload row
    once (a seeded permutation of ``tokens * routes`` rows), about one route in
    ``missing_every`` marked missing (-1), weights uniform on [0, 1) and payload rows of
    ``width`` N(0,1) values."""
    s = workload_seed(9) if seed is None else seed
    rows = tokens * routes
    order = np.argsort(splitmix64(stream_seed(s, 0), 0, rows), kind="stable").astype(np.int32)
    ids = order.reshape(tokens, routes).copy()
    if missing_every:
        miss = uniform_int(stream_seed(s, 1), rows, 0, missing_every - 1).reshape(tokens, routes) == 0
        ids[miss] = -1
    weights = uniform_f32(stream_seed(s, 2), rows, 0.0, 1.0).reshape(tokens, routes)
    payload = normal_f32(stream_seed(s, 3), rows * width).reshape(rows, width)
    return dict(ids=ids, weights=weights, payload=payload, tokens=tokens, routes=routes, rows=rows, width=width)
