"""Python binding of libloom (the C ABI in include/loom.h and loom_tuning.h).

The functions keep the C names and only marshal arguments: tensors become
device pointers, the stream defaults to torch's current stream, and a status
other than LOOM_OK raises LoomError.  Every step of the computation runs in
libloom's CUDA kernels; there is no fallback, and importing this module
fails loudly when libloom.so has not been built (see build.py).

Each function accepts either torch tensors or raw integer addresses.  Output
tensors may be passed in; when omitted they are allocated with torch (on
the inputs' device) and returned.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
#: the library this instance of the binding loads (the fault tests load a second
#: instance of this module bound to libloom_test.so, by setting LIB_PATH first)
LIB_PATH = globals().get("LIB_PATH") or os.path.join(HERE, "libloom.so")

LOOM_OK = 0
LOOM_ERR_NULL = -1
LOOM_ERR_ALIGN = -2
LOOM_ERR_SHAPE = -3
LOOM_ERR_RANGE = -4
LOOM_ERR_CUDA = -5
LOOM_ERR_TIMEOUT = -6
LOOM_ERR_ARG = -7

LOOM_DEVERR_COUNT_RANGE = 0x1
LOOM_DEVERR_TIMEOUT = 0x2

LOOM_OP_I8_UNPACK = 0
LOOM_OP_FULL_TILE_SUM = 1
LOOM_OP_ROW_SUM_BATCHED = 2
LOOM_OP_I8_DEQUANT_DOT = 3
LOOM_OP_PACKED_DOT = 4
LOOM_OP_LANE_SUMS = 5
LOOM_OP_ROUTED_COMBINE = 6
LOOM_OP_STAGE_ROWS = 7

LOOM_KERNEL_UNPACK = 1
LOOM_KERNEL_ROWSUM_STAGED = 2
LOOM_KERNEL_ROWSUM_DIRECT = 3
LOOM_KERNEL_DOT_STAGED_K = 4
LOOM_KERNEL_DOT_STAGED_B = 5
LOOM_KERNEL_DOT_DIRECT = 6
LOOM_KERNEL_DOT_TENSOR = 7
LOOM_KERNEL_DOT_TENSOR_SPLIT = 8
LOOM_KERNEL_PACKED_STAGED = 9
LOOM_KERNEL_PACKED_DIRECT = 10
LOOM_KERNEL_LANESUM_STAGED = 11
LOOM_KERNEL_LANESUM_DIRECT = 12
LOOM_KERNEL_ROUTED_STAGED = 13
LOOM_KERNEL_ROUTED_DIRECT = 14
LOOM_KERNEL_STAGE_ROWS = 15
LOOM_KERNEL_DOT_TENSOR_ROWS = 16
LOOM_KERNEL_ROWSUM_SEGMENTS = 17

LOOM_MAX_DEPTH = 8
LOOM_PATH_AUTO = 0
LOOM_PATH_STAGED = 1
LOOM_PATH_DIRECT = 2
LOOM_PATH_TENSOR = 3

LOOM_FLOOR_GRID_STRIDE = 0
LOOM_FLOOR_WARP_RANGE = 1
LOOM_FLOOR_BULK_RING = 2

#: every extern "C" symbol the headers declare
EXPORTS = (
    "loom_launch_config", "loom_full_tile_sum", "loom_row_sum_batched", "loom_i8_dequant_dot",
    "loom_i8_unpack", "loom_status_string", "loom_abi_version", "loom_row_sum_batched_ex",
    "loom_i8_dequant_dot_ex", "loom_i8_dequant_dot_workspace_bytes", "loom_i8_dequant_dot_noalloc",
    "loom_packed_dot", "loom_packed_dot_ex", "loom_sum_rows", "loom_sum_rows_ex", "loom_sum_guarded_rows",
    "loom_sum_guarded_rows_ex", "loom_routed_combine", "loom_routed_combine_ex", "loom_stage_rows",
    "loom_stream_floor",
)


class LoomError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {loom_status_string(status)} (status {status})")


class loom_launch(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_uint32 * 3), ("block", ctypes.c_uint32 * 3),
                ("cluster", ctypes.c_uint32 * 3), ("subgroup_size", ctypes.c_uint32),
                ("smem_bytes", ctypes.c_uint32), ("units_per_cta", ctypes.c_uint32),
                ("kernel", ctypes.c_uint32)]

    def as_dict(self) -> dict:
        return {"grid": tuple(self.grid), "block": tuple(self.block), "cluster": tuple(self.cluster),
                "subgroup_size": self.subgroup_size, "smem_bytes": self.smem_bytes,
                "units_per_cta": self.units_per_cta, "kernel": self.kernel}


class loom_tuning(ctypes.Structure):
    _fields_ = [("depth", ctypes.c_int32), ("path", ctypes.c_int32),
                ("units_per_warp", ctypes.c_int32), ("warps_per_cta", ctypes.c_int32),
                ("chunk_bytes", ctypes.c_int32), ("wait_ns", ctypes.c_int64),
                ("tc_units_per_stage", ctypes.c_int32),
                ("tc_a_buffers", ctypes.c_int32), ("tc_pipelines", ctypes.c_int32),
                ("tc_schedule", ctypes.c_int32)]


def _bind() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libloom.so is not built ({LIB_PATH}); run "
                          "`python int8_dequant_dot_gb300/build.py` or __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    sig = {
        "loom_launch_config": [i32, P, i32, ctypes.POINTER(loom_launch)],
        "loom_full_tile_sum": [P, i32, i32, i32, f32, i32, P, P, P, P, P],
        "loom_row_sum_batched": [P, i64, i64, i32, i32, P, P, i32, P, P, P, P, P, P],
        "loom_row_sum_batched_ex": [P, i64, i64, i32, i32, P, P, i32, P, P, P, P, P,
                                    ctypes.POINTER(loom_tuning), P],
        "loom_i8_dequant_dot": [P, P, i32, i32, P, P, i32, P, P, P, i64, P],
        "loom_i8_dequant_dot_ex": [P, P, i32, i32, P, P, i32, P, P, P, i64, P,
                                   ctypes.POINTER(loom_tuning), P],
        "loom_i8_dequant_dot_workspace_bytes": [i32, i32, i32, ctypes.POINTER(i64)],
        "loom_i8_dequant_dot_noalloc": [P, P, i32, i32, P, P, i32, P, P, P],
        "loom_packed_dot": [P, P, P, i32, i32, i32, i32, P, i32, P, P, P],
        "loom_packed_dot_ex": [P, P, P, i32, i32, i32, i32, P, i32, P, P, P, ctypes.POINTER(loom_tuning), P],
        "loom_sum_rows": [P, i64, i64, i32, i32, i32, P, i32, P, P],
        "loom_sum_rows_ex": [P, i64, i64, i32, i32, i32, P, i32, P, P, ctypes.POINTER(loom_tuning), P],
        "loom_sum_guarded_rows": [P, i64, i64, i32, i32, P, i32, i32, i32, P, P],
        "loom_sum_guarded_rows_ex": [P, i64, i64, i32, i32, P, i32, i32, i32, P, P, ctypes.POINTER(loom_tuning), P],
        "loom_routed_combine": [P, P, P, i64, i32, i32, i32, P, P],
        "loom_routed_combine_ex": [P, P, P, i64, i32, i32, i32, P, P, ctypes.POINTER(loom_tuning), P],
        "loom_stage_rows": [P, P, i64, i64, i32, i32, P, i32, P],
        "loom_i8_unpack": [P, i64, P, P],
        "loom_stream_floor": [P, i64, i32, i32, i32, P, P, P],
        "loom_status_string": [i32],
        "loom_abi_version": [],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = i32
    lib.loom_status_string.restype = ctypes.c_char_p
    return lib


_lib = _bind()


def library() -> ctypes.CDLL:
    return _lib


def loom_abi_version() -> int:
    return int(_lib.loom_abi_version())


def loom_status_string(status: int) -> str:
    return _lib.loom_status_string(int(status)).decode()


def _check(status: int, where: str):
    if status != LOOM_OK:
        raise LoomError(status, where)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream, like=None):
    if stream is None:
        import torch
        dev = like.device if like is not None and hasattr(like, "device") else None
        return torch.cuda.current_stream(dev).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def loom_launch_config(op: int, workload) -> dict:
    arr = (ctypes.c_int64 * max(1, len(workload)))(*[int(v) for v in workload])
    out = loom_launch()
    _check(_lib.loom_launch_config(int(op), arr, len(workload), ctypes.byref(out)),
           "loom_launch_config")
    return out.as_dict()


def _empty(like, shape, dtype):
    import torch
    return torch.empty(shape, dtype=dtype, device=like.device)


def loom_full_tile_sum(values, count: int, initial: float, tile_size: int = 8, *,
                       rows: int | None = None, lanes: int | None = None, out=None, stream=None):
    """One segment ``values[rows][lanes]``; returns ``(final_row, tail_count, full_sum,
    tail_sum)`` as four one-element device tensors (or fills ``out``)."""
    import torch
    if rows is None or lanes is None:
        rows, lanes = values.shape
    if out is None:
        out = (_empty(values, (1,), torch.int32), _empty(values, (1,), torch.int32),
               _empty(values, (1,), torch.float32), _empty(values, (1,), torch.float32))
    fr, tc, fs, ts = out
    _check(_lib.loom_full_tile_sum(_ptr(values), int(rows), int(lanes), int(count), float(initial),
                                   int(tile_size), _ptr(fr), _ptr(tc), _ptr(fs), _ptr(ts),
                                   _stream(stream, values)), "loom_full_tile_sum")
    return out


def _row_sum_outputs(values, n):
    import torch
    return (_empty(values, (n,), torch.int32), _empty(values, (n,), torch.int32),
            _empty(values, (n,), torch.float32), _empty(values, (n,), torch.float32))


def loom_row_sum_batched(values, num_segments: int, seg_stride: int, rows: int, lanes: int,
                         counts, initial=None, tile_size: int = 8, *, out=None, error=None,
                         stream=None):
    """Batched segments; returns ``(final_row, tail_count, full_sum, tail_sum)``."""
    if out is None:
        out = _row_sum_outputs(values, num_segments)
    fr, tc, fs, ts = out
    _check(_lib.loom_row_sum_batched(_ptr(values), int(num_segments), int(seg_stride), int(rows),
                                     int(lanes), _ptr(counts), _ptr(initial), int(tile_size),
                                     _ptr(fr), _ptr(tc), _ptr(fs), _ptr(ts), _ptr(error),
                                     _stream(stream, values)), "loom_row_sum_batched")
    return out


def make_tuning(depth: int = 0, path: int = LOOM_PATH_AUTO, units_per_warp: int = 0,
                warps_per_cta: int = 0, chunk_bytes: int = 0, wait_ns: int = 0,
                tc_units_per_stage: int = 0, tc_a_buffers: int = 0, tc_pipelines: int = 0,
                tc_schedule: int = 0) -> loom_tuning:
    return loom_tuning(int(depth), int(path), int(units_per_warp), int(warps_per_cta),
                       int(chunk_bytes), int(wait_ns), int(tc_units_per_stage), int(tc_a_buffers),
                       int(tc_pipelines), int(tc_schedule))


def loom_row_sum_batched_ex(values, num_segments: int, seg_stride: int, rows: int, lanes: int,
                            counts, initial=None, tile_size: int = 8, *, tuning=None, out=None,
                            error=None, stream=None):
    if out is None:
        out = _row_sum_outputs(values, num_segments)
    fr, tc, fs, ts = out
    tp = ctypes.byref(tuning) if tuning is not None else None
    _check(_lib.loom_row_sum_batched_ex(_ptr(values), int(num_segments), int(seg_stride), int(rows),
                                        int(lanes), _ptr(counts), _ptr(initial), int(tile_size),
                                        _ptr(fr), _ptr(tc), _ptr(fs), _ptr(ts), _ptr(error), tp,
                                        _stream(stream, values)), "loom_row_sum_batched_ex")
    return out


def _dot_outputs(w, n_rows, batch, want_acc):
    import torch
    y = _empty(w, (n_rows, batch), torch.float32)
    acc = _empty(w, (n_rows, batch), torch.int32) if want_acc else None
    return y, acc


def loom_i8_dequant_dot_workspace_bytes(n_rows: int, k: int, batch: int) -> int:
    """Bytes of the split-band workspace on the current device (0: none is used)."""
    out = ctypes.c_int64(0)
    _check(_lib.loom_i8_dequant_dot_workspace_bytes(int(n_rows), int(k), int(batch),
                                                    ctypes.byref(out)),
           "loom_i8_dequant_dot_workspace_bytes")
    return int(out.value)


def dot_workspace(n_rows: int, k: int, batch: int, device=None):
    """A workspace for ``loom_i8_dequant_dot`` on ``device`` (None when the call would not
    use one).  The caller owns it; calls that may overlap need one each."""
    import torch
    nbytes = loom_i8_dequant_dot_workspace_bytes(n_rows, k, batch)
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device if device is not None else "cuda")


#: workspace="auto": one workspace per (device, stream), kept for reuse
AUTO = "auto"
_workspaces: dict = {}
_workspaces_lock = threading.Lock()
#: the largest problem the workspace query accepts: its workspace is the most any
#: call on the device uses (the size grows with the CTAs, at most one per SM)
_MAX_PROBLEM = (0x7FFFFFFF, 16, 16)


def _workspace(workspace, like, n_rows, k, batch, stream_handle):
    """(address, bytes) of the workspace argument.  "auto" keeps one workspace per
    (device, stream), allocated once at its first use with the most any call on that
    device needs, so it never grows and no call waits for the device."""
    if workspace is None:
        return None, 0
    if not (isinstance(workspace, str) and workspace == AUTO):
        if isinstance(workspace, tuple):
            return workspace
        return _ptr(workspace), workspace.numel() * workspace.element_size()
    import torch
    if loom_i8_dequant_dot_workspace_bytes(n_rows, k, batch) == 0:
        return None, 0
    dev = like.device if hasattr(like, "device") else torch.device("cuda", torch.cuda.current_device())
    key = (dev.index, stream_handle)
    with _workspaces_lock:
        ws = _workspaces.get(key)
        if ws is None:
            nbytes = loom_i8_dequant_dot_workspace_bytes(*_MAX_PROBLEM)
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
            _workspaces[key] = ws
    return ws.data_ptr(), ws.numel()


def _on_device(t):
    """The device of tensor `t` made current for the call (the library sizes the
    tensor-core grid and finds its scratch on the current device)."""
    import contextlib
    if hasattr(t, "device") and getattr(t.device, "type", None) == "cuda":
        import torch
        return torch.cuda.device(t.device)
    return contextlib.nullcontext()


def loom_i8_dequant_dot(w_packed, scale_w, n_rows: int, k: int, x_packed, scale_x, batch: int, *,
                        y=None, acc=None, want_acc: bool = False, workspace=AUTO, stream=None):
    """``y[n_rows][batch]`` (and ``acc`` when requested); returns ``(y, acc)``.
    ``workspace``: a tensor (see ``dot_workspace``), an ``(address, bytes)`` pair, None
    (no split), or "auto" (kept per device and stream)."""
    if y is None:
        y, acc2 = _dot_outputs(w_packed, n_rows, batch, want_acc and acc is None)
        acc = acc if acc is not None else acc2
    with _on_device(w_packed):
        st = _stream(stream, w_packed)
        wp, wb = _workspace(workspace, w_packed, n_rows, k, batch, st)
        _check(_lib.loom_i8_dequant_dot(_ptr(w_packed), _ptr(scale_w), int(n_rows), int(k),
                                        _ptr(x_packed), _ptr(scale_x), int(batch), _ptr(y), _ptr(acc),
                                        wp, int(wb), st), "loom_i8_dequant_dot")
    return y, acc


def loom_i8_dequant_dot_ex(w_packed, scale_w, n_rows: int, k: int, x_packed, scale_x, batch: int,
                           *, y=None, acc=None, want_acc: bool = False, workspace=AUTO, error=None,
                           tuning=None, stream=None):
    if y is None:
        y, acc2 = _dot_outputs(w_packed, n_rows, batch, want_acc and acc is None)
        acc = acc if acc is not None else acc2
    tp = ctypes.byref(tuning) if tuning is not None else None
    with _on_device(w_packed):
        st = _stream(stream, w_packed)
        wp, wb = _workspace(workspace, w_packed, n_rows, k, batch, st)
        _check(_lib.loom_i8_dequant_dot_ex(_ptr(w_packed), _ptr(scale_w), int(n_rows), int(k),
                                           _ptr(x_packed), _ptr(scale_x), int(batch), _ptr(y), _ptr(acc),
                                           wp, int(wb), _ptr(error), tp, st),
               "loom_i8_dequant_dot_ex")
    return y, acc


def loom_i8_dequant_dot_noalloc(w_packed, scale_w, n_rows: int, k: int, x_packed, scale_x,
                                batch: int, *, y=None, acc=None, want_acc: bool = False, stream=None):
    """``loom_i8_dequant_dot`` with the library's fixed device scratch (no workspace, no
    allocation in the library); calls that may overlap must be serialised."""
    if y is None:
        y, acc2 = _dot_outputs(w_packed, n_rows, batch, want_acc and acc is None)
        acc = acc if acc is not None else acc2
    with _on_device(w_packed):
        _check(_lib.loom_i8_dequant_dot_noalloc(_ptr(w_packed), _ptr(scale_w), int(n_rows), int(k),
                                                _ptr(x_packed), _ptr(scale_x), int(batch), _ptr(y),
                                                _ptr(acc), _stream(stream, w_packed)),
               "loom_i8_dequant_dot_noalloc")
    return y, acc


def loom_packed_dot(fields, scales, rhs, counts=None, count: int = 0, initial=None, *,
                    problems: int | None = None, records: int | None = None, lanes: int | None = None,
                    streams: int | None = None, out=None, stream=None):
    """The pages' packed signed-byte dot for ``problems`` instances; returns ``out``
    float32 ``[problems][lanes]``.  ``fields`` int32 ``[P][R][L]``, ``scales`` f16 (or
    their int16 bit patterns) ``[P][R][L]``, ``rhs`` float32 ``[P][R][S][4]``; ``counts``
    int32 ``[P]`` on the device, or None with ``count`` for every instance."""
    return loom_packed_dot_ex(fields, scales, rhs, counts, count, initial, problems=problems,
                              records=records, lanes=lanes, streams=streams, out=out, stream=stream,
                              _name="loom_packed_dot")


def loom_packed_dot_ex(fields, scales, rhs, counts=None, count: int = 0, initial=None, *,
                       problems: int | None = None, records: int | None = None, lanes: int | None = None,
                       streams: int | None = None, out=None, error=None, tuning=None, stream=None,
                       _name: str = "loom_packed_dot_ex"):
    import torch
    if problems is None or records is None or lanes is None:
        problems, records, lanes = fields.shape
    if streams is None:
        streams = rhs.shape[2]
    if out is None:
        out = _empty(fields, (int(problems), int(lanes)), torch.float32)
    st = _stream(stream, fields)
    args = (_ptr(fields), _ptr(scales), _ptr(rhs), int(problems), int(records), int(lanes), int(streams),
            _ptr(counts), int(count), _ptr(initial), _ptr(out))
    if _name == "loom_packed_dot":
        _check(_lib.loom_packed_dot(*args, st), _name)
    else:
        tp = ctypes.byref(tuning) if tuning is not None else None
        _check(_lib.loom_packed_dot_ex(*args, _ptr(error), tp, st), _name)
    return out


def loom_sum_rows(values, num_segments: int, seg_stride: int, rows: int, lanes: int, width: int = 1,
                  counts=None, count: int = 0, *, out=None, error=None, tuning=None, stream=None):
    """Per-lane f32 sums (the pages' sum_rows, width 1, and sum_vector_rows, width 4):
    returns ``out`` float32 ``[num_segments][lanes]``."""
    import torch
    if out is None:
        out = _empty(values, (int(num_segments), int(lanes)), torch.float32)
    st = _stream(stream, values)
    args = (_ptr(values), int(num_segments), int(seg_stride), int(rows), int(lanes), int(width), _ptr(counts),
            int(count), _ptr(out))
    if tuning is None and error is None:
        _check(_lib.loom_sum_rows(*args, st), "loom_sum_rows")
    else:
        tp = ctypes.byref(tuning) if tuning is not None else None
        _check(_lib.loom_sum_rows_ex(*args, _ptr(error), tp, st), "loom_sum_rows_ex")
    return out


def loom_sum_guarded_rows(values, num_segments: int, seg_stride: int, rows: int, lanes: int, counts=None,
                          count: int = 0, columns: int = 4, active_lanes: int = 32, *, out=None, error=None,
                          tuning=None, stream=None):
    """The pages' guarded ragged rows over segments ``[rows][lanes][4]``: returns ``out``
    float32 ``[num_segments][lanes]``."""
    import torch
    if out is None:
        out = _empty(values, (int(num_segments), int(lanes)), torch.float32)
    st = _stream(stream, values)
    args = (_ptr(values), int(num_segments), int(seg_stride), int(rows), int(lanes), _ptr(counts), int(count),
            int(columns), int(active_lanes), _ptr(out))
    if tuning is None and error is None:
        _check(_lib.loom_sum_guarded_rows(*args, st), "loom_sum_guarded_rows")
    else:
        tp = ctypes.byref(tuning) if tuning is not None else None
        _check(_lib.loom_sum_guarded_rows_ex(*args, _ptr(error), tp, st), "loom_sum_guarded_rows_ex")
    return out


def loom_routed_combine(ids, weights, payload, *, tokens: int | None = None, routes: int | None = None,
                        rows: int | None = None, width: int | None = None, out=None, error=None, tuning=None,
                        stream=None):
    """Routed row combine: ``out`` float32 ``[tokens][width]`` from ``ids`` int32 and
    ``weights`` float32 ``[tokens][routes]`` (negative id = missing route) and
    ``payload`` float32 ``[rows][width]``."""
    import torch
    if tokens is None or routes is None:
        tokens, routes = ids.shape
    if rows is None or width is None:
        rows, width = payload.shape
    if out is None:
        out = _empty(payload, (int(tokens), int(width)), torch.float32)
    st = _stream(stream, payload)
    args = (_ptr(ids), _ptr(weights), _ptr(payload), int(tokens), int(routes), int(rows), int(width), _ptr(out))
    if tuning is None and error is None:
        _check(_lib.loom_routed_combine(*args, st), "loom_routed_combine")
    else:
        tp = ctypes.byref(tuning) if tuning is not None else None
        _check(_lib.loom_routed_combine_ex(*args, _ptr(error), tp, st), "loom_routed_combine_ex")
    return out


def loom_stage_rows(h_values, d_values, num_segments: int, seg_stride: int, rows: int, lanes: int,
                    counts=None, count: int = 0, *, stream=None):
    """Copy only each segment's first ``counts[s]`` rows from ``h_values`` (pinned host
    memory, or any memory the device can read) to the same offsets of ``d_values``."""
    _check(_lib.loom_stage_rows(_ptr(h_values), _ptr(d_values), int(num_segments), int(seg_stride), int(rows),
                                int(lanes), _ptr(counts), int(count), _stream(stream, d_values)),
           "loom_stage_rows")
    return d_values


def loom_i8_unpack(packed, n_words: int, out=None, *, stream=None):
    """``out[4j+i]`` = signed byte i of word j, as f32."""
    import torch
    if out is None:
        out = _empty(packed, (4 * int(n_words),), torch.float32)
    _check(_lib.loom_i8_unpack(_ptr(packed), int(n_words), _ptr(out), _stream(stream, packed)),
           "loom_i8_unpack")
    return out


def loom_stream_floor(src, nbytes: int, schedule: int, depth: int, ctas_per_sm: int, sink, *, error=None,
                      stream=None):
    """The read-only streaming probe: one launch reading ``nbytes`` at ``src`` (a device
    tensor or address); ``sink`` is a device int64 word."""
    _check(_lib.loom_stream_floor(_ptr(src), int(nbytes), int(schedule), int(depth), int(ctas_per_sm),
                                  _ptr(sink), _ptr(error), _stream(stream, sink)), "loom_stream_floor")
