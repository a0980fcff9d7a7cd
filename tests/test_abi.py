"""The C ABI on a machine without a GPU: symbols, launch arithmetic, validation.

No call here reaches the device: every entry-point call is rejected by host
validation (or is empty work) before anything is launched.
"""
import ctypes
import os
import re
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def loom():
    import __graft_entry__
    __graft_entry__.build()
    import int8_dequant_dot_gb300 as m
    return m


def _declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*(?:loom_status|const char \*|int32_t)\s*(loom_\w+)\(", text,
                                    re.M))
    return names


def test_every_declared_symbol_is_exported(loom):
    declared = _declared_functions()
    assert declared == set(loom.EXPORTS)
    nm = subprocess.run(["nm", "-D", "--defined-only", loom.LIB_PATH], capture_output=True, text=True)
    exported = set(re.findall(r"\sT\s(loom_\w+)$", nm.stdout, re.M))
    assert declared <= exported
    for name in declared:
        assert getattr(loom.library(), name)


def test_fault_hook_only_in_the_test_build(loom):
    # The shipping library exports the declared entry points and nothing that can
    # stall a kernel on purpose; the test build adds exactly that one hook.
    def exported(path):
        nm = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True)
        return set(re.findall(r"\sT\s(loom_\w+)$", nm.stdout, re.M))
    ship = exported(loom.LIB_PATH)
    test = exported(os.path.join(os.path.dirname(loom.LIB_PATH), "libloom_test.so"))
    assert "loom_test_inject_stall" not in ship
    assert test == ship | {"loom_test_inject_stall"}
    assert not hasattr(loom.make_tuning(), "inject_stall")


def test_version_and_strings(loom):
    assert loom.loom_abi_version() == 4
    for st in range(-7, 1):
        assert loom.loom_status_string(st)
    assert loom.loom_status_string(-99) == "unknown status"


def test_unpack_launch_matches_page_example(loom):
    # 1009 elements in 256-wide workgroups -> 4 workgroups
    # (page "Kernels and launch configuration", "Workload is not workgroup count").
    L = loom.loom_launch_config(loom.LOOM_OP_I8_UNPACK, [1009])
    assert L["grid"] == (4, 1, 1) and L["block"] == (256, 1, 1) and L["cluster"] == (1, 1, 1)
    for n in (0, 1, 255, 256, 257, 1009, 10**9):
        L = loom.loom_launch_config(loom.LOOM_OP_I8_UNPACK, [n])
        assert L["grid"][0] == oracle.workgroups(n, 256)


@pytest.mark.parametrize("rows,lanes", [(63, 32), (16384, 1), (1, 32), (1000, 1)])
def test_row_sum_launch_is_ceiling_division(loom, rows, lanes):
    for s in (0, 1, 15, 16, 17, 1000, 65536, 65537):
        L = loom.loom_launch_config(loom.LOOM_OP_ROW_SUM_BATCHED, [s, rows, lanes])
        assert L["grid"][0] == oracle.workgroups(s, L["units_per_cta"])
        assert L["block"][0] % 32 == 0 and L["subgroup_size"] == 32
        # 32-lane segments of at most 64 rows: one bulk copy per segment, 4 per warp
        segs = lanes == 32 and rows <= 64
        assert L["kernel"] == (loom.LOOM_KERNEL_ROWSUM_SEGMENTS if segs else loom.LOOM_KERNEL_ROWSUM_STAGED)
        if segs:   # a ring of 8 KiB and four barriers: four segments in flight
            assert L["units_per_cta"] == 4 and L["smem_bytes"] == 8192 + 4 * 8
        d = loom.loom_launch_config(loom.LOOM_OP_ROW_SUM_BATCHED, [s, rows, lanes, 0])
        assert d["kernel"] == loom.LOOM_KERNEL_ROWSUM_DIRECT and d["smem_bytes"] == 0
    # one stage of 4 KiB plus one barrier per warp and depth
    for depth in range(1, 5):
        for warps in (1, 2, 4, 8):
            for chunk in (512, 4096, 8192):
                wl = [10, rows, lanes, 1, depth, warps, 0, chunk]
                if lanes == 32 and rows * 128 <= chunk:   # one ring of `chunk` bytes, `depth` barriers
                    want = warps * (chunk + (8 * depth + 15) // 16 * 16)   # rings 16-byte aligned
                else:                                     # depth stages of one chunk + one barrier each
                    want = warps * depth * (chunk + 8)
                if want > 227 * 1024:   # more than a CTA may hold
                    with pytest.raises(loom.LoomError):
                        loom.loom_launch_config(loom.LOOM_OP_ROW_SUM_BATCHED, wl)
                    continue
                L = loom.loom_launch_config(loom.LOOM_OP_ROW_SUM_BATCHED, wl)
                assert L["smem_bytes"] == want and L["block"][0] == 32 * warps
    L = loom.loom_launch_config(loom.LOOM_OP_ROW_SUM_BATCHED, [10, rows, lanes, 1, 1, 1])
    segs = lanes == 32 and rows <= 64   # an 8 KiB ring and one barrier (16-byte aligned); else chunks
    assert L["smem_bytes"] == (8192 + 16 if segs else (4096 if rows * lanes <= 4096 else 8192) + 8)


SMS = 152   # SM count given to the launch configuration (no device is needed then)


def tc_expect(n_rows, k, split=True, pipes=2):
    """The tensor-core schedule: ceil(n_rows / SMs) whole rows per CTA when the CTA's
    blocks (at most 64 rows each) hold 32 rows or more and k has 16 or more 128-byte
    units; else a cluster of c CTAs per 128-row band (c = 2..4) when that keeps every SM
    busy -- or, without a workspace, at least three quarters of them; else one CTA per SM
    over equal shares of the 128-row x 128-k units (of whole bands without a workspace).
    Returns (grid, cluster, units per CTA, kind)."""
    bands = oracle.workgroups(n_rows, 128)
    ub = oracle.workgroups(k, 128)
    rpc = oracle.workgroups(n_rows, SMS)
    blocks = oracle.workgroups(rpc, 64)
    if pipes == 2 and oracle.workgroups(rpc, blocks) >= 32 and ub >= 16:
        return oracle.workgroups(n_rows, rpc), 1, rpc, "rows"
    c = min(4, SMS // bands, ub // pipes)
    if c >= 2 and (bands * c == SMS if split else 4 * bands * c >= 3 * SMS):
        return bands * c, c, oracle.workgroups(ub, c), "bands"
    if split:
        grid = min(bands * ub, SMS)
        return grid, 1, oracle.workgroups(bands * ub, grid), "split"
    grid = min(bands, SMS)
    return grid, 1, ub * oracle.workgroups(bands, grid), "bands"


def test_dot_launch(loom):
    # one vector: 2 CTAs of 8 one-stage warps on every SM, ceil(8192 / 304) = 27 rows each;
    # shared memory: 8 rings of 8 KiB and their barriers, the activations' barrier, the
    # row totals (rounded to 16 bytes) and the 16 KiB of activations
    L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, [8192, 16384, 1, 1, 0, 0, 0, 0, 1, SMS])
    assert L["kernel"] == loom.LOOM_KERNEL_DOT_STAGED_K
    assert L["units_per_cta"] == 27 and L["grid"][0] == oracle.workgroups(8192, 27) == 304
    assert L["block"] == (256, 1, 1) and L["smem_bytes"] == 8 * (8192 + 8) + 8 + 27 * 2 * 4 + 16384
    for n, ctas, rows in ((8192, 1, 54), (8192, 2, 27), (37, 3, 1), (10**6, 3, 1024)):
        L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, [n, 4096, 2, 1, 0, 0, ctas, 0, 1, SMS])
        assert (L["units_per_cta"], L["grid"][0]) == (rows, oracle.workgroups(n, rows)), (n, ctas)
    wl = [8192, 16384, 16, 1, 0, 0, 0, 0, 1, SMS]
    # 8192 rows on 152 SMs: 54 whole rows per CTA (one launch, with or without a workspace)
    for ws in (1, 0):
        L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, wl[:8] + [ws, SMS])
        assert L["kernel"] == loom.LOOM_KERNEL_DOT_TENSOR_ROWS
        assert L["grid"] == (152, 1, 1) and L["cluster"] == (1, 1, 1) and L["units_per_cta"] == 54
        assert L["block"] == (896, 1, 1)                            # two pipelines of 14 warps
        assert 120 * 1024 <= L["smem_bytes"] <= 227 * 1024          # one CTA per SM
    # asked for: equal shares of the 128 x 128 units on every SM (streaming + finishing kernel)
    L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, wl + [0, 0, 0, 2])
    assert L["kernel"] == loom.LOOM_KERNEL_DOT_TENSOR_SPLIT
    assert L["grid"] == (152, 1, 1) and L["cluster"] == (1, 1, 1) and L["units_per_cta"] == 54
    for ws, sched in ((0, 3), (1, 3)):   # asked for: a cluster of two per band
        L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, wl[:8] + [ws, SMS, 0, 0, 0, sched])
        assert L["kernel"] == loom.LOOM_KERNEL_DOT_TENSOR and L["cluster"] == (2, 1, 1)
        assert L["grid"] == (128, 1, 1) and L["units_per_cta"] == 64
    L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, wl + [0, 0, 0, 1])   # whole bands
    assert L["grid"] == (64, 1, 1) and L["units_per_cta"] == 128
    L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, wl + [0, 0, 1])      # one pipeline
    assert L["grid"] == (152, 1, 1) and L["block"] == (704, 1, 1)   # four converter groups
    assert L["kernel"] == loom.LOOM_KERNEL_DOT_TENSOR_SPLIT
    # whole rows asked for where they fill few lanes: 16384 rows -> 108 per CTA, two blocks
    # of 54; 1000 rows -> 7 per CTA, 143 CTAs
    for n, grid, per in ((16384, 152, 108), (1000, 143, 7), (9729, 150, 65)):
        L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, [n, 4096, 16, 1, 0, 0, 0, 2, 0, SMS, 0, 0, 0, 4])
        assert L["kernel"] == loom.LOOM_KERNEL_DOT_TENSOR_ROWS
        assert (L["grid"][0], L["units_per_cta"]) == (grid, per) == (oracle.workgroups(n, per), per)
    L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, [8191, 16384, 16, 1, 2, 0, 0, 1])
    assert L["kernel"] == loom.LOOM_KERNEL_DOT_STAGED_B
    assert L["grid"][0] == oracle.workgroups(8191, L["units_per_cta"])
    for n in (1, 127, 128, 129, 2049, 8192, 20000):
        for k in (16, 1024, 1040, 16384):
            for split in (0, 1):
                L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT,
                                            [n, k, 5, 1, 0, 0, 0, 0, split, SMS])
                grid, cl, per, kind = tc_expect(n, k, split=bool(split))
                assert L["kernel"] == {"split": loom.LOOM_KERNEL_DOT_TENSOR_SPLIT, "rows": loom.LOOM_KERNEL_DOT_TENSOR_ROWS,
                                       "bands": loom.LOOM_KERNEL_DOT_TENSOR}[kind], (n, k, split)
                assert (L["grid"][0], L["cluster"][0], L["units_per_cta"]) == (grid, cl, per), (n, k, split)
    with pytest.raises(loom.LoomError):   # tensor cores forced where k allows no tile
        loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, [64, 8, 16, 1, 2, 0, 0, 2])
    # stages, units per stage, A buffers, pipelines, schedule: out of range or not fitting
    for bad in ([0, 0, 4], [0, 0, 2, 0, 2], [0, 3, 0], [0, 0, 0, 3], [3, 2, 0, 0], [0, 0, 0, 0, 5], [0, 0, 6, 1],
                [3, 0, 0, 0, 4], [0, 2, 0, 0, 4], [0, 0, 4, 0, 4], [0, 0, 0, 1, 4], [10, 0, 0, 0, 4]):
        with pytest.raises(loom.LoomError) as e:
            loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT,
                                    [8192, 16384, 16, 1, bad[0], 0, 0, 2, 1, SMS] + bad[1:])
        assert e.value.status == loom.LOOM_ERR_ARG
    with pytest.raises(loom.LoomError) as e:   # the split schedule without a workspace
        loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, wl[:8] + [0, SMS, 0, 0, 0, 2])
    assert e.value.status == loom.LOOM_ERR_ARG
    L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, [8192, 16388, 16])
    assert L["kernel"] == loom.LOOM_KERNEL_DOT_DIRECT
    L = loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, [77, 64, 0, 1, 0, 0, 0, 0, 1, SMS])
    assert L["grid"][0] == 0


def test_launch_config_errors(loom):
    with pytest.raises(loom.LoomError) as e:
        loom.loom_launch_config(99, [1])
    assert e.value.status == loom.LOOM_ERR_ARG
    with pytest.raises(loom.LoomError) as e:
        loom.loom_launch_config(loom.LOOM_OP_I8_UNPACK, [-1])
    assert e.value.status == loom.LOOM_ERR_SHAPE
    for bad in ([5, 63, 7], [5, -1, 32], [5, 1 << 27, 32]):
        with pytest.raises(loom.LoomError) as e:
            loom.loom_launch_config(loom.LOOM_OP_ROW_SUM_BATCHED, bad)
        assert e.value.status == loom.LOOM_ERR_SHAPE
    for bad in ([5, 63, 32, 1, 9], [5, 63, 32, 1, 2, 3], [5, 63, 32, 1, 2, 1, 0, 1000],
                [5, 63, 32, 1, 4, 8, 0, 32768]):   # depth, warps, chunk, shared memory
        with pytest.raises(loom.LoomError) as e:
            loom.loom_launch_config(loom.LOOM_OP_ROW_SUM_BATCHED, bad)
        assert e.value.status == loom.LOOM_ERR_ARG
    for bad in ([5, 6, 1], [5, 131072, 1], [-1, 16, 1]):
        with pytest.raises(loom.LoomError) as e:
            loom.loom_launch_config(loom.LOOM_OP_I8_DEQUANT_DOT, bad)
        assert e.value.status == loom.LOOM_ERR_SHAPE


A = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


def _status(fn, *args):
    return fn(*args)


def test_row_sum_validation(loom):
    lib = loom.library()
    call = lambda values, S, stride, rows, lanes, counts, tile, outs=(A, A, A, A): \
        lib.loom_row_sum_batched(values, S, stride, rows, lanes, counts, None, tile, *outs, None, None)
    assert call(None, 0, 0, 63, 32, None, 8) == loom.LOOM_OK           # empty work
    assert call(None, 1, 2016, 63, 32, A, 8) == loom.LOOM_ERR_NULL
    assert call(A, 1, 2016, 63, 32, None, 8) == loom.LOOM_ERR_NULL
    assert call(A, 1, 2016, 63, 32, A, 8, (A, None, A, A)) == loom.LOOM_ERR_NULL
    assert call(A + 2, 1, 2016, 63, 32, A, 8) == loom.LOOM_ERR_ALIGN
    assert call(A, 1, 2016, 63, 32, A + 1, 8) == loom.LOOM_ERR_ALIGN
    assert call(A, 1, 2016, 63, 16, A, 8) == loom.LOOM_ERR_SHAPE        # lanes
    assert call(A, 1, 2016, 63, 32, A, 0) == loom.LOOM_ERR_SHAPE        # tile
    assert call(A, 1, 2016, 63, 32, A, 65) == loom.LOOM_ERR_SHAPE
    assert call(A, 2, 2000, 63, 32, A, 8) == loom.LOOM_ERR_SHAPE        # overlapping segments
    assert call(A, -1, 2016, 63, 32, A, 8) == loom.LOOM_ERR_SHAPE
    assert call(A, 1, 2016, -1, 32, A, 8) == loom.LOOM_ERR_SHAPE
    assert call(A, 1, 1 << 26, 1 << 26, 32, A, 8) == loom.LOOM_ERR_SHAPE  # rows*lanes >= 2^31
    t = loom.make_tuning(depth=9)
    st = lib.loom_row_sum_batched_ex(A, 1, 2016, 63, 32, A, None, 8, A, A, A, A, None,
                                     loom.ctypes.byref(t), None)
    assert st == loom.LOOM_ERR_ARG
    t = loom.make_tuning(path=loom.LOOM_PATH_STAGED)
    st = lib.loom_row_sum_batched_ex(A + 4, 1, 2016, 63, 32, A, None, 8, A, A, A, A, None,
                                     loom.ctypes.byref(t), None)
    assert st == loom.LOOM_ERR_ALIGN


def test_full_tile_sum_validation(loom):
    lib = loom.library()
    f = lambda values, rows, lanes, count, tile, fr=A: lib.loom_full_tile_sum(
        values, rows, lanes, count, 0.5, tile, fr, A, A, A, None)
    assert f(A, 63, 32, 64, 8) == loom.LOOM_ERR_RANGE
    assert f(A, 63, 32, -1, 8) == loom.LOOM_ERR_RANGE
    assert f(None, 63, 32, 61, 8) == loom.LOOM_ERR_NULL
    assert f(A, 63, 32, 61, 8, None) == loom.LOOM_ERR_NULL
    assert f(A, 63, 8, 61, 8) == loom.LOOM_ERR_SHAPE
    assert f(A + 1, 63, 32, 61, 8) == loom.LOOM_ERR_ALIGN


def test_dot_validation(loom):
    lib = loom.library()
    d = lambda w, n, k, x, b, y=A, acc=None, ws=None, wsb=0: lib.loom_i8_dequant_dot(
        w, A, n, k, x, A, b, y, acc, ws, wsb, None)
    assert d(None, 0, 64, None, 4) == loom.LOOM_OK       # no rows
    assert d(None, 4, 64, None, 0) == loom.LOOM_OK       # empty batch
    assert d(None, 4, 64, A, 4) == loom.LOOM_ERR_NULL
    assert d(A, 4, 64, A, 4, None) == loom.LOOM_ERR_NULL
    assert d(A, 4, 62, A, 4) == loom.LOOM_ERR_SHAPE       # k % 4
    assert d(A, 4, 131072, A, 4) == loom.LOOM_ERR_SHAPE   # |acc| could reach 2^31
    assert d(A, -4, 64, A, 4) == loom.LOOM_ERR_SHAPE
    assert d(A + 2, 4, 64, A, 4) == loom.LOOM_ERR_ALIGN
    assert d(A, 4, 64, A, 4, A, A + 3) == loom.LOOM_ERR_ALIGN
    assert d(A, 4, 64, A, 4, ws=A + 16, wsb=1 << 20) == loom.LOOM_ERR_ALIGN   # workspace: 256 B
    assert d(A, 4, 64, A, 4, ws=A, wsb=0) == loom.LOOM_ERR_ARG
    assert d(A, 4, 64, A, 4, ws=A, wsb=-1) == loom.LOOM_ERR_ARG


def test_dot_workspace_query(loom):
    lib = loom.library()
    out = ctypes.c_int64(-1)
    q = lambda n, k, b: lib.loom_i8_dequant_dot_workspace_bytes(n, k, b, ctypes.byref(out))
    for n, k, b in ((8192, 16384, 2), (8192, 16384, 0), (0, 1024, 16), (64, 8, 16), (64, 1040 + 4, 16)):
        out.value = -1
        assert q(n, k, b) == loom.LOOM_OK and out.value == 0    # no tensor-core pass
    assert lib.loom_i8_dequant_dot_workspace_bytes(64, 64, 4, None) == loom.LOOM_ERR_NULL
    assert q(-1, 64, 4) == loom.LOOM_ERR_SHAPE and q(64, 66, 4) == loom.LOOM_ERR_SHAPE


def test_unpack_validation(loom):
    lib = loom.library()
    assert lib.loom_i8_unpack(None, 0, None, None) == loom.LOOM_OK
    assert lib.loom_i8_unpack(None, 5, A, None) == loom.LOOM_ERR_NULL
    assert lib.loom_i8_unpack(A, -1, A, None) == loom.LOOM_ERR_SHAPE
    assert lib.loom_i8_unpack(A + 2, 5, A, None) == loom.LOOM_ERR_ALIGN


def test_packed_dot_launch(loom):
    # Staged (TMA ring, 128 consumer threads of two lanes each + a producer warp) when
    # lanes % 8 == 0 and streams <= 64: CTAs over tiles of 256 lanes of one instance, as
    # many per SM as their rings fit (at most seven); else 256 lanes per CTA, grid.y =
    # instances.
    def per_sm(smem):
        return max(1, min(7, (227 * 1024) // (smem + 1024)))

    L = loom.loom_launch_config(loom.LOOM_OP_PACKED_DOT, [128, 128, 2048, 64, 1, 0, 0, SMS])
    assert L["kernel"] == loom.LOOM_KERNEL_PACKED_STAGED
    # default ring: 3 stages of 4 records x (1 KiB of words + 512 B of scales + 1 KiB of activations)
    assert L["smem_bytes"] == 128 + 3 * 4 * (1024 + 512 + 64 * 16) + 16 * 3 and per_sm(L["smem_bytes"]) == 7
    assert L["grid"] == (1024, 1, 1) and L["block"] == (160, 1, 1) and L["units_per_cta"] == 1   # 1024 tiles < 7 SMs' worth
    # rings of 12 records (92 KB) fit twice per SM, of 24 records once
    L = loom.loom_launch_config(loom.LOOM_OP_PACKED_DOT, [128, 128, 2048, 64, 1, 3, 12, SMS])
    assert L["grid"] == (2 * SMS, 1, 1) and L["units_per_cta"] == 4
    L = loom.loom_launch_config(loom.LOOM_OP_PACKED_DOT, [128, 128, 2048, 64, 1, 3, 24, SMS])
    assert L["grid"] == (SMS, 1, 1) and L["units_per_cta"] == 7
    for P, R, Ln, S in ((1, 128, 2048, 64), (3, 5, 1000, 7), (2, 0, 8, 1), (65535, 1, 1, 1)):
        for aligned in (0, 1):
            L = loom.loom_launch_config(loom.LOOM_OP_PACKED_DOT, [P, R, Ln, S, aligned, 0, 0, SMS])
            staged = aligned == 1 and Ln % 8 == 0 and S <= 64
            assert L["kernel"] == (loom.LOOM_KERNEL_PACKED_STAGED if staged else loom.LOOM_KERNEL_PACKED_DIRECT)
            tiles = P * oracle.workgroups(Ln, 256)
            want = (min(tiles, per_sm(L["smem_bytes"]) * SMS), 1, 1) if staged else (oracle.workgroups(Ln, 256), P, 1)
            assert L["grid"] == want
            assert L["block"][0] == (160 if staged else 256)
    L = loom.loom_launch_config(loom.LOOM_OP_PACKED_DOT, [1, 128, 2048, 128])   # too many streams to stage
    assert L["kernel"] == loom.LOOM_KERNEL_PACKED_DIRECT and L["smem_bytes"] == 0
    for bad in ([-1, 1, 8, 1], [1, -1, 8, 1], [1, 1, -8, 1], [1, 1, 8, 0], [65536, 1, 8, 1]):
        with pytest.raises(loom.LoomError) as e:
            loom.loom_launch_config(loom.LOOM_OP_PACKED_DOT, bad)
        assert e.value.status == loom.LOOM_ERR_SHAPE
    for bad in ([1, 8, 8, 1, 1, 9], [1, 8, 8, 1, 1, 0, 33], [1, 8, 8, 64, 1, 8, 32]):   # depth, rps, smem
        with pytest.raises(loom.LoomError) as e:
            loom.loom_launch_config(loom.LOOM_OP_PACKED_DOT, bad)
        assert e.value.status == loom.LOOM_ERR_ARG


def test_packed_dot_validation(loom):
    lib = loom.library()
    f = lambda *a: lib.loom_packed_dot(*a)
    # empty work needs no pointers
    assert f(None, None, None, 0, 128, 2048, 64, None, 0, None, None, None) == loom.LOOM_OK
    assert f(None, None, None, 4, 128, 0, 64, None, 0, None, None, None) == loom.LOOM_OK
    assert f(None, None, None, 4, 8, 16, 4, None, 3, None, None, None) == loom.LOOM_ERR_NULL
    assert f(A, A, A, 4, 8, 16, 4, None, 3, None, None, None) == loom.LOOM_ERR_NULL     # no output
    assert f(A, A + 1, A, 4, 8, 16, 4, None, 3, None, A, None) == loom.LOOM_ERR_ALIGN   # scales 2-byte
    assert f(A + 2, A, A, 4, 8, 16, 4, None, 3, None, A, None) == loom.LOOM_ERR_ALIGN
    assert f(A, A, A, 4, 8, 16, 4, None, 9, None, A, None) == loom.LOOM_ERR_RANGE      # count > records
    assert f(A, A, A, 4, 8, 16, 4, None, -1, None, A, None) == loom.LOOM_ERR_RANGE
    assert f(A, A, A, 4, 8, 16, 0, None, 3, None, A, None) == loom.LOOM_ERR_SHAPE      # no streams
    assert f(A, A, A, -4, 8, 16, 4, None, 3, None, A, None) == loom.LOOM_ERR_SHAPE
    t = loom.make_tuning(path=loom.LOOM_PATH_TENSOR)
    assert lib.loom_packed_dot_ex(A, A, A, 4, 8, 16, 4, None, 3, None, A, None, ctypes.byref(t),
                                  None) == loom.LOOM_ERR_ARG
    t = loom.make_tuning(path=loom.LOOM_PATH_STAGED)   # 12 lanes cannot be staged
    assert lib.loom_packed_dot_ex(A, A, A, 4, 8, 12, 4, None, 3, None, A, None, ctypes.byref(t),
                                  None) == loom.LOOM_ERR_SHAPE


def test_lane_sum_launch(loom):
    # one warp per segment; 64 x 32 rows of width 1: four segments per warp (32 KiB of rows)
    L = loom.loom_launch_config(loom.LOOM_OP_LANE_SUMS, [65536, 64, 32, 1])
    assert L["kernel"] == loom.LOOM_KERNEL_LANESUM_STAGED
    assert L["block"] == (32, 1, 1) and L["units_per_cta"] == 4 and L["grid"] == (16384, 1, 1)
    assert L["smem_bytes"] == 2 * (4096 + 8)
    L = loom.loom_launch_config(loom.LOOM_OP_LANE_SUMS, [16384, 64, 32, 4])
    assert L["units_per_cta"] == 1 and L["grid"] == (16384, 1, 1)
    for S, R, Ln, W in ((0, 64, 32, 1), (1, 1, 1, 1), (1009, 63, 32, 4), (77, 5, 7, 1), (3, 2, 12, 1)):
        for aligned in (0, 1):
            L = loom.loom_launch_config(loom.LOOM_OP_LANE_SUMS, [S, R, Ln, W, aligned])
            staged = aligned == 1 and (Ln * W) % 4 == 0
            assert L["kernel"] == (loom.LOOM_KERNEL_LANESUM_STAGED if staged else loom.LOOM_KERNEL_LANESUM_DIRECT)
            assert L["grid"][0] == oracle.workgroups(S, L["units_per_cta"])
    for bad in ([1, 64, 33, 1], [1, 64, 0, 1], [1, 64, 32, 2], [-1, 64, 32, 1]):
        with pytest.raises(loom.LoomError) as e:
            loom.loom_launch_config(loom.LOOM_OP_LANE_SUMS, bad)
        assert e.value.status == loom.LOOM_ERR_SHAPE


def test_lane_sum_validation(loom):
    lib = loom.library()
    assert lib.loom_sum_rows(None, 0, 0, 64, 32, 1, None, 0, None, None) == loom.LOOM_OK
    assert lib.loom_sum_rows(None, 4, 2048, 64, 32, 1, None, 3, None, None) == loom.LOOM_ERR_NULL
    assert lib.loom_sum_rows(A + 2, 4, 2048, 64, 32, 1, None, 3, A, None) == loom.LOOM_ERR_ALIGN
    assert lib.loom_sum_rows(A, 4, 2048, 64, 32, 1, None, 65, A, None) == loom.LOOM_ERR_RANGE
    assert lib.loom_sum_rows(A, 4, 100, 64, 32, 1, None, 3, A, None) == loom.LOOM_ERR_SHAPE   # overlapping
    assert lib.loom_sum_rows(A, 4, 2048, 64, 32, 3, None, 3, A, None) == loom.LOOM_ERR_SHAPE   # width
    g = lib.loom_sum_guarded_rows
    assert g(A, 4, 8064, 63, 32, None, 3, 5, 32, A, None) == loom.LOOM_ERR_SHAPE   # columns > 4
    assert g(A, 4, 8064, 63, 32, None, 3, 4, 33, A, None) == loom.LOOM_ERR_SHAPE   # active > lanes
    assert g(A, 4, 8064, 63, 32, None, 64, 4, 32, A, None) == loom.LOOM_ERR_RANGE


def test_routed_combine_launch_and_validation(loom):
    L = loom.loom_launch_config(loom.LOOM_OP_ROUTED_COMBINE, [4096, 8, 32768, 2048])
    assert L["kernel"] == loom.LOOM_KERNEL_ROUTED_STAGED and L["block"] == (64, 1, 1)
    assert L["grid"] == (2048, 1, 1) and L["smem_bytes"] == 2 * 2 * (2048 + 8)
    for T, R, W, aligned, staged in ((1, 8, 2048, 1, True), (7, 33, 64, 1, False), (7, 8, 62, 1, False),
                                     (7, 8, 64, 0, False), (0, 8, 64, 1, True)):
        L = loom.loom_launch_config(loom.LOOM_OP_ROUTED_COMBINE, [T, R, 100, W, aligned])
        assert L["kernel"] == (loom.LOOM_KERNEL_ROUTED_STAGED if staged else loom.LOOM_KERNEL_ROUTED_DIRECT)
        assert L["grid"][0] == oracle.workgroups(T, 2)
    lib = loom.library()
    f = lib.loom_routed_combine
    assert f(None, None, None, 0, 8, 100, 64, None, None) == loom.LOOM_OK
    assert f(A, A, A, 4, 8, 100, 64, None, None) == loom.LOOM_ERR_NULL
    assert f(A + 2, A, A, 4, 8, 100, 64, A, None) == loom.LOOM_ERR_ALIGN
    assert f(A, A, A, -4, 8, 100, 64, A, None) == loom.LOOM_ERR_SHAPE
    t = loom.make_tuning(path=loom.LOOM_PATH_STAGED)
    assert lib.loom_routed_combine_ex(A, A, A, 4, 40, 100, 64, A, None, ctypes.byref(t), None) == loom.LOOM_ERR_SHAPE


def test_stage_rows_launch_and_validation(loom):
    L = loom.loom_launch_config(loom.LOOM_OP_STAGE_ROWS, [65536, 63, 32])
    assert L["kernel"] == loom.LOOM_KERNEL_STAGE_ROWS and L["grid"] == (65536, 1, 1) and L["block"] == (256, 1, 1)
    L = loom.loom_launch_config(loom.LOOM_OP_STAGE_ROWS, [16384, 16384, 1])
    assert L["grid"] == (16384 * 8, 1, 1)   # 8 KiB per CTA
    lib = loom.library()
    f = lib.loom_stage_rows
    assert f(None, None, 0, 0, 63, 32, None, 0, None) == loom.LOOM_OK
    assert f(None, A, 4, 2016, 63, 32, None, 3, None) == loom.LOOM_ERR_NULL
    assert f(A + 2, A, 4, 2016, 63, 32, None, 3, None) == loom.LOOM_ERR_ALIGN
    assert f(A, A, 4, 2016, 63, 32, None, 64, None) == loom.LOOM_ERR_RANGE
    assert f(A, A, 4, 100, 63, 32, None, 3, None) == loom.LOOM_ERR_SHAPE
    assert f(A, A, 4, 2016, 63, 0, None, 3, None) == loom.LOOM_ERR_SHAPE


def test_stream_floor_validation(loom):
    # the read-only probe: every rejection happens on the host, before any device access
    lib = loom.library()
    A = 1 << 20
    f = lambda src, n, kind, depth, cps, sink=A + 8: lib.loom_stream_floor(src, n, kind, depth, cps, sink, None, None)
    assert f(A, 0, 0, 4, 4) == loom.LOOM_OK                       # nothing to read: no launch
    assert f(A, -16, 0, 4, 4) == loom.LOOM_ERR_SHAPE
    assert f(A, 24, 0, 4, 4) == loom.LOOM_ERR_SHAPE                # not whole 16-byte words
    assert f(A, 64, 3, 4, 4) == loom.LOOM_ERR_ARG                  # unknown schedule
    assert f(A, 64, 0, 6, 4) == loom.LOOM_ERR_ARG                  # loads: 4 or 8 in flight
    assert f(A, 64, 2, 9, 4) == loom.LOOM_ERR_ARG                  # bulk ring: 1..8 stages
    assert f(A, 64, 1, 8, 0) == loom.LOOM_ERR_ARG
    assert f(A, 64, 1, 8, 33) == loom.LOOM_ERR_ARG
    assert f(None, 64, 0, 4, 4) == loom.LOOM_ERR_NULL
    assert f(A, 64, 0, 4, 4, None) == loom.LOOM_ERR_NULL
    assert f(A + 4, 64, 0, 4, 4) == loom.LOOM_ERR_ALIGN
    assert f(A, 64, 0, 4, 4, A + 4) == loom.LOOM_ERR_ALIGN
