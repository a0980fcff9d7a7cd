"""Host logic of the benchmark (no GPU): the algorithmic byte counts, the
reference arm's leading-fraction samples, and the step's lane plans."""
import numpy as np

import bench


def tiny_inputs():
    seg_counts = np.array([0, 5, 63, 17], np.int32)
    wide_counts = np.array([3, 0, 9], np.int32)
    return {
        "segments": {"counts": seg_counts, "num_segments": 4},
        "wide": {"counts": wide_counts, "num_segments": 3},
        "gemv": {"w": np.zeros((6, 32), np.int8), "x": np.zeros((1, 32), np.int8)},
        "batched": {"w": np.zeros((6, 32), np.int8), "x": np.zeros((16, 32), np.int8)},
    }


def test_algorithmic_bytes_by_hand():
    b = bench.algorithmic_bytes(tiny_inputs())
    assert b["segments"] == 128 * (0 + 5 + 63 + 17) + 4 * 24          # active rows + count, initial, 4 outputs
    assert b["wide"] == 4 * (3 + 0 + 9) + 3 * 20                       # active elements + count, 4 outputs
    assert b["gemv"] == 6 * 32 + 4 * 6 + 1 * 32 + 4 * 1 + 4 * 6 * 1    # W, scale_w, x, scale_x, y
    assert b["batched"] == 6 * 32 + 4 * 6 + 16 * 32 + 4 * 16 + 4 * 6 * 16


def test_leading_fraction():
    assert bench.leading(65536, 1.0) == 65536 and bench.leading(65536, 2.0) == 65536
    assert bench.leading(65536, 0.5) == 32768
    assert bench.leading(10, 0.01) == 1                                 # never empty
    assert bench.leading(10, 0.25) == 3                                 # rounds up
    half = bench.algorithmic_bytes(tiny_inputs(), 0.5)
    assert half["segments"] == 128 * (0 + 5) + 2 * 24                   # the two leading segments
    assert half["wide"] == 4 * (3 + 0) + 2 * 20
    assert half["gemv"] == 3 * 32 + 4 * 3 + 32 + 4 + 4 * 3
    full = bench.algorithmic_bytes(tiny_inputs(), 1.0)
    assert full == bench.algorithmic_bytes(tiny_inputs())


def test_lane_plans_cover_every_workload_once():
    for plan in (bench.STEP_LANES, bench.ONE_LANE):
        names = [n for lane in plan for n in lane]
        assert sorted(names) == sorted(bench.ORDER)
    assert bench.ONE_LANE == (bench.ORDER,)
    assert set(bench.E2E_INPUTS) == set(bench.ORDER) == set(bench.E2E_OUTPUTS)
    # every dense input is uploaded by exactly one workload
    keys = [k for name in bench.ORDER for k in bench.E2E_INPUTS[name]]
    assert len(keys) == len(set(keys))


def test_whole_job_value():
    # N ranks each moving B bytes per step of T ms: N * B / T
    assert bench.whole_job_gbs(1, 1_000_000_000, 1.0) == 1000.0
    assert bench.whole_job_gbs(4, 1_000_000_000, 2.0) == 2000.0


def test_source_hash_ignores_comments_only():
    src = ('int a = 1; // note\n/* block\n   comment */\nconst char *s = "a // b /* c */";\n'
           "char q = '\"';\n\n  x = 2; /* y */ z = 3;\n")
    code = bench.strip_comments(src)
    assert "note" not in code and "block" not in code and "y */" not in code
    assert '"a // b /* c */"' in code and "'\"'" in code
    assert bench.strip_comments(src.replace("note", "other words")) == code
    assert bench.strip_comments(src.replace("x = 2", "x = 4")) != code
    assert all(len(bench.source_hash(w)) == 16 for w in bench.KERNEL_SOURCES)
