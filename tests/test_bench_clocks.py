"""The benchmark's clock record: nvidia-smi lines are parsed with their own
timestamps and only the samples inside the timed region are summarised."""
import datetime

import bench


def line(t, sm, reasons=()):
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    flags = ["Active" if nm in reasons else "Not Active" for nm in bench.ClockSampler.NAMES]
    return ", ".join([stamp, str(sm), "2070", "900.5", "0x0000000000000000"] + flags)


def test_only_samples_inside_the_timed_region_count():
    t0 = 1_800_000_000.0
    out = "\n".join([line(t0 - 0.2, 1000, ("hw_slowdown",)), line(t0 + 0.01, 2070), line(t0 + 0.03, 2055),
                     line(t0 + 0.05, 2070, ("sw_power_cap",)), line(t0 + 0.5, 800)])
    rows = bench.ClockSampler.parse(out)
    assert len(rows) == 5
    s = bench.ClockSampler.summarise(rows, (t0, t0 + 0.06))
    assert s["samples"] == 3 and s["in_timed_region"] is True
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"]
    assert s["timed_region_ms"] == 60.0


def test_no_sample_inside_falls_back_to_all_and_says_so():
    t0 = 1_800_000_000.0
    rows = bench.ClockSampler.parse("\n".join([line(t0 - 0.1, 2070), line(t0 + 0.1, 2070)]))
    s = bench.ClockSampler.summarise(rows, (t0, t0 + 0.004))
    assert s["samples"] == 2 and s["in_timed_region"] is False


def test_malformed_lines_are_skipped():
    rows = bench.ClockSampler.parse("[N/A], 2070\nnot a line\n" + line(1_800_000_000.0, 1995))
    assert [r[1] for r in rows] == [1995.0]
    assert bench.ClockSampler.summarise([], None) is None
