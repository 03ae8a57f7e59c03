"""bench.py's clock record keeps the nvidia-smi samples taken inside the timed region (CPU only)."""

import datetime

import bench


def _line(t: float, sm: int, reasons=("Not Active",) * 4) -> str:
    stamp = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([stamp, str(sm), "2070", "900.00", "0x0000000000000000", *reasons])


def test_only_samples_inside_the_window_count():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 1.0, 120), _line(t0 + 0.02, 2070), _line(t0 + 0.07, 2070), _line(t0 + 0.12, 2055),
             _line(t0 + 0.9, 345, ("Not Active", "Active", "Not Active", "Not Active"))]
    rec = bench.ClockSampler.summarise("\n".join(lines), (t0, t0 + 0.15))
    assert rec["samples"] == 3 and rec["window"] == "timed region"
    assert rec["sm_mhz"] == 2070 and rec["sm_max_mhz"] == 2070
    assert rec["reasons"] == []  # the slowdown after the region is not counted


def test_reasons_inside_the_window_are_reported():
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.01, 1980, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + 0.06, 2070)]
    rec = bench.ClockSampler.summarise("\n".join(lines), (t0, t0 + 0.1))
    assert rec["reasons"] == ["sw_power_cap"] and rec["samples"] == 2


def test_falls_back_to_all_samples_without_stamps_in_the_window():
    lines = ["not a time, 2070, 2070, 900.00, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage line"]
    rec = bench.ClockSampler.summarise("\n".join(lines), (0.0, 1.0))
    assert rec["samples"] == 1 and rec["window"] == "all samples" and rec["sm_mhz"] == 2070
    assert bench.ClockSampler.summarise("", None)["sm_mhz"] is None
