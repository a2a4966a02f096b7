"""bench.py's clock record (no GPU): the median SM clock and the throttle reasons
seen inside the timed window, from nvidia-smi's CSV lines."""

import tempfile
from datetime import datetime

import bench


def line(t, uuid, mhz, active=(), power=900.0):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    ts = datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    flags = ["Active" if n in active else "Not Active" for n in names]
    return ", ".join([ts, uuid, str(mhz), "2070", str(power), "0x0"] + flags)


def sampler_with(lines, uuid="GPU-a"):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.uuid = uuid
    s.proc = None
    s.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
    s.file.write("\n".join(lines) + "\n")
    s.file.flush()
    return s


def test_median_clock_and_reasons_inside_the_window():
    t0 = 1_800_000_000.0
    lines = [line(t0 - 5, "GPU-a", 1000, ("hw_slowdown",)),           # before the window: ignored
             line(t0 + 0.1, "GPU-a", 2070),
             line(t0 + 0.2, "GPU-a", 2060, ("sw_power_cap",)),
             line(t0 + 0.3, "GPU-a", 2070),
             line(t0 + 0.3, "GPU-b", 500, ("hw_thermal_slowdown",)),  # another GPU: ignored
             "garbage line",
             line(t0 + 9, "GPU-a", 900, ("sw_thermal_slowdown",))]   # after the window: ignored
    out = sampler_with(lines).summary(t0, t0 + 1.0)
    assert out["samples"] == 3
    assert out["sm_mhz"] == 2070
    assert out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"]


def test_no_samples_gives_nulls():
    out = sampler_with([]).summary(0.0, 1.0)
    assert out == {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}


def test_without_a_uuid_every_gpu_counts():
    t0 = 1_800_000_000.0
    lines = [line(t0 + 0.1, "GPU-a", 2070), line(t0 + 0.2, "GPU-b", 1500, ("hw_slowdown",))]
    out = sampler_with(lines, uuid=None).summary(t0, t0 + 1.0)
    assert out["samples"] == 2 and out["reasons"] == ["hw_slowdown"]
