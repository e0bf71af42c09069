"""Host logic of bench.py's nvidia-smi clock fallback: only samples stamped inside the
timed region count, and a region shorter than the sampling period takes the two samples
that bracket it."""
import datetime
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _line(t, mhz, reasons=("Not Active",) * 4):
    ts = datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return ", ".join([ts, str(mhz), "2032", *reasons])


def test_samples_inside_the_region_only():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.04, 1000), _line(t0 + 0.01, 1980),
             _line(t0 + 0.03, 1965, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + 0.09, 500, ("Active", "Not Active", "Not Active", "Not Active"))]
    mhz, max_mhz, reasons, note = bench.smi_window(lines, t0, t0 + 0.05)
    assert mhz == [1980, 1965]
    assert max_mhz == 2032
    assert reasons == {"sw_power_cap"}   # the hw_slowdown sample lies outside the region
    assert note is None


def test_short_region_takes_the_bracketing_samples():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.03, 1900), _line(t0 - 0.01, 1950), _line(t0 + 0.012, 1990),
             _line(t0 + 0.03, 2000)]
    mhz, _, _, note = bench.smi_window(lines, t0, t0 + 0.005)
    assert mhz == [1950, 1990]
    assert note and "bracketing" in note


def test_garbage_and_empty_output():
    assert bench.smi_window([], 0.0, 1.0)[0] == []
    mhz, _, _, note = bench.smi_window(["", "[N/A], x", "Failed to initialize NVML"], 0.0, 1.0)
    assert mhz == [] and note


def test_ctypes_nvml_fails_cleanly_without_a_driver():
    # On a host without the driver's libnvidia-ml (or without the device), the ctypes
    # fallback raises, and the sampler then uses nvidia-smi or reports no samples.
    try:
        bench.CtypesNvml("00000000:00:00.0")
    except Exception as e:  # noqa: BLE001
        assert isinstance(e, (OSError, RuntimeError, AttributeError))
