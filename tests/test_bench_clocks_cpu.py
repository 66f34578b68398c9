"""bench.py's reading of the nvidia-smi clock samples taken during the timed region."""
import os
import sys
import tempfile

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


class _Done:
    def terminate(self):
        pass

    def wait(self):
        return 0


def _sampler_with(lines):
    fd, path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(lines) + "\n")
    c = bench.ClockSampler(0)
    c.path, c.proc = path, _Done()
    return c


def test_median_clock_and_active_reasons():
    c = _sampler_with([
        "0, 2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, [N/A], 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",  # unreadable: skipped
        "0, 2070, 2070, 1001.0, 0x0, Not Active, Active, Not Active, Not Active",
        "garbage",
    ])
    got = c.stop()
    assert got["samples"] == 3
    assert got["sm_mhz"] == 2070.0 and got["sm_max_mhz"] == 2070.0
    assert got["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert not os.path.exists(c.path)


def test_no_samples_and_no_tool():
    c = _sampler_with([])
    got = c.stop()
    assert got["samples"] == 0 and got["sm_mhz"] is None and got["reasons"] == []
    c = bench.ClockSampler(0)  # nvidia-smi could not start
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]
