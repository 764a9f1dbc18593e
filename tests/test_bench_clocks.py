"""The bench's clock sampler, against a fake nvidia-smi (no GPU needed)."""
import io
import time

import bench


class FakeSmi:
    """Emits one CSV sample every `dt` seconds, like `nvidia-smi -lms`."""

    def __init__(self, lines, dt):
        self._lines, self._dt = lines, dt
        self.stdout = self

    def __iter__(self):
        for line in self._lines:
            time.sleep(self._dt)
            yield line

    def terminate(self):
        pass

    def kill(self):
        pass

    def communicate(self, timeout=None):
        return "", ""


def _line(sm, reasons=("Not Active",) * 4):
    return "0, %d, 2070, 900.0, 0x0, %s\n" % (sm, ", ".join(reasons))


def test_samples_inside_a_long_region(monkeypatch):
    lines = [_line(2070)] * 40
    monkeypatch.setattr(bench.subprocess, "Popen", lambda *a, **k: FakeSmi(lines, 0.01))
    c = bench.Clocks(0)
    c.start()
    c.begin()
    time.sleep(0.1)
    c.end()
    r = c.stop()
    assert r["sm_mhz"] == 2070 and r["sm_max_mhz"] == 2070 and r["reasons"] == []
    assert r["samples"] >= 3 and r["sampled"].startswith("inside")


def test_short_region_is_bracketed_and_reasons_kept(monkeypatch):
    thermal = ("Not Active", "Active", "Not Active", "Not Active")
    lines = [_line(1800, thermal)] * 20
    monkeypatch.setattr(bench.subprocess, "Popen", lambda *a, **k: FakeSmi(lines, 0.05))
    c = bench.Clocks(0)
    c.start()
    c.begin()
    c.end()                       # a region far shorter than the interval
    r = c.stop()
    assert r["sampled"].startswith("bracketing") and 1 <= r["samples"] <= 2
    assert r["sm_mhz"] == 1800 and r["reasons"] == ["hw_thermal_slowdown"]
