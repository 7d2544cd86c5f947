"""Host logic of bench.py that needs no GPU: the clock record keeps only the
nvidia-smi samples stamped inside the timed region (widening the window
when the region is shorter than the sampling interval) and reports the
throttle reasons seen there; the whole-job rate divides the units of all
ranks by the slowest rank's time."""
import datetime
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def fake_clocks(lines, t_begin):
    c = bench.Clocks.__new__(bench.Clocks)
    text = "\n".join(lines) + "\n"
    c.p = subprocess.Popen([sys.executable, "-c", f"import sys; sys.stdout.write({text!r})"],
                           stdout=subprocess.PIPE, text=True)
    c.t_begin = t_begin
    return c


def sample(ts, sm, reasons=("Not Active",) * 4):
    return ", ".join([ts.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3], str(sm), "2070", "600.5", "0x0", *reasons])


def test_only_samples_inside_the_region_count():
    t0 = datetime.datetime.now()
    lines = [sample(t0 - datetime.timedelta(milliseconds=300), 1000),          # idle, before
             sample(t0 + datetime.timedelta(milliseconds=10), 2070),
             sample(t0 + datetime.timedelta(milliseconds=35), 2070,
                    ("Not Active", "Not Active", "Not Active", "Active")),     # power cap inside
             sample(t0 + datetime.timedelta(milliseconds=60), 2055),
             sample(t0 + datetime.timedelta(seconds=30), 900,
                    ("Active", "Not Active", "Not Active", "Not Active"))]     # after: ignored
    c = fake_clocks(lines, t0)
    r = c.stop(t_end=t0 + datetime.timedelta(milliseconds=100))   # after the three samples inside
    assert r["samples"] == 3
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    assert "window" not in r


def test_short_region_widens_the_window():
    t0 = datetime.datetime.now()
    lines = [sample(t0 - datetime.timedelta(milliseconds=40), 2070),
             sample(t0 - datetime.timedelta(seconds=5), 800)]
    c = fake_clocks(lines, t0)
    r = c.stop(t_end=t0 + datetime.timedelta(milliseconds=20))
    assert r["samples"] == 1 and r["sm_mhz"] == 2070.0
    assert "widened" in r["window"]


def test_unparseable_lines_are_skipped():
    t0 = datetime.datetime.now()
    lines = ["[N/A], [N/A]", "garbage", sample(t0 + datetime.timedelta(milliseconds=5), 2070)]
    r = fake_clocks(lines, t0).stop(t_end=t0 + datetime.timedelta(milliseconds=50))
    assert r["samples"] == 1


def test_whole_job_rate():
    assert bench.whole_job_rate(4096, 2, 10, 0.5) == 4096 * 2 * 10 / 0.5
