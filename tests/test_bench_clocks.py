"""bench.py's clock sampler keeps the samples taken during the timed region
(host logic; a fake nvidia-smi stands in for the real one)."""
import importlib.util
import os
import stat
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FAKE = """#!{py}
import sys, time
period = 0.05
for a, b in zip(sys.argv, sys.argv[1:]):
    if a == "-lms":
        period = int(b) / 1000
t0 = time.monotonic()
while True:
    el = time.monotonic() - t0
    mhz = 1200 if el < 0.3 else 2070          # a clock that ramps up before the region
    slow = "Active" if el > 0.9 else "Not Active"  # a throttle after it
    print(f"0, {{mhz}}, 2070, 500.0, 0x0, {{slow}}, Not Active, Not Active, Not Active", flush=True)
    time.sleep(period)
"""


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_clock_samples_are_those_of_the_timed_region(tmp_path, monkeypatch):
    tool = tmp_path / "nvidia-smi"
    tool.write_text(FAKE.format(py=sys.executable))
    tool.chmod(tool.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    bench = _bench()
    clk = bench.Clocks(0, period_ms=50).start()
    assert clk.lines, "the sampler runs before the region starts"
    time.sleep(0.45)  # past the ramp
    clk.begin()
    time.sleep(0.3)
    clk.end()
    time.sleep(0.4)  # a throttle is reported after the region only
    clk.stop()
    s = clk.summary()
    assert s is not None and s["samples"] >= 3
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == []


def test_short_region_takes_the_samples_around_it(tmp_path, monkeypatch):
    tool = tmp_path / "nvidia-smi"
    tool.write_text(FAKE.format(py=sys.executable))
    tool.chmod(tool.stat().st_mode | stat.S_IEXEC)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    bench = _bench()
    clk = bench.Clocks(0, period_ms=200).start()
    time.sleep(0.5)
    clk.begin()
    clk.end()  # shorter than the period
    clk.stop()
    s = clk.summary()
    assert s is not None and 1 <= s["samples"] <= 2


def test_no_tool_gives_no_clocks(monkeypatch, tmp_path):
    monkeypatch.setenv("PATH", str(tmp_path))
    bench = _bench()
    clk = bench.Clocks(0).start()
    clk.begin()
    clk.end()
    clk.stop()
    assert clk.summary() is None
