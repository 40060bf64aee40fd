"""The benchmark's host-side helpers on CPU: the default step count (about one second of timed
work) and the clock sampler's timed-region window, driven by a stand-in for `nvidia-smi` (a
Python script run by this interpreter) that writes one CSV sample every 50 ms."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_auto_steps():
    # 24 us per step: about 1 s of work, rounded up to a multiple of the replicas
    n = bench.auto_steps(24e-6, 25)
    assert n % 25 == 0 and 41_000 <= n <= 42_000
    # slow steps keep the floor, fast ones the cap
    assert bench.auto_steps(10e-3, 1) == 2000
    assert bench.auto_steps(1e-12, 1) == 2_000_000
    assert bench.auto_steps(1e-12, 7) % 7 == 0
    # a bad warm-up timing falls back to the floor
    assert bench.auto_steps(float("nan"), 3) == 2001
    assert bench.auto_steps(0.0, 1) == 2000
    assert bench.auto_steps(float("inf"), 4) == 2000


def _fake_smi(tmp_path, mhz_of_line):
    """The sampler command of a script that prints 9 CSV fields per line, one line per 50 ms,
    flushing each (the SM clock of line i is mhz_of_line(i)); it ignores its arguments."""
    script = tmp_path / "fake_smi.py"
    clocks = ", ".join(str(mhz_of_line(i)) for i in range(400))
    script.write_text(
        "import sys, time\n"
        f"clocks = [{clocks}]\n"
        "for i, c in enumerate(clocks):\n"
        "    print(f'0, {c}, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, "
        "{\"Active\" if c < 1000 else \"Not Active\"}', flush=True)\n"
        "    time.sleep(0.05)\n")
    return (sys.executable, str(script))


def test_clock_window_keeps_the_timed_region(tmp_path):
    # idle clocks before the region, full clocks after line 10 (the sampler is started, then
    # the region is marked once the load runs)
    s = bench.ClockSampler(0, cmd=_fake_smi(tmp_path, lambda i: 2070 if i >= 10 else 345))
    s.start()
    deadline = time.time() + 10
    while time.time() < deadline:  # wait until the idle lines have been written
        s.marks = []
        s.mark()
        if s.marks[0] >= 12:
            break
        time.sleep(0.05)
    time.sleep(0.3)
    s.mark()
    out = s.stop()
    assert out["window"] == "timed region"
    assert out["samples"] >= 3
    assert out["sm_mhz"] == 2070 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == []


def test_clock_window_falls_back_to_the_whole_run(tmp_path):
    s = bench.ClockSampler(0, cmd=_fake_smi(tmp_path, lambda i: 345 if i == 0 else 2070))
    s.start()
    s.mark()
    s.marks.append(s.marks[-1])  # no sample between the marks
    time.sleep(0.4)
    out = s.stop()
    assert out["window"] == "whole run"
    assert out["samples"] >= 2
    assert out["reasons"] == ["sw_power_cap"]  # line 0 reported it


def test_clock_sampler_without_nvidia_smi(tmp_path):
    s = bench.ClockSampler(0, cmd=(str(tmp_path / "no_such_program"),))
    s.start()
    s.mark()
    s.mark()
    assert s.stop() is None


def test_captured_traffic_follows_the_kernel_sources():
    """The line reports a kernel's ncu DRAM traffic only while the hash of its sources matches
    the one the capture was taken on; every workload's entry names a known kernel family."""
    families = {"pre4096": "tc", "pre32768": "tc", "dec1": "decode", "dec8": "decode",
                "hash64": "mma"}
    assert set(bench.TRAFFIC) <= set(families)
    for name, (nbytes, h) in bench.TRAFFIC.items():
        assert nbytes > 0 and len(h) == 16
        assert bench.captured_traffic(name, h) == nbytes
        assert bench.captured_traffic(name, "0" * 16) is None
    assert bench.captured_traffic("tiny", bench.kernel_source_hash(bench.KERNEL_SOURCES["tc"])) is None
    for fam, files in bench.KERNEL_SOURCES.items():
        assert len(bench.kernel_source_hash(files)) == 16

