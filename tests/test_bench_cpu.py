"""Host logic of bench.py that decides what a bench line reports: the clock
record's parsing and the code hash that keeps recorded ncu counters tied to
the kernel source they were taken on (runs without a GPU)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeProc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def test_clock_record_skips_lines_before_the_region_and_reads_reasons():
    c = bench.ClockSampler(0)
    c.proc = _FakeProc()
    idle = "0, 1200, 2070, 500, 0x0, Not Active, Not Active, Not Active, Not Active"
    c.lines = [idle,
               "0, 2070, 2070, 900, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 2055, 2070, 950, 0x4, Not Active, Not Active, Not Active, Active",
               "garbage"]
    c.skip = 1  # printed before the timed region started
    r = c.stop()
    assert r["samples"] == 2 and r["sm_mhz"] == 2062.5 and r["sm_max_mhz"] == 2070.0
    assert r["reasons"] == ["sw_power_cap"]
    c2 = bench.ClockSampler(0)
    c2.proc = _FakeProc()
    c2.lines = [idle]
    c2.skip = 1
    assert c2.stop()["samples"] == 0  # bench.py then reports the decode window's record


def test_code_hash_ignores_comments_and_blank_lines(tmp_path):
    a, b, c = tmp_path / "a.cuh", tmp_path / "b.cuh", tmp_path / "c.cuh"
    a.write_text("int x = 1;  // one\n\n// a note\nint y = 2;\n")
    b.write_text("// header\nint x = 1;\n   int y = 2;  // two\n")
    c.write_text("int x = 1;\nint y = 3;\n")
    assert bench._src_sha(str(a)) == bench._src_sha(str(b))
    assert bench._src_sha(str(a)) != bench._src_sha(str(c))
