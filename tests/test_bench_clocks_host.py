"""bench.py's clock record: only nvidia-smi samples taken inside the timed region count."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _FakeSmi:
    def __init__(self, text):
        self.text = text

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.text, ""


def _line(t, mhz, reasons=("Not Active",) * 4):
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(t)) + ".%03d" % int((t % 1) * 1000)
    return ", ".join(["0", str(mhz), "2070", "900.0", "0x0", *reasons, stamp])


def test_samples_outside_the_region_are_dropped():
    t0 = 1_800_000_000.0
    lines = [
        _line(t0 - 0.30, 1200, ("Not Active", "Not Active", "Not Active", "Active")),  # before the region
        _line(t0 + 0.05, 2070),
        _line(t0 + 0.10, 2055),
        _line(t0 + 0.15, 2070),
        _line(t0 + 0.60, 900, ("Active", "Not Active", "Not Active", "Not Active")),   # after it
    ]
    c = bench.Clocks("0")
    c.proc = _FakeSmi("\n".join(lines) + "\n")
    r = c.stop((t0, t0 + 0.2))
    assert r["samples"] == 3 and r["which"] == "inside the timed region"
    assert r["sm_mhz"] == 2070.0 and r["sm_max_mhz"] == 2070.0 and r["reasons"] == []


def test_no_sample_inside_falls_back_to_all_and_says_so():
    t0 = 1_800_000_000.0
    lines = [_line(t0 - 0.2, 2070), _line(t0 + 0.5, 2060, ("Not Active", "Not Active", "Not Active", "Active"))]
    c = bench.Clocks("0")
    c.proc = _FakeSmi("\n".join(lines) + "\n")
    r = c.stop((t0, t0 + 0.01))
    assert r["samples"] == 2 and r["which"].startswith("none inside")
    assert r["reasons"] == ["sw_power_cap"]


def test_unavailable_and_empty():
    c = bench.Clocks("0")
    assert c.stop()["reasons"] == ["nvidia-smi unavailable"]
    c.proc = _FakeSmi("")
    assert c.stop((0.0, 1.0))["reasons"] == ["no samples"]


def test_summary_of_a_second_window_after_stop():
    """The e2e region's clocks come from the same samples, over its own window."""
    t0 = 1_800_000_000.0
    lines = [_line(t0 + 0.05, 2070), _line(t0 + 0.10, 2060),
             _line(t0 + 1.05, 1900, ("Not Active", "Not Active", "Not Active", "Active")),
             _line(t0 + 1.10, 1950, ("Not Active", "Not Active", "Not Active", "Active"))]
    c = bench.Clocks("0")
    c.proc = _FakeSmi("\n".join(lines) + "\n")
    r = c.stop((t0, t0 + 0.2))
    assert r["samples"] == 2 and r["reasons"] == []
    r2 = c.summary((t0 + 1.0, t0 + 1.2))
    assert r2["samples"] == 2 and r2["reasons"] == ["sw_power_cap"] and r2["sm_mhz"] == 1950.0


def test_profile_tag_names_the_workload_not_its_layer_cut():
    assert bench.profile_tag("qwen14b_48L_8prefix_b368") == "qwen14b_8prefix_b368"
    assert bench.profile_tag("qwen14b_48L_8prefix_b368_first1layers") == "qwen14b_8prefix_b368"
    assert bench.profile_tag("llama8b_32L_lp16384_b64_s256-2048") == "llama8b_lp16384_b64"
    assert bench.profile_tag("llama8b_32L_lp16384_b512_s256-2048_first1layers") == "llama8b_lp16384_b512"
