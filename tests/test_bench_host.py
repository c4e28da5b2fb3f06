"""Host-side logic of bench.py that needs no GPU: the clock-sample summary
(median SM clock under load, throttle reasons seen) and the traffic lookup
keyed by the kernel sources."""
import os
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _sampler_with(lines):
    s = bench.ClockSampler(0)
    fd, s.path = tempfile.mkstemp(suffix=".csv")
    with os.fdopen(fd, "w") as f:
        f.write("\n".join(lines) + "\n")
    return s


def test_clock_summary_median_under_load_and_reasons():
    idle = "0, 345, 2070, 120.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active"
    busy = "0, {mhz}, 2070, 1300.0, 0x0000000000000004, Not Active, Not Active, Not Active, {cap}"
    lines = [idle, busy.format(mhz=2070, cap="Not Active"), busy.format(mhz=2055, cap="Active"),
             busy.format(mhz=2070, cap="Not Active"), "garbage line", idle]
    out = _sampler_with(lines).summary()
    assert out["sm_mhz"] == 2070.0          # the idle samples (345 MHz) are not under load
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples"] == 5


def test_clock_summary_reports_slowdowns():
    line = "0, 1500, 2070, 900.0, 0x0000000000000008, Active, Not Active, Active, Not Active"
    out = _sampler_with([line, line]).summary()
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_samples():
    out = _sampler_with([]).summary()
    assert out["reasons"] == ["unavailable"] and out["sm_mhz"] is None


def test_traffic_is_keyed_by_the_kernel_sources(monkeypatch):
    assert bench.kernel_traffic() == bench.TRAFFIC.get(bench.kernel_hash())
    monkeypatch.setattr(bench, "kernel_hash", lambda: "0" * 16)
    assert bench.kernel_traffic() is None


def test_kernel_hash_follows_code_not_comments(monkeypatch, tmp_path):
    import shutil
    src = os.path.join(ROOT, "w6a8_quantized_linear_gb300", "csrc")
    dst = tmp_path / "w6a8_quantized_linear_gb300" / "csrc"
    dst.mkdir(parents=True)
    for f in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(src, f), dst / f)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_hash()
    k = dst / "qlin_layout.h"
    k.write_text(k.read_text() + "\n// a remark\n/* another\n   remark */\n")
    assert bench.kernel_hash() == h0
    k.write_text(k.read_text() + "\nconstexpr int qlin_unused_constant = 1;\n")
    assert bench.kernel_hash() != h0


def test_job_throughput_is_total_bytes_over_slowest_rank():
    assert abs(bench.job_gbs(4, 10**9, 2.0) - 2000.0) < 1e-9
