"""Host logic of bench.py that needs no GPU: the roofline's DRAM traffic is taken from a committed
profile line only while that line was captured on the current source of the kernel, and the clock
record (median SM clock under load, throttle reasons) is read from nvidia-smi's samples."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.fixture()
def tree(tmp_path, monkeypatch):
    csrc = tmp_path / "complexity_matmul_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in ("gemm_pair.cu", "ptx.cuh", "epilogue.cuh", "plain_common.cuh"):
        (csrc / name).write_text(f"// {name}\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _profile(tree, source, n=16384, nbytes=123456789, kernel="gemm_pair.cu"):
    (tree / "profiles" / "k.md").write_text(
        f"# summary\n\ntraffic_per_launch: kernel={kernel} n={n} bytes={nbytes} source={source}\n")


def test_traffic_read_for_current_source(tree):
    _profile(tree, bench._kernel_source_hash("gemm_pair.cu"))
    assert bench._traffic("gemm_pair.cu", 16384) == 123456789


def test_traffic_dropped_once_any_hashed_file_changes(tree):
    _profile(tree, bench._kernel_source_hash("gemm_pair.cu"))
    for name in ("gemm_pair.cu", "ptx.cuh", "epilogue.cuh", "plain_common.cuh"):
        p = tree / "complexity_matmul_gb300" / "csrc" / name
        old = p.read_text()
        p.write_text(old + "// changed\n")
        assert bench._traffic("gemm_pair.cu", 16384) is None, name
        p.write_text(old)
    assert bench._traffic("gemm_pair.cu", 16384) == 123456789


def test_traffic_needs_matching_kernel_and_size(tree):
    _profile(tree, bench._kernel_source_hash("gemm_pair.cu"))
    assert bench._traffic("gemm_pair.cu", 8192) is None
    (tree / "complexity_matmul_gb300" / "csrc" / "lcma_pair.cu").write_text("// lcma\n")
    assert bench._traffic("lcma_pair.cu", 16384) is None


def test_no_profiles_folder_means_no_traffic(tree):
    (tree / "profiles").rmdir()
    assert bench._traffic("gemm_pair.cu", 16384) is None


def _clock_line(mhz, reasons=()):
    flags = ["Active" if r in reasons else "Not Active"
             for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")]
    return ", ".join(["0", str(mhz), "2070", "1200.5", "0x0000000000000004"] + flags)


def test_clock_summary_without_samples():
    cs = bench.ClockSampler(0)
    assert cs.summary()["reasons"] == ["clock sampling unavailable"]


def test_clock_summary_reports_power_cap_and_loaded_median():
    cs = bench.ClockSampler(0)
    idle = [_clock_line(345) for _ in range(4)]
    busy = [_clock_line(m, ("sw_power_cap",)) for m in (1980, 2010, 2040, 2070)]
    cs.out = "\n".join(idle + busy) + "\n"
    s = cs.summary()
    assert s["reasons"] == ["sw_power_cap"]
    assert s["sm_max_mhz"] == 2070.0
    assert s["sm_mhz"] == 2025.0          # median of the upper half: the samples under load
    assert s["samples"] == 8


def test_clock_summary_flags_slowdowns_and_skips_malformed_lines():
    cs = bench.ClockSampler(0)
    cs.out = "\n".join([_clock_line(1500, ("hw_slowdown",)), "0, [N/A], 2070, 1, 0x0, a, b, c, d", "garbage",
                        _clock_line(1600, ("sw_thermal_slowdown",))])
    s = cs.summary()
    assert s["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert s["samples"] == 2
