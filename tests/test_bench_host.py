"""Host logic of bench.py that needs no GPU: the roofline's DRAM traffic is taken from a committed
profile line only while that line was captured on the current source of the kernel."""
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
