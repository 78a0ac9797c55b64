"""bench.py's host logic, without a GPU: the split of M rows into sequences,
the arithmetic type it reports per path, and the rule that an ncu traffic
figure is reported only for the kernel sources it was captured on."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


@pytest.mark.parametrize("M,G", [(16, 4), (10, 3), (64, 8), (7, 7), (1, 1), (65536, 100)])
def test_group_rows_split_evenly(M, G):
    rows = bench.group_rows(M, G)
    assert len(rows) == G and sum(rows) == M
    assert max(rows) - min(rows) <= 1 and min(rows) >= 1


@pytest.mark.parametrize("M,G", [(4, 0), (4, 5)])
def test_group_rows_rejects(M, G):
    with pytest.raises(ValueError):
        bench.group_rows(M, G)


def test_path_dtype():
    assert bench.path_dtype("gemm", 8) == "f32"
    assert bench.path_dtype("gemm", 16) == "f32"
    assert bench.path_dtype("gemm", 17) == "bf16"
    assert bench.path_dtype("gateup", 64) == "bf16"
    assert bench.path_dtype("decode", 64) == "f32"


def test_source_hash_ignores_comments_and_follows_code(tmp_path, monkeypatch):
    """The hash of a kernel's sources does not move when only comments change,
    and does when code does."""
    csrc = tmp_path / "trellis_quantized_weight_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "decode_kernel.cu").write_text("int a = 1;  // note\n/* block */\n")
    (csrc / "trellis_device.cuh").write_text("int b = 2;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash("decode")
    (csrc / "decode_kernel.cu").write_text("int a = 1;  // another note\n")
    assert bench.kernel_source_hash("decode") == h0
    (csrc / "decode_kernel.cu").write_text("int a = 3;\n")
    assert bench.kernel_source_hash("decode") != h0
    (csrc / "decode_kernel.cu").write_text("int a = 1;\n")
    (csrc / "trellis_device.cuh").write_text("int b = 4;\n")   # shared device code
    assert bench.kernel_source_hash("decode") != h0


def test_traffic_only_for_the_captured_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "trellis_quantized_weight_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "gemm_tc_kernel.cu").write_text("int t = 1;\n")
    (csrc / "trellis_device.cuh").write_text("int b = 2;\n")
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash("gemm_tc")
    (prof / "gemm_tc_w.md").write_text(f"- kernel_source_hash: `{h}`\n- dram_bytes_per_launch: 12345\n")
    assert bench.profiled_traffic("gemm_tc", "w") == 12345
    (csrc / "gemm_tc_kernel.cu").write_text("int t = 2;\n")
    assert bench.profiled_traffic("gemm_tc", "w") is None
    assert bench.profiled_traffic("gemm_tc", "absent") is None
