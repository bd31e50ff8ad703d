"""bench.py host logic on CPU: the profile a run's traffic comes from, and the committed profiles."""
import glob
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def name_for(argv, M=0, N=0, workload_dbias=False):
    old = sys.argv
    sys.argv = ["bench.py"] + argv
    try:
        args = bench.parse_args()
    finally:
        sys.argv = old
    return bench.profile_name(args, M, N, workload_dbias)


@pytest.mark.parametrize("argv,wd,want", [
    ([], False, "quantize_fc1_8192x28672"),
    (["--workload", "grad_16384x8192"], True, "quantize_grad_16384x8192"),
    (["--workload", "grad_16384x8192", "--dbias"], True, "quantize_grad_16384x8192"),
    (["--workload", "moe_64x65536x7168", "--dbias"], False, "quantize_moe_64x65536x7168_dbias"),
    (["--workload", "grad_16384x8192", "--dact", "gelu"], True, "quantize_dact_grad_16384x8192_gelu"),
    (["--act", "gelu"], False, "quantize_fc1_8192x28672_gelu"),
    (["--swizzled", "--amax"], False, "quantize_fc1_8192x28672_swizzled_amax"),
    (["--glu", "silu"], False, "quantize_gated_fc1_8192x28672_silu"),
    (["--dglu", "silu"], False, "quantize_dgated_fc1_8192x28672_silu"),
])
def test_profile_name_follows_kernel_workload_and_options(argv, wd, want):
    assert name_for(argv, workload_dbias=wd) == want


def test_profile_name_with_a_shape_override():
    assert name_for(["--shape", "8192x16384"], 8192, 16384) == "quantize_fc1_8192x16384"


def test_every_committed_profile_names_its_sources_and_traffic():
    files = sorted(glob.glob(os.path.join(ROOT, "profiles", "quantize_*.md")))
    assert files
    for f in files:
        text = open(f).read()
        assert re.search(r"kernel_source_sha:\s*[0-9a-f]{16}\b", text), f
        assert re.search(r"dram_bytes_per_step:\s*[0-9]+\b", text), f
        assert "--clock-control none" in text, f


def test_traffic_is_reported_only_for_matching_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    sha = bench.kernel_source_sha()
    (tmp_path / "profiles" / "quantize_x.md").write_text(f"kernel_source_sha: {sha}\ndram_bytes_per_step: 123\n")
    (tmp_path / "profiles" / "quantize_y.md").write_text("kernel_source_sha: 0000000000000000\ndram_bytes_per_step: 9\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda: sha)
    assert bench.profiled_traffic("quantize_x") == 123
    assert bench.profiled_traffic("quantize_y") is None
    assert bench.profiled_traffic("quantize_missing") is None


def test_kernel_sources_cover_every_csrc_file():
    """The sources hashed into kernel_source_sha are exactly the CUDA sources the library builds from."""
    csrc = sorted(os.path.relpath(p, ROOT) for p in glob.glob(os.path.join(ROOT, "mxfp8_block_scaled_04_gb300",
                                                                          "csrc", "*.cu*")))
    assert sorted(bench.KERNEL_SOURCES) == csrc
