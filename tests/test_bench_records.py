"""Host logic of the benchmark's recorded DRAM traffic: a figure taken by ncu
on one build stays valid while the code of the kernel's sources (without
comments) is unchanged, and is dropped (null in the JSON line) as soon as the
code changes."""

import json
import os
import shutil

import pytest

import bench

CSRC = os.path.join(os.path.dirname(bench.__file__), "io_aware_exact_tiled_gb300", "csrc")


@pytest.fixture
def scratch_tree(tmp_path, monkeypatch):
    """A copy of the kernel sources and the profile records, with bench.py
    pointed at it."""
    root = tmp_path / "repo"
    shutil.copytree(CSRC, root / "io_aware_exact_tiled_gb300" / "csrc")
    (root / "profiles").mkdir()
    shutil.copy(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json"), root / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(root))
    return root


def test_records_match_the_committed_sources():
    d = json.load(open(os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")))
    for kernel, per in d.items():
        if not isinstance(per, dict):
            continue
        for workload, e in per.items():
            assert e["source_sha"] == bench.kernel_source_sha(kernel), (kernel, workload)
            assert bench.recorded_traffic(kernel, workload) == e["dram_bytes_per_launch"]


def test_comment_edits_keep_and_code_edits_drop_the_record(scratch_tree):
    src = scratch_tree / "io_aware_exact_tiled_gb300" / "csrc" / "fa_bwd.cu"
    before = bench.recorded_traffic("fa_bwd_kernel", "sparse16k")
    assert before is not None
    text = src.read_text()
    # a comment line, a trailing comment and blank lines do not count
    src.write_text("// a comment line\n\n" + text.replace("namespace fa {", "namespace fa {  // trailing", 1) + "\n\n")
    assert bench.recorded_traffic("fa_bwd_kernel", "sparse16k") == before
    # any change to the code does
    src.write_text(text.replace("constexpr int kBwdVisMaxTiles = 2048;", "constexpr int kBwdVisMaxTiles = 1024;", 1))
    assert bench.recorded_traffic("fa_bwd_kernel", "sparse16k") is None
    # so does a change in a shared header
    src.write_text(text)
    hdr = scratch_tree / "io_aware_exact_tiled_gb300" / "csrc" / "fa_common.cuh"
    hdr.write_text(hdr.read_text() + "\nnamespace fa { constexpr int kUnused = 1; }\n")
    assert bench.recorded_traffic("fa_bwd_kernel", "sparse16k") is None
