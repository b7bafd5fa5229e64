"""Host-side pieces of bench.py that need no GPU: the profile-traffic lookup (only while the
kernel's sources are unchanged since the capture) and the command-line rules."""
import os
import shutil

import pytest

import bench


def test_committed_profiles_name_their_command_and_digest():
    # every ncu summary that bench.py can read states the command and the source digest
    for name in os.listdir(os.path.join(bench.ROOT, "profiles")):
        if not (name.startswith("sgemm_ffma_") or name.startswith("hgemm_tcgen05_")):
            continue
        text = open(os.path.join(bench.ROOT, "profiles", name)).read()
        assert "ncu " in text and "--clock-control none" in text, name
        assert "source_sha256_16:" in text and "dram_bytes_per_launch:" in text, name


def test_traffic_is_reported_only_for_the_captured_sources(tmp_path, monkeypatch):
    # A copy of the repository layout with one summary: the digest line decides.
    root = tmp_path
    (root / "profiles").mkdir()
    shutil.copytree(os.path.join(bench.ROOT, "dense_gemm_sgemm_gb300", "csrc"),
                    root / "dense_gemm_sgemm_gb300" / "csrc")
    monkeypatch.setattr(bench, "ROOT", str(root))
    digest = bench.csrc_digest("sgemm_ffma")
    prof = root / "profiles" / "p.txt"
    prof.write_text(f"# comment: 1\nsource_sha256_16: {digest}\ndram_bytes_per_launch: 1234\n"
                    "duration_us: 56.5\n")
    assert bench._traffic_from_profile("sgemm_ffma", "p.txt") == 1234.0
    assert bench._ncu_duration_us("sgemm_ffma", "p.txt") == 56.5
    # any change to the kernel's sources makes the captured counters stale
    src = root / "dense_gemm_sgemm_gb300" / "csrc" / "sgemm_kernel.cuh"
    src.write_text(src.read_text() + "\n")
    assert bench._traffic_from_profile("sgemm_ffma", "p.txt") is None
    assert bench._ncu_duration_us("sgemm_ffma", "p.txt") is None
    # the other kernel's digest does not depend on the SGEMM sources
    assert bench.csrc_digest("hgemm_tcgen05") != bench.csrc_digest("sgemm_ffma")
    assert bench._traffic_from_profile("sgemm_ffma", "missing.txt") is None


def test_warmup_must_be_at_least_three():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
