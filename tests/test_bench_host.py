"""Host-side logic of bench.py that decides what a timing means, on CPU:
the L2 rule (weight copies whose calls stream more than 4x L2), the
whole-job rate of N replicas, and the rule that a committed ncu summary's
DRAM bytes count only while the profiled kernel's sources are unchanged."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import synthetic  # noqa: E402


@pytest.mark.parametrize("nbytes", [
    5120 * 17408 * 4 // 8,   # gate_proj, 4 bits (44.6 MB)
    5120 * 17408 * 3 // 8,   # gate_proj, 3 bits
    5120 * 248320 * 6 // 8,  # odd-vocab logits, 6 bits (953 MB)
    512 * 512 * 4 // 8,      # tiny
])
def test_weight_copies_exceed_four_l2(nbytes):
    n = bench.copies_for(nbytes)
    assert 2 <= n <= bench.WEIGHT_COPIES
    # more than 4x L2 in a row, unless the cap of copies is reached
    assert n * nbytes > 4 * bench.L2_BYTES or n == bench.WEIGHT_COPIES


def test_gate_copies_are_the_headline_count():
    g = synthetic.GATE_DECODE
    assert bench.copies_for(g["K"] * g["N"] * g["bits"] // 8) == bench.WEIGHT_COPIES == 12


def test_whole_job_rate_counts_every_rank_over_the_slowest():
    assert bench.whole_job_rate(100.0, 1, 2.0) == 50.0
    assert bench.whole_job_rate(100.0, 4, 2.0) == 200.0


def test_headline_config_names_workload_and_l2_rule():
    c = bench.headline_config(1)
    assert c["workload"] == synthetic.GATE_DECODE["name"]
    assert "M=1,4,8,16" in c["step"]
    assert "> 129 MB" in c["l2"] and "12 rotating weight copies" in c["l2"]
    assert c["parallelism"] == "replicas x1"


def test_profiled_traffic_only_for_unchanged_sources(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("__global__ void k() {}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.source_hash("k.cu")
    (tmp_path / "profiles" / "k.md").write_text(f"# k\nsource_sha256_16: {h}\ndram_bytes_per_launch: 1234\n")
    assert bench.profiled_traffic(("k.cu",), "k.md") == 1234.0
    src.write_text("__global__ void k() { }\n")  # any change to the kernel's sources
    assert bench.profiled_traffic(("k.cu",), "k.md") is None
    assert bench.profiled_traffic(("k.cu",), "missing.md") is None


def test_committed_decode_profile_carries_hash_and_bytes():
    with open(os.path.join(ROOT, "profiles", "decode_gemm_gate_k5120_n17408_b4.md")) as f:
        lines = f.read().splitlines()
    assert any(ln.startswith("source_sha256_16: ") and len(ln.split(": ")[1]) == 16 for ln in lines)
    assert any(ln.startswith("dram_bytes_per_launch: ") for ln in lines)
