"""Host-side statistics and bookkeeping of bench.py (no GPU).

The rows report the mean of the middle 60% of their timed runs; the
roofline's DRAM traffic is read from a committed ncu record only while the
GEMM's source still hashes to the value recorded with it.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_trimmed_mean_drops_a_fifth_at_each_end():
    ts = [100.0, 1.0, 2.0, 2.0, 2.0, 4.0, 4.0, 4.0, 4.0, 0.0]    # sorted: 0,1,2,2,2,4,4,4,4,100
    assert bench.trimmed_mean(ts) == (2 + 2 + 2 + 4 + 4 + 4) / 6
    # event times in ~2 us steps: a mix of two steps averages between them
    assert abs(bench.trimmed_mean([18.4] * 12 + [16.4] * 8) - (18.4 * 8 + 16.4 * 4) / 12) < 1e-12


def test_trimmed_mean_of_few_samples_keeps_them_all():
    assert bench.trimmed_mean([3.0]) == 3.0
    assert bench.trimmed_mean([1.0, 3.0]) == 2.0


def test_traffic_is_reported_only_for_the_source_it_was_taken_on():
    rec = json.load(open(os.path.join(ROOT, "profiles", "gemm_dense_linear_traffic.json")))
    assert rec["dram_bytes_per_launch"] == rec["dram_read_bytes"] + rec["dram_write_bytes"]
    if rec["kernel_src_sha"] == bench.kernel_source_sha():
        assert bench.ncu_traffic() == rec["dram_bytes_per_launch"]
    else:
        assert bench.ncu_traffic() is None


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """A comment edit keeps the record; a code edit does not."""
    import shutil
    src = os.path.join(ROOT, "fp8_fine_grained_16_b300", "csrc")
    dst = tmp_path / "fp8_fine_grained_16_b300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_sha()
    g = dst / "gemm.cu"
    g.write_text(g.read_text() + "\n// a comment\n\n")
    assert bench.kernel_source_sha() == h0
    g.write_text(g.read_text() + "static int unused_for_the_hash_test = 1;\n")
    assert bench.kernel_source_sha() != h0


def test_job_throughput_counts_every_rank():
    assert bench.job_throughput(4.2e11, 1, 0.2) == 4.2e11 / 0.2e-3
    assert bench.job_throughput(4.2e11, 8, 0.2) == 8 * 4.2e11 / 0.2e-3
