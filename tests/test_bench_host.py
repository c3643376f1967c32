"""Host logic of bench.py that needs no GPU: the DRAM traffic reported beside
the roofline is taken from the committed ncu summary only when that summary
was measured on the current decode-kernel source and covers the benchmarked
batch with the automatic split; otherwise the key is null."""

import hashlib
import os

import pytest

import bench

SRC_REL = os.path.join("nvfp4_quantised_paged_gb300", "csrc", "decode_attention.cu")


def _tree(tmp_path, source: bytes, sha: str):
    src = tmp_path / SRC_REL
    src.parent.mkdir(parents=True)
    src.write_bytes(source)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "decode_kernel_dram.txt").write_text(
        "# comment: with a colon\n"
        "kernel_source_sha256_16: %s\n"
        "dram_bytes_per_launch_batch8: 305571072\n"
        "dram_bytes_per_launch_full_size: 2444568576\n" % sha)


@pytest.fixture
def fake_root(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def test_traffic_for_the_measured_batches_of_the_current_source(fake_root):
    source = b"// kernel source\n"
    _tree(fake_root, source, hashlib.sha256(source).hexdigest()[:16])
    assert bench.decode_kernel_traffic(64, 0) == 2444568576.0
    assert bench.decode_kernel_traffic(8, 0) == 305571072.0


def test_no_traffic_for_other_batches_or_explicit_splits(fake_root):
    source = b"// kernel source\n"
    _tree(fake_root, source, hashlib.sha256(source).hexdigest()[:16])
    assert bench.decode_kernel_traffic(16, 0) is None
    assert bench.decode_kernel_traffic(64, 500) is None


def test_no_traffic_once_the_source_changed(fake_root):
    _tree(fake_root, b"// kernel source, edited\n", hashlib.sha256(b"// kernel source\n").hexdigest()[:16])
    assert bench.decode_kernel_traffic(64, 0) is None


def test_no_traffic_without_a_summary(fake_root):
    src = fake_root / SRC_REL
    src.parent.mkdir(parents=True)
    src.write_bytes(b"x")
    assert bench.decode_kernel_traffic(64, 0) is None


def test_both_arms_report_the_same_workload_keys():
    import workloads
    w = workloads.decode_32k()
    c = bench.workload_config(w, 1)
    assert c["workload"] == w.name and c["batch"] == 64 and c["seq_len"] == 32768
    assert (c["num_q_heads"], c["num_kv_heads"], c["head_dim"], c["page_size"]) == (64, 8, 128, 64)
    assert c["parallelism"] == "single GPU" and bench.workload_config(w, 4)["parallelism"] == "replicas"


def test_roofline_kernel_is_timed_over_many_launches_whatever_the_steps():
    """The decode kernel's roofline time is the mean of a fixed number of
    dedicated launches after the timed region, not of a sample of it."""
    assert bench.ROOFLINE_LAUNCHES >= 50
    assert bench.PROFILE_EVERY >= 1
