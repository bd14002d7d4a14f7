"""Host logic of the benchmark's stored DRAM traffic (no GPU).

A traffic record under profiles/ counts only while the sources of the kernels it was measured on
are unchanged: the record carries a digest of those sources and the local headers they include,
and bench.py reports the stored bytes only when that digest still matches.  Checked here on a
scratch copy of the source tree: the digest follows every included header, a step with two kernel
files depends on both, and a record goes stale when any of them changes.
"""
import os
import shutil

import pytest

import bench

WORKLOADS = sorted(bench.KERNEL_SOURCE)


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """bench.ROOT pointed at a copy of the kernel sources and the committed traffic records."""
    src = os.path.join(bench.ROOT, "lightning_attention_gb300", "csrc")
    dst = tmp_path / "lightning_attention_gb300" / "csrc"
    shutil.copytree(src, dst, ignore=shutil.ignore_patterns("*.o", "*.so", "__pycache__"))
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def touch(path):
    with open(path, "a") as f:
        f.write("\n// edited\n")


def test_every_workload_names_existing_sources():
    csrc = os.path.join(bench.ROOT, "lightning_attention_gb300", "csrc")
    for w in WORKLOADS:
        files = bench.KERNEL_SOURCE[w]
        for f in [files] if isinstance(files, str) else files:
            assert os.path.exists(os.path.join(csrc, f)), (w, f)
        assert len(bench.source_digest(files)) == 16


def test_digest_follows_included_headers(tree):
    before = bench.source_digest("la_recurrent.cu")
    touch(tree / "lightning_attention_gb300" / "csrc" / "la_internal.h")
    assert bench.source_digest("la_recurrent.cu") != before


def test_two_file_step_depends_on_both_files(tree):
    files = bench.KERNEL_SOURCE["long_prefill"]
    assert not isinstance(files, str) and len(files) == 2
    before = bench.source_digest(files)
    touch(tree / "lightning_attention_gb300" / "csrc" / files[1])
    assert bench.source_digest(files) != before
    assert bench.source_digest(files[0]) != bench.source_digest(files)


def test_record_goes_stale_when_its_source_changes(tree):
    records = [w for w in WORKLOADS if (tree / "profiles" / f"traffic_{w}.txt").exists()]
    assert records, "no traffic records to check"
    fresh = [w for w in records if bench.stored_traffic(w) is not None]
    for w in fresh:
        assert bench.stored_traffic(w) > 0
    files = bench.KERNEL_SOURCE[records[0]]
    touch(tree / "lightning_attention_gb300" / "csrc" / (files if isinstance(files, str) else files[0]))
    same = [w for w in records if bench.KERNEL_SOURCE[w] == files]
    for w in same:
        assert bench.stored_traffic(w) is None, w


def test_missing_or_malformed_record_reads_as_none(tree):
    (tree / "profiles" / "traffic_decode.txt").write_text("source_sha256_16: 0\n")
    assert bench.stored_traffic("decode") is None
    (tree / "profiles" / "traffic_decode.txt").unlink()
    assert bench.stored_traffic("decode") is None
