"""Host logic of bench.py: reading a kernel's DRAM traffic from a committed ncu summary.

The roofline's ``traffic`` must come only from a summary captured on the kernel
sources as they are now (same source hash), and be null otherwise.
"""

import os

import bench


def _profiles(tmp_path, text):
    d = tmp_path / "profiles"
    d.mkdir()
    (d / "kernel_case.md").write_text(text)


def test_traffic_read_when_the_hash_matches(tmp_path, monkeypatch):
    _profiles(tmp_path, "# k\n\n- workload: wl_a (notes)\n- source_sha: abc123 (three files)\n"
                        "- traffic_bytes_per_launch: 540299520\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda sources=bench.KERNEL_SOURCES: "abc123")
    assert bench.recorded_traffic("wl_a") == 540299520


def test_traffic_null_for_stale_sources_or_other_workloads(tmp_path, monkeypatch):
    _profiles(tmp_path, "- workload: wl_a\n- source_sha: abc123\n- traffic_bytes_per_launch: 7\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_hash", lambda sources=bench.KERNEL_SOURCES: "def456")
    assert bench.recorded_traffic("wl_a") is None
    monkeypatch.setattr(bench, "source_hash", lambda sources=bench.KERNEL_SOURCES: "abc123")
    assert bench.recorded_traffic("wl_b") is None


def test_source_hash_covers_device_files_only():
    """Each hash is over its kernel's device sources, and the two kernels' hashes differ."""
    csrc = os.path.join(bench.ROOT, "split_kv_decode_fd_gb300", "csrc")
    for name in bench.KERNEL_SOURCES + bench.PREFILL_SOURCES:
        assert os.path.exists(os.path.join(csrc, name)), name
    assert "fd_api.cu" not in bench.KERNEL_SOURCES + bench.PREFILL_SOURCES
    assert bench.source_hash() != bench.source_hash(bench.PREFILL_SOURCES)
    assert len(bench.source_hash()) == 12


def test_committed_summaries_describe_the_current_sources():
    """Every committed ncu summary names the device-source hash of the kernel it
    covers, and that hash is the one of the sources as they are now: a kernel
    edited after its capture shows up here, not as a silently null traffic."""
    import glob
    import re

    paths = sorted(glob.glob(os.path.join(bench.ROOT, "profiles", "*.md")))
    assert paths, "no ncu summaries committed"
    current = {"split": bench.source_hash(), "prefill": bench.source_hash(bench.PREFILL_SOURCES)}
    for p in paths:
        text = open(p).read()
        m = re.search(r"source_sha:\s*`?([0-9a-f]{12})", text)
        assert m, f"{os.path.basename(p)} names no source hash"
        kind = "prefill" if "fd_prefill_kernel" in os.path.basename(p) else "split"
        assert m.group(1) == current[kind], f"{os.path.basename(p)} was taken on other {kind} sources"
