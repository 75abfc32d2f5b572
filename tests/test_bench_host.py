"""The benchmark's host-side bookkeeping, on CPU.

`roofline.traffic` is the DRAM bytes of one launch of the headline kernel from
a committed ncu capture, reported only while the kernel's sources are the ones
the capture was taken of (a SHA-256 over them); a changed kernel reports null.
"""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SOURCES = ["gemm_collective_gb300/csrc/fcc_gemm.cu", "gemm_collective_gb300/csrc/fcc_ptx.cuh"]


def _write_capture(root, sha, total=123456789):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "k.traffic.txt"), "w") as f:
        f.write(f"# a comment = with an equals sign\nsource_sha256 = {sha}\n"
                f"dram_bytes_read = 1\nbytes_per_launch_full = {total}\n")


def _sources(root, texts):
    paths = []
    for i, t in enumerate(texts):
        p = f"src{i}.cu"
        with open(os.path.join(root, p), "w") as f:
            f.write(t)
        paths.append(p)
    return paths


def test_traffic_reported_while_sources_match(tmp_path, monkeypatch):
    root = str(tmp_path)
    paths = _sources(root, ["kernel a", "header b"])
    sha = hashlib.sha256(b"kernel a" + b"header b").hexdigest()
    _write_capture(root, sha)
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.kernel_traffic("k", paths) == 123456789.0


def test_traffic_null_once_a_source_changes(tmp_path, monkeypatch):
    root = str(tmp_path)
    sha = hashlib.sha256(b"kernel a" + b"header b").hexdigest()
    _write_capture(root, sha)
    paths = _sources(root, ["kernel a", "header b, edited"])
    monkeypatch.setattr(bench, "ROOT", root)
    assert bench.kernel_traffic("k", paths) is None
    assert bench.kernel_traffic("missing", paths) is None


def test_committed_headline_capture_is_parsed():
    """The committed capture holds a positive per-launch byte count; it is
    reported as long as its hash names the committed kernel sources."""
    got = bench.kernel_traffic("gemm_rs_fused", SOURCES)
    h = hashlib.sha256()
    for s in SOURCES:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    with open(os.path.join(ROOT, "profiles", "gemm_rs_fused.traffic.txt")) as f:
        recorded = [ln.split("=", 1)[1].strip() for ln in f if ln.startswith("source_sha256")]
    assert recorded, "no source_sha256 line"
    if recorded[0] == h.hexdigest():
        assert got is not None and got > 0
    else:
        assert got is None
