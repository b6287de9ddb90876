"""Host-side logic of bench.py that needs no GPU: the decode traffic figure is
reported only while the kernel sources hash to the value recorded with it."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_source_sha_is_the_sha256_prefix_of_the_concatenation(tmp_path):
    a, b = tmp_path / "a.cu", tmp_path / "b.cuh"
    a.write_bytes(b"__global__ void k() {}\n")
    b.write_bytes(b"#pragma once\n")
    want = hashlib.sha256(b"__global__ void k() {}\n" + b"#pragma once\n").hexdigest()[:16]
    assert bench.source_sha([str(a), str(b)]) == want
    assert bench.source_sha([str(b), str(a)]) != want   # order matters


def _record(path, sha, traffic=1.23e8):
    path.write_text(json.dumps({"sources": list(bench.DECODE_SOURCES), "source_sha256_16": sha,
                                "traffic_bytes_per_launch": traffic}))


@pytest.fixture
def sources_sha():
    srcs = [os.path.join(bench.ROOT, "encoder_decoder_speech_gb300", "csrc", f) for f in bench.DECODE_SOURCES]
    return bench.source_sha(srcs)


def test_recorded_traffic_follows_the_source_hash(tmp_path, monkeypatch, sources_sha):
    rec = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(rec))
    _record(rec, sources_sha)
    assert bench.recorded_traffic() == pytest.approx(1.23e8)
    _record(rec, "0" * 16)                      # sources changed since the capture
    assert bench.recorded_traffic() is None


def test_recorded_traffic_without_a_record(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(tmp_path / "missing.json"))
    assert bench.recorded_traffic() is None
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(bad))
    assert bench.recorded_traffic() is None
