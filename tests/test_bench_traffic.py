"""The bench's indexer traffic figure (roofline.traffic): the committed ncu
summary holds DRAM bytes per full-size launch; a run of another size scales
them by its algorithmic bytes, and a summary whose source hash no longer
matches the indexer's sources gives null rather than a stale number."""

from __future__ import annotations

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _summary(tmp_path, sha, per_launch, alg):
    d = tmp_path / "profiles"
    d.mkdir()
    (d / "indexer_traffic.json").write_text(
        json.dumps({"source_sha256": sha, "per_launch_bytes": per_launch, "algorithmic_bytes_per_launch": alg}))


def test_full_size_and_scaled_runs(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    _summary(tmp_path, "abc", {"paged": 1_100}, {"paged": 1_000})
    assert bench.indexer_traffic("paged", 1_000) == 1_100
    assert bench.indexer_traffic("paged", 500) == 550  # half the keys scanned, half the traffic
    assert bench.indexer_traffic("long_fp8", 1_000) is None  # no capture for this workload


def test_stale_or_incomplete_summary_gives_null(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "changed")
    _summary(tmp_path, "abc", {"paged": 1_100}, {"paged": 1_000})
    assert bench.indexer_traffic("paged", 1_000) is None


def test_summary_without_algorithmic_bytes_gives_null(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "abc")
    _summary(tmp_path, "abc", {"paged": 1_100}, {})
    assert bench.indexer_traffic("paged", 1_000) is None


def test_committed_summary_covers_its_workloads():
    with open(os.path.join(ROOT, "profiles", "indexer_traffic.json")) as f:
        j = json.load(f)
    for w, b in j["per_launch_bytes"].items():
        alg = j["algorithmic_bytes_per_launch"][w]
        assert 0.95 < b / alg < 1.05, f"{w}: traffic {b} against {alg} algorithmic bytes"
