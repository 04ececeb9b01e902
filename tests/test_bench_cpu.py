"""Host-side accounting of the benchmark (no GPU): the algorithmic bytes a rejection needs, the
source hash that keys the recorded DRAM traffic, and the traffic lookup."""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.join(os.path.dirname(__file__), ".."))
import bench  # noqa: E402


def test_q_bytes_per_rejection():
    w = dict(V=128256, top_k=None)
    assert bench.q_bytes_per_rejection(w, False) == 128256 * 4
    assert bench.q_bytes_per_rejection(w, True) == 128256 * 4  # no top-k: the whole row
    w["top_k"] = np.full(8, 50, dtype=np.int32)
    assert bench.q_bytes_per_rejection(w, True) == 32 * 50  # a sector per kept token
    assert bench.q_bytes_per_rejection(w, False) == 128256 * 4  # the full pass reads whole rows
    w["top_k"] = np.array([50, 0, 50], dtype=np.int32)  # a request without top-k keeps all
    assert bench.q_bytes_per_rejection(w, True) == 128256 * 4
    w["top_k"] = np.full(4, 1000, dtype=np.int32)  # too many kept tokens for the list
    assert bench.q_bytes_per_rejection(w, True) == 128256 * 4


def test_source_hash_ignores_comments_and_layout(tmp_path, monkeypatch):
    common = tmp_path / "common.cuh"
    source = tmp_path / "spec_reject.cu"
    common.write_text("int a;  // one\n")
    source.write_text("/* block */ int b = 1;\n// K1F: top-k / top-p cut\nint c;\n")
    monkeypatch.setattr(bench, "KERNEL_COMMON", str(common))
    monkeypatch.setattr(bench, "KERNEL_SOURCE", str(source))
    h0, f0 = bench.source_sha(), bench.source_sha(full=True)
    common.write_text("int  a;\n\n// another comment\n")
    source.write_text("int b = 1;  /* x */\n// K1F: top-k / top-p cut\nint c;   // y\n")
    assert bench.source_sha() == h0 and bench.source_sha(full=True) == f0
    source.write_text("int b = 1;\n// K1F: top-k / top-p cut\nint d;\n")  # code after the cut point
    assert bench.source_sha() == h0 and bench.source_sha(full=True) != f0
    common.write_text("int a2;\n")
    assert bench.source_sha() != h0


def test_traffic_reported_only_for_the_recorded_source(tmp_path, monkeypatch):
    rec = {"lazy": {"source_sha": bench.source_sha(full=True), "dram_bytes_per_launch": {"large-128": 123}},
           "rowstats": {"source_sha": "0" * 16, "dram_bytes_per_launch": {"probabilistic": 456}}}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.traffic_lazy_for("large-128") == 123
    assert bench.traffic_lazy_for("large-512") is None
    assert bench.traffic_for("probabilistic") is None  # taken on another source


def test_committed_traffic_record_is_consistent():
    with open(bench.TRAFFIC_FILE) as f:
        rec = json.load(f)["lazy"]
    dram, alg = rec["dram_bytes_per_launch"], rec["algorithmic_bytes_per_launch"]
    assert set(dram) == set(alg)
    for k in dram:  # DRAM bytes at or a little above the algorithmic bytes
        assert 1.0 <= dram[k] / alg[k] < 1.2, k
