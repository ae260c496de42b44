"""Host logic of bench.py's measurement record, on the CPU: a committed ncu traffic figure
(profiles/traffic.json) is reported only while the CUDA sources are the ones it was taken on, and
the committed figures were taken on the current sources."""
import json
import os
import shutil

import pytest

import bench

WORKLOADS = ("long_context_decode", "gqa_decode_batch", "mixed_prefill_decode", "write_throughput")


def test_traffic_figures_match_the_current_sources():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        table = json.load(f)
    for w in WORKLOADS:
        assert table[w]["sources_sha"] == bench.sources_sha(), w
        got = bench._traffic(w)
        assert isinstance(got, int) and got > 0, w


def test_traffic_is_withheld_for_other_sources(monkeypatch):
    monkeypatch.setattr(bench, "sources_sha", lambda: "0" * 16)
    for w in WORKLOADS:
        assert bench._traffic(w) is None
    assert bench._traffic("no_such_workload") is None


def test_sources_digest_covers_every_cuda_source(tmp_path, monkeypatch):
    src = tmp_path / "csrc"
    shutil.copytree(bench.CSRC, src)
    monkeypatch.setattr(bench, "CSRC", str(src))
    base = bench.sources_sha()
    assert base == bench.sources_sha()   # deterministic
    for name in sorted(os.listdir(src)):
        if not name.endswith((".cu", ".cuh", ".h")):
            continue
        p = src / name
        text = p.read_bytes()
        p.write_bytes(text + b"\n")
        assert bench.sources_sha() != base, name
        p.write_bytes(text)
    assert bench.sources_sha() == base
    (src / "notes.txt").write_text("not a source")
    assert bench.sources_sha() == base
