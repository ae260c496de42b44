"""Host logic of bench.py's measurement record, on the CPU: a committed ncu traffic figure
(profiles/traffic.json) is reported only while the CUDA sources are the ones it was taken on, the
committed figures were taken on the current sources, and the oracle timing behind the CPU baseline
counts the bytes of the sample it times."""
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


def _timing(*args):
    import subprocess
    import sys
    res = subprocess.run([sys.executable, "-m", "oracle.timing", *args], cwd=bench.ROOT, capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    return json.loads(res.stdout.strip().splitlines()[-1])


def test_oracle_timing_counts_the_bytes_of_its_sample():
    # the CPU baseline's unit: bytes of the sample / seconds.  Write: K and V in (bf16), the packed
    # rows out, the slot; decode: the packed K/V of the sampled contexts plus Q and O (bf16).
    import workloads
    w = _timing("write", "512", "0")
    assert w["units"] == 512 and w["seconds"] > 0
    assert w["bytes"] == 512 * (2 * 8 * 128 * 2 + 2 * 8 * (128 // 2 + 4) + 8)
    d = _timing("decode", "1", "0")
    L0 = int(workloads.gqa_decode_batch().seq_lens[0])
    assert d["units"] == 1 and d["seconds"] > 0
    assert d["bytes"] == L0 * 2 * 8 * 68 + 32 * 128 * 2 * 2
