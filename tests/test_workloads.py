"""The five named workloads carry the shapes, dtypes and value distributions of the configurations
the library is measured on (tiny write + decode; GQA decode batch; long-context decode; write
throughput; mixed chunked prefill + decode).  The builders' arguments are checked without drawing
the full-size data, so that the benchmark and the parity tests cannot drift off them; the tiny
case is also built in full."""
import numpy as np
import pytest
import torch

import workloads


@pytest.fixture
def calls(monkeypatch):
    seen = []

    def record(name, seq_lens, query_lens, num_q_heads, num_kv_heads, head_size, **kw):
        seen.append(dict(name=name, seq_lens=np.asarray(seq_lens), query_lens=np.asarray(query_lens),
                         Hq=num_q_heads, H=num_kv_heads, d=head_size, **kw))
        return seen[-1]

    monkeypatch.setattr(workloads, "make_attention_workload", record)
    return seen


def test_tiny_write_decode_full():
    wl = workloads.tiny_write_decode()
    assert wl.seq_lens.tolist() == [42, 7] and wl.query_lens.tolist() == [1, 1]
    assert wl.key.shape == (49, 4, 64) and wl.key.dtype == torch.float16
    assert wl.query.shape == (2, 4, 64) and wl.num_q_heads == 4 and wl.block_size == 16
    # contiguous blocks: sequence 0 owns blocks 0..2, sequence 1 block 3
    assert wl.block_tables[0, :3].tolist() == [0, 1, 2] and wl.block_tables[1, 0] == 3


def test_gqa_decode_batch(calls):
    w = workloads.gqa_decode_batch()
    assert (w["Hq"], w["H"], w["d"]) == (32, 8, 128) and w["dtype"] == torch.bfloat16
    assert len(w["seq_lens"]) == 32 and w["seq_lens"].min() >= 512 and w["seq_lens"].max() <= 4096
    assert np.all(w["query_lens"] == 1)
    assert w["k_outlier_channels"] == 4 and w.get("block_order", "permuted") == "permuted"
    assert w.get("k_outlier_gain", 10.0) == 10.0


def test_long_context_decode(calls):
    w = workloads.long_context_decode()
    assert (w["Hq"], w["H"], w["d"]) == (64, 8, 128) and w["dtype"] == torch.bfloat16
    assert w["seq_lens"].tolist() == [131072] * 8 and w["query_lens"].tolist() == [1] * 8
    assert w["kv_dist"] == "student_t3" and w["segment_len"] == 4096


def test_mixed_prefill_decode(calls):
    w = workloads.mixed_prefill_decode()
    assert (w["Hq"], w["H"], w["d"]) == (32, 8, 128) and w["dtype"] == torch.bfloat16
    L, q = w["seq_lens"], w["query_lens"]
    assert len(L) == 64 and L[:4].tolist() == [4096] * 4 and q[:4].tolist() == [2048] * 4
    assert np.all(q[4:] == 1) and L[4:].min() >= 1 and L[4:].max() <= 32768


def test_write_throughput(monkeypatch):
    seen = []

    def fill(shape, dtype, seq, dist, row_scale=None):
        seen.append((shape, dtype, dist, row_scale))
        return torch.zeros(shape, dtype=dtype)

    monkeypatch.setattr(workloads, "_fill_random", fill)
    wl = workloads.write_throughput()
    assert [s[0] for s in seen] == [(65536, 8, 128)] * 2
    assert all(s[1] == torch.bfloat16 and s[2] == "normal" for s in seen)
    for *_, m in seen:   # per-token magnitudes 10^U(-2, 2)
        assert m.shape == (65536,) and m.min() >= 1e-2 * (1 - 1e-6) and m.max() <= 1e2 * (1 + 1e-6)
        assert m.min() < 2e-2 and m.max() > 50.0
    assert wl.num_blocks == 8192 and wl.block_size == 16
    slots = np.asarray(wl.slot_mapping)
    assert len(slots) == 65536 and len(np.unique(slots)) == 65536
    assert slots.min() >= 0 and slots.max() < 8192 * 16
