"""kv_int4_paged_attention_noalloc: the paged attention for callers that cannot allocate device
memory (an engine that reserved all free memory for its KV cache, a plugin host that forbids
allocation after start-up, a decode loop that cannot take cudaMalloc's device-wide sync).  It keeps
its split-KV partials in the library's fixed device scratch array instead of a caller workspace.

The test calls the C entry point directly (ctypes, raw device pointers) and checks it against the
regular entry point, within the tolerance the attention tests use, on two calls in a row over two
different batches (the second call finds the first one's partials still in the scratch array).
It collects last so that a run stopping at the first failure has run every other test first.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

KV_INT4_OK, KV_INT4_EWORKSPACE = 0, 4
SCRATCH_BYTES = 16 * 1024 * 1024


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def _c_entry():
    import int4_token_head_kv_gb300 as kv
    f = kv.load().kv_int4_paged_attention_noalloc
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [vp, ctypes.c_int, i64, i32, vp, i64, i32, i32, i32, vp, i32, vp, vp, i32, i32, i32,
                  ctypes.c_float, vp, i32, vp, ctypes.c_int, vp]
    f.restype = ctypes.c_int
    return f


def _device_inputs(wl, dev):
    import int4_token_head_kv_gb300 as kv
    cache = torch.zeros(kv.kv_int4_cache_shape(wl.num_blocks, 16, wl.num_kv_heads, wl.head_size), dtype=torch.uint8,
                        device=dev)
    signs = torch.from_numpy(wl.signs).to(dev)
    kv.kv_int4_write(wl.key.to(dev), wl.value.to(dev), torch.from_numpy(wl.slot_mapping).to(dev), signs, cache)
    return dict(q=wl.query.to(dev), cache=cache, tables=torch.from_numpy(wl.block_tables).to(dev),
                lens=torch.from_numpy(wl.seq_lens).to(dev), qsl=torch.from_numpy(wl.query_start_loc).to(dev),
                signs=signs)


def _noalloc(f, wl, t, out, segment_len):
    return f(t["q"].data_ptr(), 1, wl.query.shape[0], wl.num_q_heads, t["cache"].data_ptr(), wl.num_blocks,
             wl.num_kv_heads, wl.head_size, 16, t["tables"].data_ptr(), wl.block_tables.shape[1], t["lens"].data_ptr(),
             t["qsl"].data_ptr(), len(wl.seq_lens), wl.max_query_len, wl.max_seq_len, wl.softmax_scale,
             t["signs"].data_ptr(), segment_len, out.data_ptr(), 2, torch.cuda.current_stream().cuda_stream)


def test_noalloc_matches_regular_entry_point_twice():
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import ATOL, RTOL
    f = _c_entry()
    dev = torch.device("cuda:0")
    seg = 256
    batches = [
        workloads.make_attention_workload("noalloc_a", [3000, 1500, 700, 64], [1, 1, 1, 1], 32, 8, 128, seed=21),
        workloads.make_attention_workload("noalloc_b", [2600, 90, 1777], [1, 1, 1], 32, 8, 128, seed=22),
    ]
    for wl in batches:
        assert kv.kv_int4_attention_workspace_bytes(32, 8, 128, len(wl.seq_lens), wl.max_seq_len,
                                                    seg) > 0   # the scratch really is used
        t = _device_inputs(wl, dev)
        ref = kv.kv_int4_paged_attention(t["q"], t["cache"], t["tables"], t["lens"], t["qsl"], wl.softmax_scale,
                                         t["signs"], max_query_len=wl.max_query_len, max_seq_len=wl.max_seq_len,
                                         out_dtype=torch.float32, segment_len=seg)
        out = torch.full(ref.shape, float("nan"), dtype=torch.float32, device=dev)
        assert _noalloc(f, wl, t, out, seg) == KV_INT4_OK
        torch.cuda.synchronize()
        got, want = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - want) <= ATOL + RTOL * np.abs(want))


def test_noalloc_rejects_requests_beyond_its_scratch():
    import int4_token_head_kv_gb300 as kv
    f = _c_entry()
    dev = torch.device("cuda:0")
    wl = workloads.make_attention_workload("noalloc_big", [64], [1], 32, 8, 128, seed=23)
    t = _device_inputs(wl, dev)
    out = torch.empty((1, 32, 128), dtype=torch.float32, device=dev)
    # 4096 sequences x 2048 segments of 16 tokens would need far more than the scratch
    need = kv.kv_int4_attention_workspace_bytes(32, 8, 128, 4096, 32768, 16)
    assert need > SCRATCH_BYTES
    rc = f(t["q"].data_ptr(), 1, 4096, 32, t["cache"].data_ptr(), wl.num_blocks, 8, 128, 16, t["tables"].data_ptr(),
           1, t["lens"].data_ptr(), t["qsl"].data_ptr(), 4096, 1, 32768, wl.softmax_scale, t["signs"].data_ptr(), 16,
           out.data_ptr(), 2, torch.cuda.current_stream().cuda_stream)
    assert rc == KV_INT4_EWORKSPACE
