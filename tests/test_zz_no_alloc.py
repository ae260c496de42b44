"""kv_int4_paged_attention_noalloc: the paged attention for callers that cannot allocate device
memory (an engine that reserved all free memory for its KV cache, a plugin host that forbids
allocation after start-up, a decode loop that cannot take cudaMalloc's device-wide sync).  It keeps
its split-KV partials in the library's fixed device scratch array instead of a caller workspace.

The tests call the C entry point directly (ctypes, raw device pointers).  With the same segment
length the no-allocation call runs the same kernels as kv_int4_paged_attention, so its output must
be bit-identical to the regular entry point's; both are also checked against the oracle.  Two calls
in a row go over two different batches, the second with fewer split-KV segments than the first, so
the first call's partials are still in the scratch array when the second runs and must never be
read.  With segment_len 0 on the GQA decode batch's shapes (32 sequences up to 4096 tokens) the
library's usual choice needs more than the scratch array, so the call must raise the segment length
to the first multiple of 32 that fits.  The file collects last, so that a run stopping at the first
failure has run every other test first.
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
    from gpu_helpers import clear_status
    clear_status()


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


def _regular(wl, t, seg):
    import int4_token_head_kv_gb300 as kv
    return kv.kv_int4_paged_attention(t["q"], t["cache"], t["tables"], t["lens"], t["qsl"], wl.softmax_scale,
                                      t["signs"], max_query_len=wl.max_query_len, max_seq_len=wl.max_seq_len,
                                      out_dtype=torch.float32, segment_len=seg)


def _segments(wl, seg):
    return int(sum(-(-int(L) // seg) for L in wl.seq_lens))


def _check_against_oracle(wl, t, got, seqs=None):
    from gpu_helpers import assert_attention_close, oracle_attention, oracle_cache
    rows = None if seqs is None else np.concatenate(
        [np.arange(wl.token_start[b], wl.token_start[b + 1]) for b in seqs])
    ref = oracle_attention(wl, oracle_cache(wl, rows=rows), seqs=seqs)
    assert_attention_close(got, ref, wl.name)


def test_noalloc_matches_regular_entry_point_twice():
    from gpu_helpers import status
    import int4_token_head_kv_gb300 as kv
    f = _c_entry()
    dev = torch.device("cuda:0")
    seg = 256
    batches = [
        workloads.make_attention_workload("noalloc_a", [3000, 1500, 700, 64], [1, 1, 1, 1], 32, 8, 128, seed=21),
        workloads.make_attention_workload("noalloc_b", [2600, 90, 1777], [1, 1, 1], 32, 8, 128, seed=22),
    ]
    assert _segments(batches[1], seg) < _segments(batches[0], seg)   # stale partials stay behind
    for wl in batches:
        assert kv.kv_int4_attention_workspace_bytes(32, 8, 128, len(wl.seq_lens), wl.max_seq_len,
                                                    seg) > 0   # the scratch really is used
        t = _device_inputs(wl, dev)
        ref = _regular(wl, t, seg)
        out = torch.full(ref.shape, float("nan"), dtype=torch.float32, device=dev)
        assert _noalloc(f, wl, t, out, seg) == KV_INT4_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"{wl.name}: no-allocation output differs from the regular entry point"
        _check_against_oracle(wl, t, out)
    assert not any(status().values())


def _noalloc_auto_segment(kv, wl):
    """The segment length the no-allocation call picks for segment_len 0 (its documented rule)."""
    args = (wl.num_q_heads, wl.num_kv_heads, wl.head_size, len(wl.seq_lens), wl.max_seq_len)
    seg = kv.kv_int4_attention_segment_len(len(wl.seq_lens), wl.max_seq_len, 0)
    if kv.kv_int4_attention_workspace_bytes(*args, seg) <= SCRATCH_BYTES:
        return seg
    while seg < 4096:
        seg = min(4096, seg + 32)
        if kv.kv_int4_attention_workspace_bytes(*args, seg) <= SCRATCH_BYTES:
            return seg
    return None


def test_noalloc_auto_segment_fits_the_scratch_on_the_gqa_batch():
    from gpu_helpers import status
    import int4_token_head_kv_gb300 as kv
    f = _c_entry()
    dev = torch.device("cuda:0")
    wl = workloads.gqa_decode_batch()
    args = (wl.num_q_heads, wl.num_kv_heads, wl.head_size, len(wl.seq_lens), wl.max_seq_len)
    assert kv.kv_int4_attention_workspace_bytes(*args, 0) > SCRATCH_BYTES   # the usual choice would not fit
    seg = _noalloc_auto_segment(kv, wl)
    assert seg is not None and seg % 32 == 0 and seg > kv.kv_int4_attention_segment_len(len(wl.seq_lens),
                                                                                          wl.max_seq_len, 0)
    t = _device_inputs(wl, dev)
    ref = _regular(wl, t, seg)
    for _ in range(2):
        out = torch.full(ref.shape, float("nan"), dtype=torch.float32, device=dev)
        assert _noalloc(f, wl, t, out, 0) == KV_INT4_OK
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    _check_against_oracle(wl, t, out, seqs=[0, 9, 31])
    assert not any(status().values())


def test_noalloc_rejects_requests_beyond_its_scratch():
    import int4_token_head_kv_gb300 as kv
    f = _c_entry()
    dev = torch.device("cuda:0")
    wl = workloads.make_attention_workload("noalloc_big", [64], [1], 32, 8, 128, seed=23)
    t = _device_inputs(wl, dev)
    out = torch.empty((1, 32, 128), dtype=torch.float32, device=dev)
    # 4096 sequences x 2048 segments of 16 tokens would need far more than the scratch, and so
    # would 4096 sequences of 32768 tokens in segments of 4096 (the largest automatic choice)
    for seg in (16, 0):
        need = kv.kv_int4_attention_workspace_bytes(32, 8, 128, 4096, 32768, seg if seg else 4096)
        assert need > SCRATCH_BYTES
        rc = f(t["q"].data_ptr(), 1, 4096, 32, t["cache"].data_ptr(), wl.num_blocks, 8, 128, 16,
               t["tables"].data_ptr(), 1, t["lens"].data_ptr(), t["qsl"].data_ptr(), 4096, 1, 32768,
               wl.softmax_scale, t["signs"].data_ptr(), seg, out.data_ptr(), 2, torch.cuda.current_stream().cuda_stream)
        assert rc == KV_INT4_EWORKSPACE


def test_python_binding_matches_regular_entry_point():
    # the binding's kv_int4_paged_attention_noalloc marshals the same call: bit-identical output
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev, gpu_attention, gpu_cache, gpu_write
    wl = workloads.make_attention_workload("noalloc_py", [900, 40, 2500], [1, 1, 1], 16, 4, 128, seed=23,
                                           segment_len=256)
    cache = gpu_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_size)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    ref = gpu_attention(wl, cache, out_dtype=torch.float32, segment_len=256)
    got = kv.kv_int4_paged_attention_noalloc(
        wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
        torch.from_numpy(wl.seq_lens).to(dev()), torch.from_numpy(wl.query_start_loc).to(dev()),
        wl.softmax_scale, torch.from_numpy(wl.signs).to(dev()), max_query_len=wl.max_query_len,
        max_seq_len=wl.max_seq_len, out_dtype=torch.float32, segment_len=256)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)


def test_python_binding_with_options_matches_regular_entry_point():
    # every option (window, softcap, ALiBi, qq_bias) through kv_int4_paged_attention_noalloc_ex on a
    # batch of decodes and a prefill chunk: bit-identical to kv_int4_paged_attention_ex
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev, gpu_cache, gpu_write, status
    wl = workloads.make_attention_workload("noalloc_opts", [900, 40, 2500, 300], [1, 1, 1, 120], 16, 4, 128,
                                           seed=24, segment_len=256)
    wl.query = (wl.query.float() * 3.0).to(wl.query.dtype)
    cache = gpu_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_size)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    r = np.random.default_rng(24)
    opts = dict(window_left=500, softcap=10.0,
                alibi_slopes=torch.tensor([0.02 * (i + 1) for i in range(16)], dtype=torch.float32, device=dev()),
                qq_bias=torch.from_numpy(r.uniform(-1.5, 1.5, (120, 128)).astype(np.float32)).to(dev()))
    args = (wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
            torch.from_numpy(wl.seq_lens).to(dev()), torch.from_numpy(wl.query_start_loc).to(dev()),
            wl.softmax_scale, torch.from_numpy(wl.signs).to(dev()))
    kw = dict(max_query_len=wl.max_query_len, max_seq_len=wl.max_seq_len, out_dtype=torch.float32, segment_len=256)
    ref = kv.kv_int4_paged_attention(*args, **kw, **opts)
    got = kv.kv_int4_paged_attention_noalloc(*args, **kw, **opts)
    plain = kv.kv_int4_paged_attention_noalloc(*args, **kw)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
    assert not torch.equal(plain, ref)   # the options reached the kernels
    st = status()
    assert not any(st.values()), st
