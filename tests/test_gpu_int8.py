"""GPU parity of kv_int8_write (the INT8 per-(token, head) comparator) against its oracle: the
whole cache, byte for byte, on the page-test shapes, the write-throughput workload at full size,
skipped and out-of-range slots, and quantiser edge cases (zero, constant, tiny, huge, exact ties)."""
import numpy as np
import pytest
import torch

from oracle import int8 as o8
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gpu_helpers import clear_status
    clear_status()


def _check(wl, fill=0):
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev
    H, d = wl.num_kv_heads, wl.head_size
    ref = np.full(o8.cache_shape(wl.num_blocks, wl.block_size, H, d), fill, np.uint8)
    bad = o8.write(wl.key, wl.value, wl.slot_mapping, ref)
    cache = torch.full(kv.kv_int8_cache_shape(wl.num_blocks, wl.block_size, H, d), fill, dtype=torch.uint8,
                       device=dev())
    kv.kv_int8_write(wl.key.to(dev()).contiguous(), wl.value.to(dev()).contiguous(),
                     torch.from_numpy(np.ascontiguousarray(wl.slot_mapping)).to(dev()), cache)
    got = cache.cpu().numpy()
    if not np.array_equal(got, ref):
        diff = np.argwhere(got != ref)
        raise AssertionError(f"{len(diff)} cache bytes differ; first at {diff[0].tolist()}: "
                             f"gpu {got[tuple(diff[0])]:#x} oracle {ref[tuple(diff[0])]:#x}")
    return bad


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("head_size", [64, 128])
@pytest.mark.parametrize("num_heads", [1, 2, 8])
@pytest.mark.parametrize("num_tokens", [1, 7, 42])
def test_int8_write_page_shapes_bit_exact(num_tokens, num_heads, head_size, dtype):
    wl = workloads.random_write(num_tokens, num_heads, head_size, dtype=dtype, seed=5)
    _check(wl, fill=0xA5)


@pytest.mark.parametrize("num_heads", [3, 16, 64])
def test_int8_write_other_head_counts(num_heads):
    wl = workloads.random_write(37, num_heads, 128, seed=60 + num_heads)
    _check(wl, fill=0x5A)


def test_int8_write_throughput_workload_full_size():
    _check(workloads.write_throughput())


def test_int8_skipped_and_out_of_range_slots():
    from gpu_helpers import status
    wl = workloads.random_write(40, 8, 128, seed=6, num_blocks=4)
    wl.slot_mapping[3] = wl.num_blocks * wl.block_size
    wl.slot_mapping[9] = 10 ** 9
    wl.slot_mapping[11] = -1
    assert _check(wl, fill=0x33) == 2
    assert status()["slot_out_of_range"] == 2


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_int8_edge_vectors(dtype):
    d = 128
    rng = np.random.default_rng(7)
    rows = [np.zeros(d), np.full(d, 3.0), np.full(d, -1e-3), rng.standard_normal(d) * 1e-6,
            rng.standard_normal(d) * (1e4 if dtype == torch.float16 else 1e30),
            np.concatenate([[127.0], rng.integers(-126, 126, d - 1) + 0.5]),   # exact .5 ties at scale 1
            np.concatenate([[-254.0], np.arange(-63, 64)]),                       # scale 2: every x.5 tie
            np.eye(d)[5] * -9.0]
    x = np.stack(rows).astype(np.float32)
    T = x.shape[0]
    wl = workloads.random_write(T, 1, d, dtype=dtype, seed=8)
    wl.key = torch.from_numpy(x[:, None, :]).to(dtype)
    wl.value = torch.from_numpy(-x[:, None, :]).to(dtype)
    _check(wl, fill=0x11)


# ---------------------------------------------------------------------------- INT8 decode attention
# kv_int8_paged_attention against oracle/int8.py's paged_attention over the oracle's own INT8 cache
# (checked byte-identical to the GPU's first): |gpu - oracle| <= 2e-3 + 1e-2 |oracle|, as for INT4.

def _int8_attention_case(wl, seqs=None, kv_heads=None, segment_len=None, out_dtype=torch.float32):
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import assert_attention_close, dev, status
    H, d = wl.num_kv_heads, wl.head_size
    cache = torch.zeros(kv.kv_int8_cache_shape(wl.num_blocks, wl.block_size, H, d), dtype=torch.uint8, device=dev())
    rows = None if seqs is None else np.concatenate([np.arange(wl.token_start[b], wl.token_start[b + 1]) for b in seqs])
    k, v, s = (wl.key, wl.value, wl.slot_mapping) if rows is None else (wl.key[rows], wl.value[rows], wl.slot_mapping[rows])
    kv.kv_int8_write(k.to(dev()).contiguous(), v.to(dev()).contiguous(),
                     torch.from_numpy(np.ascontiguousarray(s)).to(dev()), cache)
    seg = wl.segment_len if segment_len is None else segment_len
    out = kv.kv_int8_paged_attention(
        wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
        torch.from_numpy(wl.seq_lens).to(dev()), torch.from_numpy(wl.query_start_loc).to(dev()),
        wl.softmax_scale, max_query_len=wl.max_query_len, max_seq_len=wl.max_seq_len, out_dtype=out_dtype,
        segment_len=seg)
    torch.cuda.synchronize()
    ref_cache = np.zeros(o8.cache_shape(wl.num_blocks, wl.block_size, H, d), np.uint8)
    o8.write(k, v, s, ref_cache)
    got = cache.cpu().numpy()
    if seqs is None:
        assert np.array_equal(got, ref_cache), "GPU INT8 cache differs from the oracle's"
    ref = o8.paged_attention(wl.query, ref_cache, wl.block_tables, wl.seq_lens, wl.query_start_loc, wl.softmax_scale,
                             seqs=seqs, kv_heads=kv_heads)
    err = assert_attention_close(out, ref, wl.name + " (int8)")
    st = status()
    assert not any(st.values()), st
    return err


@pytest.mark.parametrize("H,G,d", [(1, 1, 64), (2, 4, 128), (4, 2, 64), (8, 8, 128), (8, 1, 64), (1, 8, 128)])
def test_int8_decode_head_groupings(H, G, d):
    # ragged contexts across block and segment edges
    wl = workloads.make_attention_workload("int8_groupings", [1, 15, 16, 17, 300, 64, 1024, 77], [1] * 8, H * G, H, d,
                                           seed=11, segment_len=64)
    _int8_attention_case(wl)


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_int8_decode_output_dtypes(out_dtype):
    wl = workloads.tiny_write_decode()
    _int8_attention_case(wl, out_dtype=out_dtype)


def test_int8_decode_gqa_batch_full_size():
    _int8_attention_case(workloads.gqa_decode_batch(), segment_len=0)


def test_int8_decode_long_context_full_size_sampled():
    # at the library's segment length (what the benchmark times)
    wl = workloads.long_context_decode()
    _int8_attention_case(wl, seqs=[0, 7], kv_heads=[0, 5], segment_len=0)


def test_int8_decode_mixed_magnitudes():
    wl = workloads.make_attention_workload("int8_magnitudes", [500, 33, 2000], [1, 1, 1], 16, 4, 128, seed=12,
                                           segment_len=256)
    scale = torch.ones(wl.key.shape[0], 1, 1)
    scale[::7] = 300.0
    scale[3::11] = 1e-3
    wl.key = (wl.key.float() * scale).to(wl.key.dtype)
    wl.value = (wl.value.float() * scale).to(wl.value.dtype)
    _int8_attention_case(wl)


def test_int8_attention_rejects_prefill_chunks():
    import int4_token_head_kv_gb300 as kv
    wl = workloads.make_attention_workload("int8_prefill", [64], [8], 4, 4, 64, seed=13)
    from gpu_helpers import dev
    cache = torch.zeros(kv.kv_int8_cache_shape(wl.num_blocks, 16, 4, 64), dtype=torch.uint8, device=dev())
    with pytest.raises(RuntimeError):
        kv.kv_int8_paged_attention(wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
                                   torch.from_numpy(wl.seq_lens).to(dev()),
                                   torch.from_numpy(wl.query_start_loc).to(dev()), wl.softmax_scale,
                                   max_query_len=8, max_seq_len=64)


def test_int8_empty_context_gives_zeros():
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev
    d = 128
    cache = torch.zeros(kv.kv_int8_cache_shape(4, 16, 2, d), dtype=torch.uint8, device=dev())
    q = torch.randn(2, 4, d, device=dev(), dtype=torch.bfloat16)
    out = kv.kv_int8_paged_attention(q, cache, torch.zeros(2, 1, dtype=torch.int32, device=dev()),
                                     torch.tensor([0, 0], dtype=torch.int32, device=dev()),
                                     torch.tensor([0, 1, 2], dtype=torch.int32, device=dev()), d ** -0.5,
                                     max_query_len=1, max_seq_len=0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
