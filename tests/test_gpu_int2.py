"""GPU parity of the INT2 Lloyd-Max mode against its oracle (oracle/int2.py): kv_int2_write byte for
byte on the page-test shapes, the write-throughput workload at full size, skipped and out-of-range
slots and quantiser edge cases; kv_int2_paged_attention against the oracle's fp64 attention over
the oracle's own INT2 cache (checked byte-identical to the GPU's first) within
|gpu - oracle| <= 2e-3 + 1e-2 |oracle|, as for INT4.  The decode walker holds the centroids as fp16
(relative error at most 2.3e-4 each), well inside that bar."""
import numpy as np
import pytest
import torch

from oracle import int2 as o2
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gpu_helpers import clear_status
    clear_status()


def _write_both(key, value, slots, signs, num_blocks, block_size, H, d, fill=0):
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev
    ref = np.full(o2.cache_shape(num_blocks, block_size, H, d), fill, np.uint8)
    bad = o2.write(key, value, slots, signs, ref)
    cache = torch.full(kv.kv_int2_cache_shape(num_blocks, block_size, H, d), fill, dtype=torch.uint8, device=dev())
    kv.kv_int2_write(key.to(dev()).contiguous(), value.to(dev()).contiguous(),
                     torch.from_numpy(np.ascontiguousarray(slots)).to(dev()), torch.from_numpy(signs).to(dev()), cache)
    return cache, ref, bad


def _check(wl, fill=0):
    cache, ref, bad = _write_both(wl.key, wl.value, wl.slot_mapping, wl.signs, wl.num_blocks, wl.block_size,
                                  wl.num_kv_heads, wl.head_size, fill)
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
def test_int2_write_page_shapes_bit_exact(num_tokens, num_heads, head_size, dtype):
    wl = workloads.random_write(num_tokens, num_heads, head_size, dtype=dtype, seed=25)
    _check(wl, fill=0xA5)


@pytest.mark.parametrize("num_heads", [3, 16, 64])
def test_int2_write_other_head_counts(num_heads):
    wl = workloads.random_write(37, num_heads, 128, seed=60 + num_heads)
    _check(wl, fill=0x5A)


def test_int2_write_throughput_workload_full_size():
    _check(workloads.write_throughput())


def test_int2_skipped_and_out_of_range_slots():
    from gpu_helpers import status
    wl = workloads.random_write(40, 8, 128, seed=26, num_blocks=4)
    wl.slot_mapping[3] = wl.num_blocks * wl.block_size
    wl.slot_mapping[9] = 10 ** 9
    wl.slot_mapping[11] = -1
    assert _check(wl, fill=0x33) == 2
    assert status()["slot_out_of_range"] == 2


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_int2_edge_vectors(dtype):
    d = 128
    rng = np.random.default_rng(27)
    big = 1e4 if dtype == torch.float16 else 1e30
    rows = [np.zeros(d), -np.zeros(d), np.full(d, 3.0), np.full(d, -1e-3), rng.standard_normal(d) * 1e-6,
            rng.standard_normal(d) * big, np.eye(d)[5] * -9.0, np.eye(d)[0] + np.eye(d)[64],
            rng.integers(-3, 4, d).astype(np.float64), np.where(np.arange(d) % 2, 1.0, -1.0)]
    x = np.stack(rows).astype(np.float32)
    T = x.shape[0]
    wl = workloads.random_write(T, 1, d, dtype=dtype, seed=28)
    wl.key = torch.from_numpy(x[:, None, :]).to(dtype)
    wl.value = torch.from_numpy(-x[:, None, :]).to(dtype)
    _check(wl, fill=0x11)


# ---------------------------------------------------------------------------- INT2 decode attention

def _int2_attention_case(wl, seqs=None, kv_heads=None, segment_len=None, out_dtype=torch.float32):
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import assert_attention_close, dev, status
    H, d = wl.num_kv_heads, wl.head_size
    rows = None if seqs is None else np.concatenate([np.arange(wl.token_start[b], wl.token_start[b + 1]) for b in seqs])
    k, v, s = (wl.key, wl.value, wl.slot_mapping) if rows is None else (wl.key[rows], wl.value[rows], wl.slot_mapping[rows])
    cache, ref_cache, _ = _write_both(k, v, s, wl.signs, wl.num_blocks, wl.block_size, H, d)
    seg = wl.segment_len if segment_len is None else segment_len
    out = kv.kv_int2_paged_attention(
        wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
        torch.from_numpy(wl.seq_lens).to(dev()), torch.from_numpy(wl.query_start_loc).to(dev()),
        wl.softmax_scale, torch.from_numpy(wl.signs).to(dev()), max_query_len=wl.max_query_len,
        max_seq_len=wl.max_seq_len, out_dtype=out_dtype, segment_len=seg)
    torch.cuda.synchronize()
    if seqs is None:
        assert np.array_equal(cache.cpu().numpy(), ref_cache), "GPU INT2 cache differs from the oracle's"
    ref = o2.paged_attention(wl.query, ref_cache, wl.block_tables, wl.seq_lens, wl.query_start_loc, wl.softmax_scale,
                             wl.signs, seqs=seqs, kv_heads=kv_heads)
    err = assert_attention_close(out, ref, wl.name + " (int2)")
    st = status()
    assert not any(st.values()), st
    return err


@pytest.mark.parametrize("H,G,d", [(1, 1, 64), (2, 4, 128), (4, 2, 64), (8, 8, 128), (8, 1, 64), (1, 8, 128),
                                   (8, 4, 128)])
def test_int2_decode_head_groupings(H, G, d):
    # ragged contexts across block and segment edges
    wl = workloads.make_attention_workload("int2_groupings", [1, 15, 16, 17, 300, 64, 1024, 77], [1] * 8, H * G, H, d,
                                           seed=31, segment_len=64)
    _int2_attention_case(wl)


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_int2_decode_output_dtypes(out_dtype):
    _int2_attention_case(workloads.tiny_write_decode(), out_dtype=out_dtype)


def test_int2_decode_gqa_batch_full_size():
    _int2_attention_case(workloads.gqa_decode_batch(), segment_len=0)


def test_int2_decode_long_context_full_size_sampled():
    # at the library's segment length (what the benchmark times)
    wl = workloads.long_context_decode()
    _int2_attention_case(wl, seqs=[0, 7], kv_heads=[0, 5], segment_len=0)


def test_int2_decode_mixed_magnitudes():
    wl = workloads.make_attention_workload("int2_magnitudes", [500, 33, 2000], [1, 1, 1], 16, 4, 128, seed=32,
                                           segment_len=256)
    scale = torch.ones(wl.key.shape[0], 1, 1)
    scale[::7] = 300.0
    scale[3::11] = 1e-3
    wl.key = (wl.key.float() * scale).to(wl.key.dtype)
    wl.value = (wl.value.float() * scale).to(wl.value.dtype)
    _int2_attention_case(wl)


def test_int2_attention_rejects_prefill_chunks():
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev
    wl = workloads.make_attention_workload("int2_prefill", [64], [8], 4, 4, 64, seed=33)
    cache = torch.zeros(kv.kv_int2_cache_shape(wl.num_blocks, 16, 4, 64), dtype=torch.uint8, device=dev())
    with pytest.raises(RuntimeError):
        kv.kv_int2_paged_attention(wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
                                   torch.from_numpy(wl.seq_lens).to(dev()),
                                   torch.from_numpy(wl.query_start_loc).to(dev()), wl.softmax_scale,
                                   torch.from_numpy(wl.signs).to(dev()), max_query_len=8, max_seq_len=64)


def test_int2_empty_context_gives_zeros():
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev
    d = 128
    cache = torch.zeros(kv.kv_int2_cache_shape(4, 16, 2, d), dtype=torch.uint8, device=dev())
    q = torch.randn(2, 4, d, device=dev(), dtype=torch.bfloat16)
    signs = torch.ones(d, dtype=torch.float32, device=dev())
    out = kv.kv_int2_paged_attention(q, cache, torch.zeros(2, 1, dtype=torch.int32, device=dev()),
                                     torch.tensor([0, 0], dtype=torch.int32, device=dev()),
                                     torch.tensor([0, 1, 2], dtype=torch.int32, device=dev()), d ** -0.5, signs,
                                     max_query_len=1, max_seq_len=0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
