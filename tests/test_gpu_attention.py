"""GPU parity of kv_int4_paged_attention against the fp64 oracle.

Each case writes the same seeded K/V twice -- with the CUDA write kernel into the GPU cache and
with the oracle into its own cache -- checks that the caches are byte-identical, then compares the
GPU attention (fp32 output) with the oracle's attention over its own cache:
|gpu - oracle| <= 2e-3 + 1e-2 |oracle|.

Workloads: the five named ones (tiny write + decode, GQA decode batch, long-context decode,
mixed chunked prefill + decode; full size where the oracle is fast enough, otherwise at full size
on sampled sequences and kv heads plus a scaled-down copy checked everywhere), the pages' own
unified-attention shapes, every supported head grouping, and edge cases (single-token and empty
contexts, block-boundary lengths, a whole-sequence prefill chunk, mixed value magnitudes, invalid
block ids, segment / batch invariance, determinism).
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gpu_helpers import clear_status
    clear_status()


def _run_case(wl, out_dtype=torch.float32, segment_len=None, seqs=None, kv_heads=None, check_cache=True):
    from gpu_helpers import (assert_attention_close, gpu_attention, gpu_cache, gpu_write, oracle_attention,
                             oracle_cache, status)
    H, d = wl.num_kv_heads, wl.head_size
    cache = gpu_cache(wl.num_blocks, wl.block_size, H, d)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    out = gpu_attention(wl, cache, out_dtype=out_dtype, segment_len=segment_len)
    torch.cuda.synchronize()
    if seqs is None:
        ref_cache = oracle_cache(wl)
        if check_cache:
            assert np.array_equal(cache.cpu().numpy(), ref_cache), "GPU cache differs from the oracle's"
    else:
        rows = np.concatenate([np.arange(wl.token_start[b], wl.token_start[b + 1]) for b in seqs])
        ref_cache = oracle_cache(wl, rows=rows)
        got = cache.cpu().numpy()
        for b in seqs:
            blocks = wl.block_tables[b, : (int(wl.seq_lens[b]) + 15) // 16]
            assert np.array_equal(got[blocks], ref_cache[blocks]), f"cache blocks of sequence {b} differ"
    ref = oracle_attention(wl, ref_cache, seqs=seqs, kv_heads=kv_heads)
    err = assert_attention_close(out, ref, wl.name)
    st = status()
    assert not any(st.values()), st
    return out, err


@pytest.mark.parametrize("G", [1, 4, 8])
def test_prefill_chunks_among_many_decodes(G):
    # a few ragged prefill chunks scattered through a large decode batch: the prefill grid covers the
    # batch's query tiles, found through the walker's per-sequence tile index, not every sequence
    r = np.random.default_rng(40 + G)
    n = 150
    qlens = np.ones(n, dtype=np.int64)
    qlens[[3, 77, 149]] = [100, 33, 257]
    qlens[120] = 0 if G == 4 else 1     # an empty query range in the middle
    lens = r.integers(1, 300, n)
    lens = np.maximum(lens, qlens + r.integers(0, 40, n) * (qlens > 1))
    wl = workloads.make_attention_workload("pf_scatter", lens.tolist(), qlens.tolist(), 2 * G, 2, 128, seed=40 + G,
                                           segment_len=64)
    _run_case(wl)


def test_tiny_write_decode():
    wl = workloads.tiny_write_decode()
    _run_case(wl)


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_tiny_output_dtypes(out_dtype):
    wl = workloads.tiny_write_decode()
    _run_case(wl, out_dtype=out_dtype)


@pytest.mark.parametrize("seq_lens", [[128], [64, 32]])
def test_pages_unified_attention_shapes(seq_lens):
    # 1 query per sequence, 4 q / 4 kv heads, head 128, block 16, 2048-block cache
    need = sum((L + 15) // 16 for L in seq_lens)
    wl = workloads.make_attention_workload("pages_shape", seq_lens, [1] * len(seq_lens), 4, 4, 128,
                                           extra_blocks=2048 - need, seed=0)
    _run_case(wl)


def test_gqa_decode_batch_full_size():
    wl = workloads.gqa_decode_batch()
    _run_case(wl)


def test_long_context_decode_scaled():
    wl = workloads.long_context_decode(num_seqs=2, seq_len=20000, segment_len=4096)
    _run_case(wl)


@pytest.mark.parametrize("segment_len", [4096, 0])
def test_long_context_decode_full_size_sampled(segment_len):
    # the workload's own segments of 4096, and the library's choice (what the benchmark times)
    wl = workloads.long_context_decode()
    _run_case(wl, segment_len=segment_len, seqs=[0, 7], kv_heads=[0, 5])


def test_mixed_prefill_decode_scaled():
    wl = workloads.make_attention_workload("mixed_scaled", [300, 64, 1, 17, 700, 3000, 5000],
                                           [200, 64, 1, 1, 1, 1, 1], 32, 8, 128, seed=3, segment_len=1024)
    _run_case(wl)


def test_mixed_prefill_decode_full_size_sampled():
    # at the library's segment length (what the benchmark times): every prefill sequence, the
    # longest and shortest decode contexts and a few others
    wl = workloads.mixed_prefill_decode()
    assert wl.segment_len == 0
    dec = np.arange(4, len(wl.seq_lens))
    pick = [int(dec[np.argmax(wl.seq_lens[dec])]), int(dec[np.argmin(wl.seq_lens[dec])]), 4, 30, 63]
    _run_case(wl, seqs=sorted(set([0, 1, 2, 3] + pick)), kv_heads=[0, 3, 7])


@pytest.mark.parametrize("H,G,d", [(1, 1, 64), (2, 4, 128), (4, 2, 64), (8, 8, 128), (1, 8, 128), (8, 1, 64),
                                   (4, 4, 128), (2, 2, 64)])
def test_head_groupings(H, G, d):
    wl = workloads.make_attention_workload(f"grp{H}x{G}d{d}", [1, 15, 16, 17, 250, 90], [1, 1, 1, 1, 1, 37],
                                           H * G, H, d, dtype=torch.float16 if d == 64 else torch.bfloat16,
                                           seed=H * 100 + G, segment_len=64)
    _run_case(wl)


@pytest.mark.parametrize("segment_len", [16, 64, 256, 0])
def test_segment_lengths(segment_len):
    wl = workloads.make_attention_workload("segs", [1000, 333, 2048], [1, 1, 1], 32, 8, 128, seed=5)
    _run_case(wl, segment_len=segment_len)


def test_segment_longer_than_the_staged_block_table():
    # one 600-block segment: the walker stages the first 256 block ids in shared memory and looks
    # the rest up in the block table as it goes
    wl = workloads.make_attention_workload("bigseg", [9600, 700], [1, 1], 16, 4, 128, seed=12)
    _run_case(wl, segment_len=9600)


def test_units_longer_than_a_cta_share():
    # 6 x 5000 tokens in segments of 2048: 18 units of up to 128 blocks over 18 CTAs whose shares
    # are about 104 blocks, so most units straddle a share boundary (some two); each unit belongs to
    # the share its first block falls in
    wl = workloads.make_attention_workload("strad", [5000, 4999, 4097, 5000, 2049, 5000], [1] * 6, 32, 8, 128,
                                           seed=14)
    out, _ = _run_case(wl, segment_len=2048)
    from gpu_helpers import gpu_attention, gpu_cache, gpu_write
    cache = gpu_cache(wl.num_blocks, 16, 8, 128)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    for _ in range(3):   # repeated calls give the same bits
        assert torch.equal(gpu_attention(wl, cache, segment_len=2048), out)


def test_many_short_sequences_per_cta():
    # 3000 one-block decode sequences of 1..16 tokens: each walker CTA runs about ten sequences,
    # cycling its rotated-query buffers
    r = np.random.default_rng(13)
    lens = r.integers(1, 17, 3000).tolist()
    wl = workloads.make_attention_workload("short", lens, [1] * 3000, 8, 2, 64, seed=13)
    _run_case(wl, segment_len=16, seqs=list(range(0, 3000, 37)))


def test_segment_split_changes_only_rounding():
    from gpu_helpers import gpu_attention, gpu_cache, gpu_write
    wl = workloads.make_attention_workload("segs", [3000], [1], 32, 8, 128, seed=6)
    cache = gpu_cache(wl.num_blocks, 16, 8, 128)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    a = gpu_attention(wl, cache, segment_len=16 * 1024)
    b = gpu_attention(wl, cache, segment_len=128)
    torch.testing.assert_close(a, b, atol=2e-4, rtol=2e-3)


def test_batch_invariance_and_determinism():
    from gpu_helpers import gpu_attention, gpu_cache, gpu_write
    big = workloads.make_attention_workload("batch", [700, 1500, 90, 2600], [1, 1, 1, 1], 32, 8, 128, seed=7,
                                            segment_len=512)
    cache = gpu_cache(big.num_blocks, 16, 8, 128)
    gpu_write(big.key, big.value, big.slot_mapping, big.signs, cache)
    out1 = gpu_attention(big, cache)
    out2 = gpu_attention(big, cache)
    assert torch.equal(out1, out2)
    # sequence 1 alone, reading the same cache blocks
    solo = workloads.make_attention_workload("solo", [1500], [1], 32, 8, 128, seed=7, segment_len=512)
    solo.block_tables = big.block_tables[1:2].copy()
    solo.query = big.query[1:2].clone()
    solo.num_blocks = big.num_blocks
    alone = gpu_attention(solo, cache)
    assert torch.equal(alone[0], out1[1])


def test_mixed_value_magnitudes():
    # per-token V magnitudes spanning 1e-3 .. 1e3: the fp16 attention weights carry V's scale
    wl = workloads.make_attention_workload("vmag", [2000, 37], [1, 1], 16, 4, 128, seed=8)
    r = np.random.default_rng(8)
    mags = torch.from_numpy((10.0 ** r.uniform(-3, 3, wl.value.shape[0])).astype(np.float32))
    wl.value = (wl.value.float() * mags[:, None, None]).to(wl.value.dtype)
    _run_case(wl, segment_len=512)


def test_whole_sequence_prefill_and_block_edges():
    wl = workloads.make_attention_workload("edges", [16, 33, 48, 129], [16, 2, 47, 1], 8, 2, 128, seed=9)
    _run_case(wl)


def test_empty_context_gives_zeros():
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev, gpu_cache
    d = 128
    cache = gpu_cache(4, 16, 2, d)
    q = torch.randn(2, 4, d, device=dev(), dtype=torch.bfloat16)
    out = kv.kv_int4_paged_attention(q, cache, torch.zeros(2, 1, dtype=torch.int32, device=dev()),
                                     torch.tensor([0, 0], dtype=torch.int32, device=dev()),
                                     torch.tensor([0, 1, 2], dtype=torch.int32, device=dev()), d ** -0.5,
                                     torch.from_numpy(workloads.splitmix64_signs(d)).to(dev()), max_query_len=1,
                                     max_seq_len=0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0


def test_invalid_block_ids_are_counted():
    from gpu_helpers import assert_attention_close, gpu_attention, gpu_cache, gpu_write, oracle_attention, \
        oracle_cache, status
    wl = workloads.make_attention_workload("badblk", [100, 60], [1, 1], 8, 2, 128, seed=10)
    cache = gpu_cache(wl.num_blocks, 16, 2, 128)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    tables = wl.block_tables.copy()
    wl.block_tables[0, 2] = wl.num_blocks + 5      # sequence 0 reads past the cache
    out = gpu_attention(wl, cache)
    torch.cuda.synchronize()
    assert status()["block_out_of_range"] >= 1
    wl.block_tables = tables
    ref = oracle_attention(wl, oracle_cache(wl), seqs=[1])   # the other sequence is unaffected
    assert_attention_close(out, ref, "unaffected sequence")


def test_contexts_longer_than_max_seq_len_are_clamped_alike():
    # one decode and one prefill sequence both longer than the max_seq_len the caller passes: both
    # paths cap the context at max_seq_len (counted as bad metadata), so each sees the first 150
    # tokens with its queries at the last positions of that window
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import assert_attention_close, dev, gpu_cache, gpu_write, oracle_attention, oracle_cache, \
        status
    wl = workloads.make_attention_workload("overlong", [300, 200], [1, 40], 16, 4, 128, seed=15)
    cache = gpu_cache(wl.num_blocks, 16, 4, 128)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    cap = 150
    out = kv.kv_int4_paged_attention(wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
                                     torch.from_numpy(wl.seq_lens).to(dev()),
                                     torch.from_numpy(wl.query_start_loc).to(dev()), wl.softmax_scale,
                                     torch.from_numpy(wl.signs).to(dev()), max_query_len=wl.max_query_len,
                                     max_seq_len=cap, out_dtype=torch.float32, segment_len=64)
    torch.cuda.synchronize()
    assert status()["bad_sequence"] >= 2
    ref_cache = oracle_cache(wl)
    wl.seq_lens = np.minimum(wl.seq_lens, cap).astype(np.int32)
    assert_attention_close(out, oracle_attention(wl, ref_cache), "clamped contexts")


# ------------------------------------------------------------ window / softcap / ALiBi / qq_bias options
# kv_int4_paged_attention_ex against the oracle's definition of the same options (decode split-KV
# walker and prefill kernel alike; several segments per sequence so the options meet the combine).

def _run_opts(wl, window_left=-1, softcap=0.0, slopes=None, segment_len=None, qq_bias=None):
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import assert_attention_close, dev, gpu_cache, gpu_write, oracle_cache, status
    cache = gpu_cache(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_size)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    seg = wl.segment_len if segment_len is None else segment_len
    out = kv.kv_int4_paged_attention(
        wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
        torch.from_numpy(wl.seq_lens).to(dev()), torch.from_numpy(wl.query_start_loc).to(dev()),
        wl.softmax_scale, torch.from_numpy(wl.signs).to(dev()), max_query_len=wl.max_query_len,
        max_seq_len=wl.max_seq_len, out_dtype=torch.float32, segment_len=seg, window_left=window_left,
        softcap=softcap, alibi_slopes=None if slopes is None else torch.tensor(slopes, dtype=torch.float32,
                                                                                 device=dev()),
        qq_bias=None if qq_bias is None else torch.from_numpy(np.ascontiguousarray(qq_bias, np.float32)).to(dev()))
    torch.cuda.synchronize()
    import oracle
    ref = oracle.paged_attention(wl.query, oracle_cache(wl), wl.block_tables, wl.seq_lens, wl.query_start_loc,
                                 wl.softmax_scale, wl.signs, window_left=window_left, softcap=softcap,
                                 alibi_slopes=slopes, qq_bias=None if qq_bias is None else np.asarray(qq_bias, np.float32))
    assert_attention_close(out, ref, wl.name + " (options)")
    st = status()
    assert not any(st.values()), st


def _opts_workload(G, seed):
    # decode contexts across segment edges and two prefill chunks (a diagonal and a full tile)
    return workloads.make_attention_workload("opts", [700, 33, 1, 2100, 300, 1500], [1, 1, 1, 1, 160, 200],
                                             8 * G, 8, 128, seed=seed, segment_len=256)


@pytest.mark.parametrize("G", [4, 8])
@pytest.mark.parametrize("window", [0, 37, 1000])
def test_sliding_window(G, window):
    _run_opts(_opts_workload(G, 31), window_left=window)


@pytest.mark.parametrize("G", [4, 8])
def test_softcap(G):
    wl = _opts_workload(G, 32)
    wl.query = (wl.query.float() * 6.0).to(wl.query.dtype)   # logits large enough for the cap to bite
    _run_opts(wl, softcap=5.0)


@pytest.mark.parametrize("G", [1, 8])
def test_alibi(G):
    wl = _opts_workload(G, 33)
    slopes = [2.0 ** (-(i % 8) - 1) for i in range(8 * G)]
    _run_opts(wl, slopes=slopes)


@pytest.mark.parametrize("G", [4, 8])
def test_qq_bias(G):
    # a random bias over the 200-query chunks, -inf entries (masked keys) included; decode
    # sequences take bias[0, 0] on their own key
    wl = _opts_workload(G, 35)
    r = np.random.default_rng(35)
    bias = r.uniform(-4, 4, (200, 208)).astype(np.float32)
    bias[r.random(bias.shape) < 0.05] = -np.inf
    np.fill_diagonal(bias, 0.5)   # every query keeps a visible key of its own
    _run_opts(wl, qq_bias=bias)


@pytest.mark.parametrize("tiled", [True, False])
def test_options_head64(tiled):
    # head size 64 with every option; many decode sequences put the prefill on its tile grid, a
    # prefill-only batch on one slice per sequence
    lens, qlens = ([400, 90, 1200, 33, 700, 64, 250, 900], [1, 1, 130, 1, 1, 64, 1, 1]) if tiled else \
        ([400, 1200, 300], [100, 130, 64])
    wl = workloads.make_attention_workload("opts64", lens, qlens, 16, 4, 64, seed=37, segment_len=128)
    wl.query = (wl.query.float() * 3.0).to(wl.query.dtype)
    r = np.random.default_rng(37)
    _run_opts(wl, window_left=200, softcap=10.0, slopes=[0.05 * (i + 1) for i in range(16)],
              qq_bias=r.uniform(-1.5, 1.5, (130, 136)))


def test_options_together():
    wl = _opts_workload(4, 34)
    wl.query = (wl.query.float() * 4.0).to(wl.query.dtype)
    _run_opts(wl, window_left=150, softcap=8.0, slopes=[0.03 * (i + 1) for i in range(32)],
              qq_bias=np.random.default_rng(36).uniform(-2, 2, (200, 200)))
