"""Pins of the INT8 per-(token, head) oracle against what the definition fixes: hand examples with
exactly representable values, the quantiser's invariants, the tie rule, the byte layout, the paged
addressing, and closed forms of the attention (one key, identical keys, causality, shared kv
heads)."""
import struct

import numpy as np
import pytest

from oracle import int8 as o8


def test_hand_examples():
    # absmax 127 -> s = 1: codes are the values rounded half away from zero
    q, s = o8.quantize(np.array([[127.0, -63.5, 0.0, 1.0]], np.float32))
    assert s.tolist() == [1.0] and q.tolist() == [[127, -64, 0, 1]]
    # absmax 254 -> s = 2, r = 0.5: 1 -> 0.5 -> 1, -1 -> -0.5 -> -1 (ties away), 0.5 -> 0.25 -> 0
    q, s = o8.quantize(np.array([[254.0, 1.0, -1.0, 0.5]], np.float32))
    assert s.tolist() == [2.0] and q.tolist() == [[127, 1, -1, 0]]
    # the all-zero vector takes the 1e-6 floor and codes 0
    q, s = o8.quantize(np.zeros((1, 8), np.float32))
    assert s[0] == np.float32(1e-6) and not q.any()


def test_pages_raw_cache_vector():
    # "tests/quantization/test_per_token_kv_cache.py", test_int8_per_token_head_raw_cache_matches_
    # round_reference: one bf16 vector of 8 elements, V = -K, a cache of one block of 4 slots, slot 2.
    # bf16 (8 significant bits) holds 127 exactly and rounds the others to the nearest multiple of
    # 2^-6 (for 2 <= |x| < 4), 2^-7 (1 <= |x| < 2), 2^-8 (0.5 <= |x| < 1) or 2^-9 (0.25 <= |x| < 0.5):
    #   2.6 -> 166/64 = 2.59375, 2.4 -> 154/64 = 2.40625, 1.6 -> 205/128 = 1.6015625,
    #   1.4 -> 179/128 = 1.3984375, 0.6 -> 154/256 = 0.6015625, 0.4 -> 205/512 = 0.400390625.
    # absmax = 127, so s = 127 / 127 = 1 and r = 1: the codes are the values rounded to the nearest
    # integer (no ties here), -127 -3 -2 -2 -1 -1 0 127, where truncation toward zero -- the bug the
    # page's INT8 reshape-kernel fix removes -- would give -127 -2 -2 -1 -1 0 0 127.
    import torch
    key = torch.tensor([[[-127.0, -2.6, -2.4, -1.6, -1.4, -0.6, -0.4, 127.0]]], dtype=torch.bfloat16)
    assert key.float().flatten().tolist() == [-127.0, -2.59375, -2.40625, -1.6015625, -1.3984375, -0.6015625,
                                              -0.400390625, 127.0]
    cache = np.zeros(o8.cache_shape(1, 4, 1, 8), np.uint8)
    assert o8.write(key, -key, np.array([2]), cache) == 0
    k_codes = cache[0, 0, 2, 0, :8].view(np.int8).tolist()
    v_codes = cache[0, 1, 2, 0, :8].view(np.int8).tolist()
    assert k_codes == [-127, -3, -2, -2, -1, -1, 0, 127]
    assert v_codes == [127, 3, 2, 2, 1, 1, 0, -127]
    for p in (0, 1):
        assert struct.unpack("<f", bytes(cache[0, p, 2, 0, 8:12]))[0] == 1.0
    assert not cache[0, :, [0, 1, 3]].any()   # the other slots of the block are untouched


def test_quantizer_invariants():
    r = np.random.default_rng(1)
    x = (r.standard_normal((512, 128)) * 10.0 ** r.uniform(-3, 3, (512, 1))).astype(np.float32)
    q, s = o8.quantize(x)
    assert q.dtype == np.int8 and q.min() >= -127 and q.max() <= 127   # |v| <= 127 up to rounding
    am = np.argmax(np.abs(x), axis=1)
    assert np.all(np.abs(q[np.arange(512), am]) == 127)                 # the absmax element
    err = np.abs(q.astype(np.float64) * s[:, None] - x.astype(np.float64))
    assert np.all(err <= s[:, None].astype(np.float64) * (0.5 + 1e-5))     # one half step at most
    assert np.all(np.sign(q) * np.sign(x) >= 0)                           # no sign flips


def test_ties_round_away_and_only_ties_differ_from_nearest_even():
    r = np.random.default_rng(2)
    # values that land exactly on k + 1/2 after scaling by 1/s = 1 (absmax 127)
    x = np.concatenate([np.full((64, 1), 127.0), r.integers(-126, 126, (64, 31)) + 0.5], 1).astype(np.float32)
    q, _ = o8.quantize(x)
    v = x[:, 1:]
    assert np.array_equal(q[:, 1:], (np.trunc(v + np.sign(v) * 0.5)).astype(np.int8))
    ne = o8.codes_nearest_even_form(x)
    diff = q != ne
    assert diff.any()
    assert np.all(np.abs(x[diff] - np.floor(x[diff])) == 0.5)   # every difference is a tie
    # random data has (almost) no ties
    y = r.standard_normal((256, 128)).astype(np.float32)
    assert (o8.quantize(y)[0] != o8.codes_nearest_even_form(y)).mean() < 1e-4


def test_row_layout():
    x = np.array([[3.0, -127.0, 0.25, -0.5, 64.0, 1.0, -1.0, 126.6]], np.float32)
    row = o8.encode_rows(x)[0]
    q, s = o8.quantize(x)
    assert row.shape == (o8.row_bytes(8),)
    assert [struct.unpack("b", bytes([b]))[0] for b in row[:8]] == q[0].tolist()   # two's complement
    assert struct.unpack("<f", bytes(row[8:12]))[0] == s[0]                        # scale, little-endian
    np.testing.assert_allclose(o8.decode_rows(row[None])[0], q[0] * np.float64(s[0]))


def test_write_addressing_and_skips():
    r = np.random.default_rng(3)
    T, H, d, nb, bs = 6, 2, 16, 4, 4
    k = r.standard_normal((T, H, d)).astype(np.float32)
    v = r.standard_normal((T, H, d)).astype(np.float32)
    slots = np.array([0, 5, -1, 15, 16, 7])      # -1 skipped, 16 past the cache (counted)
    cache = np.full(o8.cache_shape(nb, bs, H, d), 0xAB, np.uint8)
    bad = o8.write(k, v, slots, cache)
    assert bad == 1
    for t, sl in enumerate(slots):
        if 0 <= sl < nb * bs:
            assert np.array_equal(cache[sl // bs, 0, sl % bs], o8.encode_rows(k[t]))
            assert np.array_equal(cache[sl // bs, 1, sl % bs], o8.encode_rows(v[t]))
    untouched = np.ones(nb * bs, bool)
    untouched[[0, 5, 15, 7]] = False
    for sl in np.nonzero(untouched)[0]:
        assert np.all(cache[sl // bs, :, sl % bs] == 0xAB)


def _cache_from(k, v, bs=4):
    T, H, d = k.shape
    nb = (T + bs - 1) // bs
    cache = np.zeros(o8.cache_shape(nb, bs, H, d), np.uint8)
    o8.write(k, v, np.arange(T), cache)
    return cache, np.arange(nb)[None]


def test_single_key_returns_its_value():
    r = np.random.default_rng(4)
    k = r.standard_normal((1, 2, 32)).astype(np.float32)
    v = r.standard_normal((1, 2, 32)).astype(np.float32)
    cache, tables = _cache_from(k, v)
    q = r.standard_normal((1, 4, 32)).astype(np.float32)
    out = o8.paged_attention(q, cache, tables, [1], [0, 1], 0.3)
    vhat = o8.decode_rows(cache[0, 1, 0])
    for g in range(4):
        np.testing.assert_allclose(out[0, g], vhat[g // 2], rtol=0, atol=1e-15)


def test_identical_keys_give_the_mean_value_and_causality_holds():
    r = np.random.default_rng(5)
    T, H, d = 9, 1, 16
    k = np.repeat(r.standard_normal((1, H, d)), T, 0).astype(np.float32)
    v = r.standard_normal((T, H, d)).astype(np.float32)
    cache, tables = _cache_from(k, v)
    q = r.standard_normal((1, 1, d)).astype(np.float32)
    out = o8.paged_attention(q, cache, tables, [T], [0, 1], 0.7)
    vhat = o8.decode_rows(cache[tables[0][np.arange(T) // 4], 1, np.arange(T) % 4, 0])
    np.testing.assert_allclose(out[0, 0], vhat.mean(0), rtol=1e-12, atol=1e-14)
    # a chunk of 3 queries at positions 6, 7, 8: changing the last key changes only the last query
    q3 = r.standard_normal((3, 1, d)).astype(np.float32)
    a = o8.paged_attention(q3, cache, tables, [T], [0, 3], 0.7)
    k2 = k.copy()
    k2[8] *= -3.0
    cache2, _ = _cache_from(k2, v)
    b = o8.paged_attention(q3, cache2, tables, [T], [0, 3], 0.7)
    np.testing.assert_array_equal(a[:2], b[:2])
    assert not np.allclose(a[2], b[2])


@pytest.mark.parametrize("G", [1, 4])
def test_matches_plain_softmax_over_dequantised_rows(G):
    # brute force on a tiny case: every (query, head) as an explicit loop over keys
    r = np.random.default_rng(6 + G)
    T, H, d = 7, 2, 8
    k = r.standard_normal((T, H, d)).astype(np.float32)
    v = r.standard_normal((T, H, d)).astype(np.float32)
    cache, tables = _cache_from(k, v)
    q = r.standard_normal((2, H * G, d)).astype(np.float32)
    out = o8.paged_attention(q, cache, tables, [T], [0, 2], 0.5)
    kq, ks = o8.quantize(k)
    vq, vs = o8.quantize(v)
    for t in range(2):
        n = T - 2 + t + 1
        for g in range(H * G):
            h = g // G
            sc = [0.5 * sum(float(q[t, g, i]) * float(kq[j, h, i]) * float(ks[j, h]) for i in range(d)) for j in range(n)]
            m = max(sc)
            w = [np.exp(x - m) for x in sc]
            ref = [sum(w[j] * float(vq[j, h, i]) * float(vs[j, h]) for j in range(n)) / sum(w) for i in range(d)]
            np.testing.assert_allclose(out[t, g], ref, rtol=1e-12, atol=1e-12)
