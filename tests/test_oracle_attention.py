"""Pins for the read side of the oracle (dequantise, un-rotate, causal softmax attention), each
against something other than the oracle itself: the round trip through the independently written
C encoder, closed forms of attention, and a brute force built from scipy routines.

Pages: "tests/quantization/test_per_token_kv_cache.py" (INT4 dequant: lo/hi nibbles to even/odd
elements, zp = bits & 0xF, scale = bits & -16, (code - zp) * scale, then the inverse rotation;
causal attention over cu_seqlens_q / seqused_k / block_table) and "[Feature] Triton INT4 / INT2
per-token-head KV cache quantization" (the asymmetry is corrected on the score side).
"""
import numpy as np
import pytest
import scipy.linalg
import scipy.special

import oracle
import workloads


def _roundtrip_bound(rows):
    """||x_hat - x||_2 <= ||y_hat - y||_2 (the rotation is orthogonal) <= sqrt(d) * s'/2 for rows
    whose codes are not clamped; 1.5 steps covers clamped extremes.  Slack for fp32 rotation."""
    _, _, sp = oracle.unpack_rows(rows)
    d = (rows.shape[1] - 4) * 2
    return np.sqrt(d) * 1.5 * sp + 1e-5


@pytest.mark.parametrize("d", [64, 128])
def test_decode_rows_inverts_the_c_encoder(d):
    signs = workloads.splitmix64_signs(d)
    x = np.random.default_rng(1).standard_normal((500, d)).astype(np.float32)
    x[:, 3] *= 10.0   # an outlier channel, spread by the rotation
    rows = oracle.encode_rows(x, signs)
    xhat = oracle.decode_rows(rows, signs)
    err = np.linalg.norm(xhat - x, axis=1)
    assert np.all(err <= _roundtrip_bound(rows))
    # the typical error is far below the bound (uniform rounding: sqrt(d/12) steps)
    _, _, sp = oracle.unpack_rows(rows)
    assert np.median(err / (np.sqrt(d) * sp)) < 0.35


def test_wrong_inverse_fails_the_round_trip():
    """The bound is tight enough to catch a transposed or mis-signed inverse."""
    d = 64
    signs = workloads.splitmix64_signs(d)
    x = np.random.default_rng(2).standard_normal((50, d)).astype(np.float32)
    rows = oracle.encode_rows(x, signs)
    yhat = oracle.dequantize_rotated(rows)
    bad = (yhat @ oracle.hadamard(d).T) / np.sqrt(d)          # signs dropped
    assert np.any(np.linalg.norm(bad - x, axis=1) > _roundtrip_bound(rows))
    bad2 = oracle.unrotate(yhat, -signs)                       # wrong signs
    assert np.any(np.linalg.norm(bad2 - x, axis=1) > _roundtrip_bound(rows))


def _cache_for(wl):
    cache = np.zeros(oracle.cache_shape(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_size), np.uint8)
    oracle.write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    return cache


def _run(wl, cache, **kw):
    return oracle.paged_attention(wl.query, cache, wl.block_tables, wl.seq_lens, wl.query_start_loc,
                                  wl.softmax_scale, wl.signs, **kw)


def test_single_key_returns_its_value():
    wl = workloads.make_attention_workload("t", [1, 1], [1, 1], 4, 2, 64, seed=3)
    cache = _cache_for(wl)
    out = _run(wl, cache)
    for b in range(2):
        for g in range(4):
            h = g // 2
            vrow = oracle.gather_rows(cache, wl.block_tables[b], 1, 1, h)
            np.testing.assert_allclose(out[b, g], oracle.decode_rows(vrow, wl.signs)[0], rtol=0, atol=1e-12)
            # and that is the stored value up to quantisation
            v = wl.value[wl.token_start[b], h].float().numpy()
            assert np.linalg.norm(out[b, g] - v) <= _roundtrip_bound(vrow)[0]


def test_identical_keys_give_the_mean_value():
    wl = workloads.make_attention_workload("t", [37], [1], 2, 1, 64, seed=4)
    wl.key[:] = wl.key[0:1]          # every key the same vector
    cache = _cache_for(wl)
    out = _run(wl, cache)
    vhat = oracle.decode_rows(oracle.gather_rows(cache, wl.block_tables[0], 37, 1, 0), wl.signs)
    np.testing.assert_allclose(out[0, 0], vhat.mean(0), atol=1e-12)
    np.testing.assert_allclose(out[0, 1], vhat.mean(0), atol=1e-12)


def _brute_force(wl, cache, bias=None, chunk_bias=None):
    """Independent restatement: scipy's Hadamard and softmax, explicit per-key loops.  bias(g, j,
    pos, s) -> the logit of key j (None: masked) overrides the plain scaled dot product;
    chunk_bias(t, u) is added to the logit of the chunk's u-th token as a key, for its t-th query."""
    d = wl.head_size
    hm = scipy.linalg.hadamard(d).astype(np.float64)
    G = wl.num_q_heads // wl.num_kv_heads
    q = wl.query.float().numpy().astype(np.float64)
    out = np.zeros_like(q)
    for b in range(len(wl.seq_lens)):
        L = int(wl.seq_lens[b])
        q0, q1 = int(wl.query_start_loc[b]), int(wl.query_start_loc[b + 1])
        for t in range(q1 - q0):
            pos = L - (q1 - q0) + t
            for g in range(wl.num_q_heads):
                h = g // G
                ks, vs = [], []
                for j in range(pos + 1):
                    blk = wl.block_tables[b, j // 16]
                    vecs = []
                    for plane in (0, 1):
                        row = cache[blk, plane, j % 16, h]
                        lo = (row[: d // 2] & 15).astype(np.float64)
                        hi = (row[: d // 2] >> 4).astype(np.float64)
                        code = np.empty(d)
                        code[0::2], code[1::2] = lo, hi
                        word = int(row[d // 2]) | int(row[d // 2 + 1]) << 8 | int(row[d // 2 + 2]) << 16 | int(row[d // 2 + 3]) << 24
                        zp = word & 15
                        sc = float(np.array([word & ~15 & 0xFFFFFFFF], dtype=np.uint32).view(np.float32)[0])
                        y = (code - zp) * sc
                        vecs.append(wl.signs * (hm @ y) / np.sqrt(d))
                    ks.append(vecs[0])
                    vs.append(vecs[1])
                logits = wl.softmax_scale * np.array(ks) @ q[q0 + t, g]
                if chunk_bias is not None:
                    start = L - (q1 - q0)
                    for j in range(start, pos + 1):
                        logits[j] += chunk_bias(t, j - start)
                if bias is not None:
                    kept = [(bias(g, j, pos, float(logits[j])), j) for j in range(pos + 1)]
                    kept = [(x, j) for x, j in kept if x is not None]
                    if not kept:
                        continue
                    p = scipy.special.softmax(np.array([x for x, _ in kept]))
                    out[q0 + t, g] = p @ np.array([vs[j] for _, j in kept])
                    continue
                p = scipy.special.softmax(logits)
                out[q0 + t, g] = p @ np.array(vs)
    return out


def test_matches_brute_force_with_gqa_and_prefill_chunks():
    wl = workloads.make_attention_workload("t", [19, 5, 33], [4, 1, 7], 6, 2, 64, seed=5)
    cache = _cache_for(wl)
    np.testing.assert_allclose(_run(wl, cache), _brute_force(wl, cache), rtol=1e-10, atol=1e-12)


def test_gqa_heads_share_their_kv_head():
    wl = workloads.make_attention_workload("t", [40], [1], 8, 2, 64, seed=6)
    wl.query[0, 1] = wl.query[0, 0]      # same group (kv head 0)
    wl.query[0, 4] = wl.query[0, 0]      # other group (kv head 1)
    out = _run(wl, _cache_for(wl))
    np.testing.assert_array_equal(out[0, 1], out[0, 0])
    assert not np.allclose(out[0, 4], out[0, 0])


def test_causality():
    wl = workloads.make_attention_workload("t", [30], [6], 2, 1, 64, seed=7)
    base = _run(wl, _cache_for(wl))
    wl.key[27:] = -wl.key[27:]           # future of the first three queries (positions 24..26)
    wl.value[27:] = 3 * wl.value[27:]
    out = _run(wl, _cache_for(wl))
    np.testing.assert_array_equal(out[:3], base[:3])
    assert not np.allclose(out[3:], base[3:])


def test_block_table_is_pure_indirection():
    a = workloads.make_attention_workload("t", [50, 20], [1, 1], 4, 2, 64, seed=8, block_order="contiguous")
    b = workloads.make_attention_workload("t", [50, 20], [1, 1], 4, 2, 64, seed=8, block_order="permuted",
                                          extra_blocks=3)
    assert not np.array_equal(a.block_tables, b.block_tables[:, : a.block_tables.shape[1]])
    np.testing.assert_array_equal(_run(a, _cache_for(a)), _run(b, _cache_for(b)))


def test_score_side_correction_identity():
    """The packed read path scores with sum_i q'_i * code_i - zp * sum_i q'_i in the rotated domain;
    by orthogonality that equals q . x_hat / s'.  Check the identity on the oracle's own rows."""
    d = 128
    signs = workloads.splitmix64_signs(d)
    rng = np.random.default_rng(9)
    k = rng.standard_normal((64, d)).astype(np.float32)
    q = rng.standard_normal(d)
    rows = oracle.encode_rows(k, signs)
    codes, zp, sp = oracle.unpack_rows(rows)
    qrot = (oracle.hadamard(d) @ (signs * q)) / np.sqrt(d)       # R q in fp64
    split = sp * (codes.astype(np.float64) @ qrot - zp * qrot.sum())
    np.testing.assert_allclose(split, oracle.decode_rows(rows, signs) @ q, rtol=1e-10, atol=1e-10)


# ---------------------------------------------------------------- options: window, softcap, ALiBi
# The unified-attention interface's window_size / softcap arguments ("tests/quantization/
# test_per_token_kv_cache.py") and the ALiBi helper the PR #40633 description lists, each pinned
# against the brute force (its own per-key loop, math.tanh, explicit bias) and closed forms.

def test_window_zero_returns_the_current_value():
    wl = workloads.make_attention_workload("t", [29, 40], [1, 3], 4, 2, 64, seed=21)
    cache = _cache_for(wl)
    out = _run(wl, cache, window_left=0)
    for b in range(2):
        L = int(wl.seq_lens[b])
        q0, q1 = int(wl.query_start_loc[b]), int(wl.query_start_loc[b + 1])
        for t in range(q1 - q0):
            pos = L - (q1 - q0) + t
            for g in range(4):
                vhat = oracle.decode_rows(oracle.gather_rows(cache, wl.block_tables[b], L, 1, g // 2), wl.signs)
                np.testing.assert_allclose(out[q0 + t, g], vhat[pos], atol=1e-12)


@pytest.mark.parametrize("window", [3, 16, 100])
def test_window_matches_brute_force(window):
    wl = workloads.make_attention_workload("t", [19, 5, 33], [4, 1, 7], 6, 2, 64, seed=22)
    cache = _cache_for(wl)
    ref = _brute_force(wl, cache, bias=lambda g, j, pos, s: s if pos - j <= window else None)
    np.testing.assert_allclose(_run(wl, cache, window_left=window), ref, rtol=1e-10, atol=1e-12)


def test_softcap_matches_brute_force_and_vanishes_when_large():
    import math
    wl = workloads.make_attention_workload("t", [19, 5, 33], [4, 1, 7], 6, 2, 64, seed=23)
    wl.query = (wl.query.float() * 8.0).to(wl.query.dtype)   # logits large enough for the cap to bite
    cache = _cache_for(wl)
    cap = 5.0
    ref = _brute_force(wl, cache, bias=lambda g, j, pos, s: cap * math.tanh(s / cap))
    np.testing.assert_allclose(_run(wl, cache, softcap=cap), ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(_run(wl, cache, softcap=1e12), _run(wl, cache), rtol=1e-9, atol=1e-12)


def test_alibi_matches_brute_force_and_limits():
    wl = workloads.make_attention_workload("t", [19, 5, 33], [4, 1, 7], 6, 2, 64, seed=24)
    cache = _cache_for(wl)
    slopes = np.array([0.0, 0.5, 0.125, 1.0, 0.03125, 2.0])
    ref = _brute_force(wl, cache, bias=lambda g, j, pos, s: s + slopes[g] * (j - pos))
    np.testing.assert_allclose(_run(wl, cache, alibi_slopes=slopes), ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(_run(wl, cache, alibi_slopes=np.zeros(6)), _run(wl, cache), atol=0)
    # a steep slope leaves only the newest key
    steep = _run(wl, cache, alibi_slopes=np.full(6, 1e4))
    np.testing.assert_allclose(steep, _run(wl, cache, window_left=0), atol=1e-12)


def test_qq_bias_matches_brute_force_and_closed_forms():
    wl = workloads.make_attention_workload("t", [21, 9, 40], [5, 1, 8], 4, 2, 64, seed=26)
    cache = _cache_for(wl)
    r = np.random.default_rng(26)
    bias = r.uniform(-3, 3, (8, 8))
    ref = _brute_force(wl, cache, chunk_bias=lambda t, u: bias[t, u])
    np.testing.assert_allclose(_run(wl, cache, qq_bias=bias), ref, rtol=1e-10, atol=1e-12)
    # a zero bias changes nothing; a larger matrix than the chunks reads only its leading block
    np.testing.assert_allclose(_run(wl, cache, qq_bias=np.zeros((8, 8))), _run(wl, cache), atol=0)
    big = np.full((12, 12), 99.0)
    big[:8, :8] = bias
    np.testing.assert_allclose(_run(wl, cache, qq_bias=big), _run(wl, cache, qq_bias=bias), atol=0)
    # -inf off the diagonal: each query sees the context before its chunk and itself only; with a
    # one-query chunk (sequence 1) the bias only moves the query's own key, by bias[0, 0]
    diag = np.where(np.eye(8) > 0, 0.0, -np.inf)
    out = _run(wl, cache, qq_bias=diag)
    for b in (0, 2):
        L = int(wl.seq_lens[b])
        q0, q1 = int(wl.query_start_loc[b]), int(wl.query_start_loc[b + 1])
        start = L - (q1 - q0)
        for t in range(q1 - q0):
            keep = lambda g, j, pos, s, t=t, start=start: s if (j < start or j == start + t) else None  # noqa: E731
            one = _brute_force(wl, cache, bias=keep)
            np.testing.assert_allclose(out[q0 + t], one[q0 + t], rtol=1e-10, atol=1e-12)
    shift = np.zeros((8, 8))
    shift[0, 0] = 1.5
    own = _brute_force(wl, cache, bias=lambda g, j, pos, s: s + 1.5 if j == pos else s)
    np.testing.assert_allclose(_run(wl, cache, qq_bias=shift)[5], own[5], rtol=1e-10, atol=1e-12)


def test_options_compose_in_order():
    import math
    wl = workloads.make_attention_workload("t", [33], [5], 4, 2, 64, seed=25)
    wl.query = (wl.query.float() * 6.0).to(wl.query.dtype)
    cache = _cache_for(wl)
    cap, window = 4.0, 9
    slopes = np.array([0.25, 0.5, 0.0625, 1.0])

    def bias(g, j, pos, s):
        if pos - j > window:
            return None
        return cap * math.tanh(s / cap) + slopes[g] * (j - pos)

    ref = _brute_force(wl, cache, bias=bias)
    got = _run(wl, cache, window_left=window, softcap=cap, alibi_slopes=slopes)
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)
