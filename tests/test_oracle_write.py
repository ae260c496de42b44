"""Pins for the write side of the oracle, each against something other than the oracle itself:
a library Hadamard matrix, closed forms, hand-derived examples and mathematical bounds.

Pages: "[Feature] Triton INT4 / INT2 per-token-head KV cache quantization" (rotation, asymmetric
codes, zero-point in the scale's low mantissa bits, truncated-scale review note) and
"tests/quantization/test_per_token_kv_cache.py" (INT4 reference quantiser and dequant, slot
addressing, negative-slot skip).
"""
import os

import numpy as np
import pytest
import scipy.linalg

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "write_hand_examples.txt")


def _parse_golden():
    cases = []
    cur = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("quant ") or line.startswith("row "):
                kind, name = line.split()
                cur = {"kind": kind, "name": name}
                cases.append(cur)
                continue
            key, val = [s.strip() for s in line.split("=", 1)]
            cur[key] = val
    return cases


GOLDEN_CASES = _parse_golden()


@pytest.mark.parametrize("case", [c for c in GOLDEN_CASES if c["kind"] == "quant"], ids=lambda c: c["name"])
def test_quantizer_hand_examples(case):
    y = np.array([float(t) for t in case["y"].split()], dtype=np.float32)
    codes, words = oracle.quantize_rotated(y)
    assert codes[0].tolist() == [int(t) for t in case["codes"].split()]
    assert int(words[0]) == int(case["word"], 16)


@pytest.mark.parametrize("case", [c for c in GOLDEN_CASES if c["kind"] == "row"], ids=lambda c: c["name"])
def test_encode_row_hand_examples(case):
    x = np.array([float(t) for t in case["x"].split()], dtype=np.float32)
    s = np.array([float(t) for t in case["signs"].split()], dtype=np.float32)
    row = oracle.encode_rows(x, s)[0]
    assert row.tolist() == [int(t, 16) for t in case["bytes"].split()]


@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_is_sylvester(d):
    h = oracle.hadamard(d)
    assert np.array_equal(h, scipy.linalg.hadamard(d).astype(np.float64))
    assert np.array_equal(h @ h.T, d * np.eye(d))


@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128])
def test_rotation_matches_dense_hadamard(d):
    rng = np.random.default_rng(d)
    signs = workloads.splitmix64_signs(d)
    x = rng.standard_normal((64, d)).astype(np.float32)
    y = oracle.rotate(x, signs)
    ref = (x.astype(np.float64) * signs) @ scipy.linalg.hadamard(d).T / np.sqrt(d)
    # fp32 butterflies: every output is a sum of d terms formed by a depth-log2(d) tree of
    # rounded adds, then one rounded multiply.
    bound = (np.log2(d) + 2) * 2.0 ** -24 * np.abs(x).sum(axis=1, keepdims=True) / np.sqrt(d) * 1.01
    assert np.all(np.abs(y - ref) <= bound)


@pytest.mark.parametrize("d", [4, 16, 64])
def test_rotation_exact_on_small_integers(d):
    # d = 4, 16, 64 have c = 1/2, 1/4, 1/8 exactly, and integer sums stay exact in fp32
    rng = np.random.default_rng(7)
    signs = workloads.splitmix64_signs(d)
    x = rng.integers(-100, 101, size=(16, d)).astype(np.float32)
    y = oracle.rotate(x, signs)
    ref = (x.astype(np.int64) * signs.astype(np.int64)) @ scipy.linalg.hadamard(d).T
    assert np.array_equal(y.astype(np.float64), ref / np.sqrt(d))


@pytest.mark.parametrize("d", [8, 64, 128])
def test_one_hot_spreads_to_constant_magnitude(d):
    signs = workloads.splitmix64_signs(d)
    c = np.float32(1.0 / np.sqrt(d))
    hm = scipy.linalg.hadamard(d)
    for k in [0, 1, d // 2, d - 1]:
        x = np.zeros(d, np.float32)
        x[k] = 1.0
        y = oracle.rotate(x, signs)[0]
        assert np.all(np.abs(y) == c)
        assert np.array_equal(np.sign(y), signs[k] * hm[:, k])


def test_rotation_preserves_norms_and_dot_products():
    d = 128
    rng = np.random.default_rng(3)
    signs = workloads.splitmix64_signs(d)
    q = rng.standard_normal((32, d)).astype(np.float32)
    k = rng.standard_normal((32, d)).astype(np.float32)
    rq = oracle.rotate(q, signs).astype(np.float64)
    rk = oracle.rotate(k, signs).astype(np.float64)
    np.testing.assert_allclose((rq * rk).sum(1), (q.astype(np.float64) * k).sum(1), atol=1e-4)
    np.testing.assert_allclose(np.linalg.norm(rq, axis=1), np.linalg.norm(q.astype(np.float64), axis=1), rtol=1e-6)


def _rotated_gaussians(n, d, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d)).astype(np.float32)
    return oracle.rotate(x, workloads.splitmix64_signs(d))


@pytest.mark.parametrize("d", [64, 128])
def test_quantizer_invariants(d):
    y = _rotated_gaussians(2000, d, d + 11)
    codes, words = oracle.quantize_rotated(y)
    assert codes.max() <= 15
    zp = (words & 0xF).astype(np.int64)
    sp = (words & np.uint32(0xFFFFFFF0)).view(np.float32).astype(np.float64)
    assert np.all(zp <= 15)
    # the truncated scale is within 15 ulp below the plain one, and never above it
    s = ((y.max(1).astype(np.float32) - y.min(1).astype(np.float32)) / np.float32(15)).astype(np.float32)
    s = np.maximum(s, np.float32(1e-6))
    assert np.all((s.view(np.uint32) & np.uint32(0xFFFFFFF0)) == (words & np.uint32(0xFFFFFFF0)))
    assert np.all(sp <= s) and np.all(sp >= s * (1 - 16 * 2.0 ** -23))
    # reconstruction error in the rotated domain: half a step for every code strictly inside
    # (0, 15), plus the rounding of the reciprocal
    err = np.abs((codes - zp[:, None]) * sp[:, None] - y.astype(np.float64))
    inner = (codes > 0) & (codes < 15)
    bound = 0.5 * sp[:, None] + np.abs(y) * 2.0 ** -23
    assert np.all(err[inner] <= bound.repeat(1, axis=0)[inner] * (1 + 1e-6))
    # the extremes sit at the ends of the code range (one step of slack for exact ties)
    assert np.all(codes.min(1) <= 1) and np.all(codes.max(1) >= 14)
    assert np.all(np.take_along_axis(codes, y.argmin(1)[:, None], 1) <= 1)
    assert np.all(np.take_along_axis(codes, y.argmax(1)[:, None], 1) >= 14)
    # the whole vector stays within 1.5 steps even where a code is clamped
    assert np.all(err <= 1.5 * sp[:, None] + np.abs(y) * 2.0 ** -23)


def test_one_rounding_codes_rarely_differ_from_division_form():
    """The pages' reference divides (y / s' + zp, two roundings); the spec multiplies by the
    reciprocal with one rounding.  They may differ by one step only next to a rounding tie."""
    y = _rotated_gaussians(20000, 128, 5)
    a, _ = oracle.quantize_rotated(y)
    b = oracle.codes_division_form(y)
    diff = np.abs(a.astype(np.int64) - b.astype(np.int64))
    assert diff.max() <= 1
    assert diff.astype(bool).mean() <= 1e-4


def test_write_addressing_and_skips():
    """slot -> (slot // block_size, slot % block_size); K in plane 0, V in plane 1; slots < 0 are
    skipped; slots past the cache are skipped and counted."""
    wl = workloads.random_write(12, 3, 64, seed=4, num_blocks=3, negative_every=4)
    slots = wl.slot_mapping.copy()
    slots[5] = wl.num_blocks * wl.block_size + 7     # out of range
    cache = np.full(oracle.cache_shape(wl.num_blocks, wl.block_size, 3, 64), 0xA5, np.uint8)
    before = cache.copy()
    bad = oracle.write(wl.key, wl.value, slots, wl.signs, cache)
    assert bad == 1
    touched = np.zeros(cache.shape[:3], dtype=bool)
    for t, slot in enumerate(slots.tolist()):
        if slot < 0 or slot >= wl.num_blocks * wl.block_size:
            continue
        blk, off = divmod(slot, wl.block_size)
        for p, src in enumerate([wl.key, wl.value]):
            exp = oracle.encode_rows(src[t], wl.signs)
            assert np.array_equal(cache[blk, p, off], exp)
            touched[blk, p, off] = True
    assert np.array_equal(cache[~touched], before[~touched])
    assert touched.sum() == 2 * sum(1 for s in slots if 0 <= s < wl.num_blocks * wl.block_size)


def test_negative_slots_leave_cache_unchanged():
    # shape of the pages' negative-slot test: 4 tokens, 2 heads, d 64, 2 blocks, slots [0,-1,1,-1]
    wl = workloads.random_write(4, 2, 64, seed=0, num_blocks=2)
    slots = np.array([0, -1, 1, -1], np.int64)
    cache = np.zeros(oracle.cache_shape(2, 16, 2, 64), np.uint8)
    oracle.write(wl.key, wl.value, slots, wl.signs, cache)
    assert cache[0, :, :2].any(axis=(-1, -2)).all()
    assert not cache[0, :, 2:].any() and not cache[1].any()


def test_pack_unpack_round_trip():
    """The C packer and the numpy unpacker are written independently; codes and scale word must
    survive the trip (the hand examples pin the byte order itself: even element in the low nibble)."""
    for d in (64, 128):
        signs = workloads.splitmix64_signs(d)
        x = np.random.default_rng(d).standard_normal((300, d)).astype(np.float32)
        rows = oracle.encode_rows(x, signs)
        codes, words = oracle.quantize_rotated(oracle.rotate(x, signs))
        c2, zp, sp = oracle.unpack_rows(rows)
        assert np.array_equal(c2, codes)
        assert np.array_equal(zp, (words & 0xF).astype(np.int64))
        assert np.array_equal(sp, (words & np.uint32(0xFFFFFFF0)).view(np.float32).astype(np.float64))
