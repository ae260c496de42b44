"""Pins of the INT2 Lloyd-Max oracle against what the mathematics and the readings fix: the
published table of the 4-level Lloyd-Max quantiser of N(0, 1), its optimality conditions checked by
quadrature, nearest-centroid decisions by brute force, the fold summation against an exact sum,
hand examples (tests/golden/int2_hand_examples.txt), the round-trip distortion of Gaussian-like
rotated vectors, the paged addressing, and closed forms of the attention."""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import int2 as o2

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "int2_hand_examples.txt")


def _parse_golden():
    cases, cur = [], None
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


def test_centroids_match_published_table():
    # J. Max (1960), optimum 4-level quantiser of a unit normal: outputs +-0.4528, +-1.510,
    # thresholds 0, +-0.9816, mean squared error 0.1175
    a, b, t = o2.lloyd_max_normal4()
    assert abs(a - 0.4528) < 5e-5 and abs(b - 1.5104) < 5e-4 and abs(t - 0.9816) < 5e-5
    assert o2.CENTROIDS.dtype == np.float32 and o2.CENTROIDS.tolist() == [
        float(np.float32(-b)), float(np.float32(-a)), float(np.float32(a)), float(np.float32(b))]
    assert o2.THRESHOLD == np.float32(t)


def test_centroid_conditions_by_quadrature():
    # independent route: the conditional means and the distortion by numerical integration
    quad = pytest.importorskip("scipy.integrate").quad
    a, b, t = o2.lloyd_max_normal4()
    pdf = lambda x: math.exp(-0.5 * x * x) / math.sqrt(2 * math.pi)   # noqa: E731
    mass_in = quad(pdf, 0, t)[0]
    mass_out = quad(pdf, t, np.inf)[0]
    assert abs(quad(lambda x: x * pdf(x), 0, t)[0] / mass_in - a) < 1e-9
    assert abs(quad(lambda x: x * pdf(x), t, np.inf)[0] / mass_out - b) < 1e-9
    assert abs(t - 0.5 * (a + b)) < 1e-15

    def mse(a_, b_, t_):
        return 2 * (quad(lambda x: (x - a_) ** 2 * pdf(x), 0, t_)[0] +
                    quad(lambda x: (x - b_) ** 2 * pdf(x), t_, np.inf)[0])

    d0 = mse(a, b, t)
    assert abs(d0 - 0.1175) < 1e-4
    for da, db in ((1e-3, 0), (-1e-3, 0), (0, 1e-3), (0, -1e-3)):   # a local minimum
        assert mse(a + da, b + db, 0.5 * (a + da + b + db)) > d0


def test_decisions_are_nearest_centroid():
    # brute force: the code of z = y / sigma is the index of the nearest centroid (fp64 distances)
    # wherever z is not within 1e-6 of a midpoint
    r = np.random.default_rng(3)
    y = (r.standard_normal((4000, 64)) * 10.0 ** r.uniform(-2, 2, (4000, 1))).astype(np.float32)
    codes, s = o2.quantize_rotated(y)
    z = (y * (np.float32(1) / s)[:, None]).astype(np.float32).astype(np.float64)
    c = o2.CENTROIDS.astype(np.float64)
    nearest = np.argmin(np.abs(z[..., None] - c), axis=-1)
    mids = np.array([-(c[3] + c[2]) / 2, 0.0, (c[3] + c[2]) / 2])
    clear = np.min(np.abs(z[..., None] - mids), axis=-1) > 1e-6
    assert clear.mean() > 0.999
    assert np.array_equal(codes[clear], nearest[clear])
    assert np.all(codes <= 3)


def test_fold_sum_against_exact_sum():
    r = np.random.default_rng(4)
    y = r.standard_normal((500, 128)).astype(np.float32)
    got = o2.fold_sum_of_squares(y).astype(np.float64)
    exact = np.array([math.fsum(float(v) ** 2 for v in row) for row in y])
    assert np.all(np.abs(got - exact) <= exact * 128 * 2.0 ** -23)
    # small integers: every partial sum is exact, so the fold is exact
    yi = r.integers(-20, 21, (50, 64)).astype(np.float32)
    assert np.array_equal(o2.fold_sum_of_squares(yi).astype(np.int64), (yi.astype(np.int64) ** 2).sum(1))
    # the fold order itself, (a0 + a2) + (a1 + a3): squares 2^24, 1, 0, 1 fold to (2^24, 2) and
    # then 2^24 + 2 exactly, where the sequential order and adjacent pairs both lose each 1 to the
    # tie-to-even rounding of 2^24 + 1 and end at 2^24
    yo = np.array([[4096.0, 1.0, 0.0, 1.0]], np.float32)
    assert o2.fold_sum_of_squares(yo)[0] == np.float32(2 ** 24 + 2)


def test_scale_is_rms_of_rotated_vector():
    r = np.random.default_rng(5)
    y = (r.standard_normal((300, 128)) * 10.0 ** r.uniform(-3, 3, (300, 1))).astype(np.float32)
    s = o2.scale_of_rotated(y).astype(np.float64)
    rms = np.sqrt((y.astype(np.float64) ** 2).mean(1))
    assert np.all(np.abs(s - rms) <= rms * 2e-5)
    assert o2.scale_of_rotated(np.zeros((1, 64), np.float32))[0] == np.float32(1e-6)


@pytest.mark.parametrize("case", [c for c in GOLDEN_CASES if c["kind"] == "row"], ids=lambda c: c["name"])
def test_row_hand_examples(case):
    x = np.array([float(t) for t in case["x"].split()], dtype=np.float32)
    signs = np.array([float(t) for t in case["signs"].split()], dtype=np.float32)
    want = bytes(int(h, 16) for h in case["bytes"].split())
    assert bytes(o2.encode_rows(x[None], signs)[0]) == want


@pytest.mark.parametrize("case", [c for c in GOLDEN_CASES if c["kind"] == "quant"], ids=lambda c: c["name"])
def test_quant_hand_examples(case):
    y = np.array([float(t) for t in case["y"].split()], dtype=np.float32)
    codes, s = o2.quantize_rotated(y)
    assert codes[0].tolist() == [int(t) for t in case["codes"].split()]
    kind, v = case["scale"].split()
    assert kind == "sqrt" and s[0] == np.float32(math.sqrt(float(v)))


def test_pack_unpack_roundtrip():
    r = np.random.default_rng(6)
    codes = r.integers(0, 4, (20, 128)).astype(np.uint8)
    s = r.uniform(0.1, 10, 20).astype(np.float32)
    rows = o2.pack_rows(codes, s)
    assert rows.shape == (20, 36)
    c2, s2 = o2.unpack_rows(rows)
    assert np.array_equal(c2, codes) and np.array_equal(s2, s)


def test_roundtrip_distortion_is_lloyd_max():
    # Gaussian head vectors stay Gaussian under the rotation: the relative squared error of the
    # round trip is the quantiser's distortion, 0.1175, up to the fluctuation of sigma
    r = np.random.default_rng(7)
    d = 128
    signs = np.where(r.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    x = r.standard_normal((2000, d)).astype(np.float32)
    xh = o2.decode_rows(o2.encode_rows(x, signs), signs)
    rel = ((xh - x) ** 2).sum() / (x.astype(np.float64) ** 2).sum()
    assert abs(rel - 0.1175) < 0.005
    # outliers: a vector with one huge coordinate is spread by the rotation and still decodes
    # with the same relative error
    xo = x[:200].copy()
    xo[:, 7] += 40.0
    xoh = o2.decode_rows(o2.encode_rows(xo, signs), signs)
    relo = ((xoh - xo) ** 2).sum() / (xo.astype(np.float64) ** 2).sum()
    assert relo < 0.2


def test_write_paged_addressing():
    r = np.random.default_rng(8)
    T, H, d, bs, nb = 5, 2, 64, 16, 3
    k = r.standard_normal((T, H, d)).astype(np.float32)
    v = r.standard_normal((T, H, d)).astype(np.float32)
    signs = np.where(r.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    slots = np.array([0, 17, -1, 47, 48])   # 48 is past the 3 blocks
    cache = np.zeros(o2.cache_shape(nb, bs, H, d), np.uint8)
    assert o2.write(k, v, slots, signs, cache) == 1
    for t, sl in enumerate(slots[:4]):
        if sl < 0:
            continue
        assert np.array_equal(cache[sl // bs, 0, sl % bs], o2.encode_rows(k[t], signs))
        assert np.array_equal(cache[sl // bs, 1, sl % bs], o2.encode_rows(v[t], signs))
    written = {0, 17, 47}
    for sl in range(nb * bs):
        if sl not in written:
            assert not cache[sl // bs, :, sl % bs].any()


def test_attention_closed_forms():
    # identical keys: uniform weights, the output is the mean of the decoded values; a single key:
    # the output is that key's decoded value
    r = np.random.default_rng(9)
    H, G, d, bs = 1, 2, 64, 16
    signs = np.where(r.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    L = 21
    kvec = r.standard_normal(d).astype(np.float32)
    k = np.repeat(kvec[None, None], L, 0).repeat(H, 1)
    v = r.standard_normal((L, H, d)).astype(np.float32)
    cache = np.zeros(o2.cache_shape(2, bs, H, d), np.uint8)
    o2.write(k, v, np.arange(L), signs, cache)
    q = r.standard_normal((2, H * G, d)).astype(np.float32)
    bt = np.array([[0, 1], [0, 1]], np.int32)
    out = o2.paged_attention(q, cache, bt, np.array([L, 1]), np.array([0, 1, 2]), 0.125, signs)
    vh = o2.decode_rows(cache[[0] * 16 + [1] * 5, 1, list(range(16)) + list(range(5)), 0], signs)
    np.testing.assert_allclose(out[0], np.repeat(vh.mean(0)[None], G, 0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out[1], np.repeat(vh[:1], G, 0), rtol=1e-12, atol=1e-12)
    # the INT4 oracle's attention with the INT2 decoder is the same function of the decoded rows
    assert not np.isnan(out).any()


def test_hadamard_rotation_is_shared_with_int4():
    # the INT2 row rotates exactly as the INT4 row: the sign of each rotated element agrees with the
    # side of 0 the INT2 code falls on
    r = np.random.default_rng(10)
    d = 128
    signs = np.where(r.random(d) < 0.5, -1.0, 1.0).astype(np.float32)
    x = r.standard_normal((50, d)).astype(np.float32)
    y = oracle.rotate(x, signs)
    codes, _ = o2.unpack_rows(o2.encode_rows(x, signs))
    assert np.array_equal(codes >= 2, y >= 0)
