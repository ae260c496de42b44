"""CPU oracle for the INT2 per-(token, head) Lloyd-Max KV cache.

TEST INFRASTRUCTURE ONLY: the tests and the benchmark may import it; the library never does, and
the two share no code.

Page followed: "[Feature] Triton INT4 / INT2 per-token-head KV cache quantization" (vLLM PR #40633),
description and commit notes: the INT2 mode packs four 2-bit values per byte, rotates each head
vector with a Hadamard transform over the whole head dimension, and dequantises by looking up one
of four Lloyd-Max centroids fitted to the standard normal distribution, with its scale factor
folded in when the cache is written.  The page gives neither the centroids nor the scale, so this
module takes the plainest reading that fits the rest of the description:

* rotation: the INT4 mode's y = c * H_d * (D x) (the package's ``rotate``: same signs, the same
  fp32 butterfly order); a caller that wants the unsigned transform passes signs of all +1;
* scale: the root mean square of the rotated vector, which puts its coordinates on the unit
  normal the centroids are fitted to (a Hadamard-rotated head vector is close to Gaussian):
      a_i = fp32(y_i * y_i);  fold in halves: a_i <- fp32(a_i + a_{i+h}) for h = d/2, d/4, .., 1
      sigma = max(fp32(sqrt(fp32(a_0 / d))), 1e-6)
  (the fold is the fixed summation order of a vectorised reduction; the floor is the INT4 mode's);
  the page's "d1.5" factor is garbled in the text: any constant factor would be folded into the
  stored scale, so the read side (sigma * centroid) does not depend on it;
* centroids: the 4-level Lloyd-Max quantiser of N(0, 1) (J. Max, "Quantizing for minimum
  distortion", 1960): outputs -b, -a, a, b and decision thresholds -t, 0, t with t = (a + b) / 2,
  a = E[X | 0 < X < t], b = E[X | X > t]; computed here by the Lloyd iteration in fp64, then
  rounded to fp32 (outputs and threshold alike);
* codes: z_i = fp32(y_i * fp32(1 / sigma)); code_i = [z_i >= -t] + [z_i >= 0] + [z_i >= t], so
  codes 0, 1, 2, 3 stand for -b, -a, a, b (a value exactly on a threshold takes the upper code);
* row: d / 4 bytes, element 4j + k in bits 2k, 2k + 1 of byte j (the low bits first, as the INT4
  mode puts the even element in the low nibble), then the 4 little-endian bytes of sigma;
  cache shape (num_blocks, 2, block_size, num_kv_heads, d / 4 + 4);
* read: y_hat_i = sigma * centroid[code_i] (fp64 of the fp32 values), x_hat = the inverse rotation,
  then the same causal attention as the INT4 oracle.
"""
from __future__ import annotations

import math

import numpy as np

from . import _as_f32_array, paged_attention as _attention_over, rotate, unrotate

SCALE_FLOOR = np.float32(1e-6)


def _phi(x: float) -> float:
    return math.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def _Phi(x: float) -> float:
    return 0.5 * (1.0 + math.erf(x / math.sqrt(2.0)))


def lloyd_max_normal4(iterations: int = 20000) -> tuple[float, float, float]:
    """(a, b, t) of the symmetric 4-level Lloyd-Max quantiser of N(0, 1) in fp64.

    Lloyd's two conditions, alternated until they stop moving: each threshold is the midpoint of
    its neighbouring outputs (t = (a + b) / 2, and 0 by symmetry), each output the mean of the
    density over its cell (a over (0, t), b over (t, inf))."""
    a, b = 0.5, 1.5
    for _ in range(iterations):
        t = 0.5 * (a + b)
        na = (_phi(0.0) - _phi(t)) / (_Phi(t) - 0.5)
        nb = _phi(t) / (1.0 - _Phi(t))
        if abs(na - a) < 1e-16 and abs(nb - b) < 1e-16:
            a, b = na, nb
            break
        a, b = na, nb
    return a, b, 0.5 * (a + b)


_A, _B, _T = lloyd_max_normal4()
CENTROIDS = np.array([-_B, -_A, _A, _B], dtype=np.float32)    # code 0..3
THRESHOLD = np.float32(_T)                                     # decisions at -t, 0, t


def row_bytes(head_size: int) -> int:
    """d / 4 code bytes + the fp32 scale."""
    return head_size // 4 + 4


def cache_shape(num_blocks: int, block_size: int, num_kv_heads: int, head_size: int):
    return (num_blocks, 2, block_size, num_kv_heads, row_bytes(head_size))


def fold_sum_of_squares(y: np.ndarray) -> np.ndarray:
    """sum_i y_i^2 of each row in fp32, folded in halves (a_i + a_{i + d/2}, then + a_{i + d/4}, ...)."""
    with np.errstate(over="ignore"):   # squares past fp32 range are inf, as in IEEE arithmetic
        a = (y * y).astype(np.float32)
    while a.shape[-1] > 1:
        h = a.shape[-1] // 2
        a = (a[..., :h] + a[..., h:]).astype(np.float32)
    return a[..., 0]


def scale_of_rotated(y) -> np.ndarray:
    """sigma of each already-rotated row (fp32)."""
    y = np.asarray(y, dtype=np.float32)
    d = y.shape[-1]
    ms = (fold_sum_of_squares(y) / np.float32(d)).astype(np.float32)
    s = np.sqrt(ms).astype(np.float32)
    return np.where(s >= SCALE_FLOOR, s, SCALE_FLOOR).astype(np.float32)   # also catches NaN


def quantize_rotated(y) -> tuple[np.ndarray, np.ndarray]:
    """Codes [N, d] (uint8, 0..3) and scales [N] (fp32) of already-rotated rows."""
    y = np.atleast_2d(np.asarray(y, dtype=np.float32))
    s = scale_of_rotated(y)
    r = (np.float32(1.0) / s).astype(np.float32)
    z = (y * r[:, None]).astype(np.float32)
    codes = (z >= -THRESHOLD).astype(np.uint8) + (z >= 0).astype(np.uint8) + (z >= THRESHOLD).astype(np.uint8)
    return codes, s


def pack_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """codes [N, d] (0..3), scales [N] -> rows [N, d/4 + 4] uint8."""
    n, d = codes.shape
    c = codes.astype(np.uint8).reshape(n, d // 4, 4)
    data = c[:, :, 0] | (c[:, :, 1] << 2) | (c[:, :, 2] << 4) | (c[:, :, 3] << 6)
    rows = np.empty((n, row_bytes(d)), dtype=np.uint8)
    rows[:, : d // 4] = data
    rows[:, d // 4:] = np.asarray(scales, dtype="<f4").view(np.uint8).reshape(n, 4)
    return rows


def encode_rows(x, signs) -> np.ndarray:
    """Head vectors x [N, d] -> cache rows [N, d/4 + 4]."""
    x = np.atleast_2d(_as_f32_array(x))
    if x.shape[1] % 4:
        raise ValueError("head size must be a multiple of 4")
    codes, s = quantize_rotated(rotate(x, signs))
    return pack_rows(codes, s)


def write(key, value, slot_mapping, signs, cache: np.ndarray) -> int:
    """Paged store of K and V [T, H, d] at slot_mapping [T] (slot < 0: skipped).  Returns the
    number of tokens whose slot lies past the cache (skipped and counted)."""
    k, v = _as_f32_array(key), _as_f32_array(value)
    T, H, d = k.shape
    nb, _, bs, _, rb = cache.shape
    assert rb == row_bytes(d)
    bad = 0
    slots = np.asarray(slot_mapping).astype(np.int64)
    for p, x in ((0, k), (1, v)):
        rows = encode_rows(x.reshape(T * H, d), signs).reshape(T, H, rb)
        for t in range(T):
            sl = int(slots[t])
            if sl < 0:
                continue
            if sl >= nb * bs:
                bad += p == 0
                continue
            cache[sl // bs, p, sl % bs] = rows[t]
    return bad


def unpack_rows(rows: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """rows [N, d/4 + 4] -> (codes [N, d] uint8, sigma [N] fp32)."""
    rows = np.atleast_2d(np.ascontiguousarray(rows))
    nb = rows.shape[1] - 4
    data = rows[:, :nb]
    codes = np.stack([(data >> (2 * k)) & 3 for k in range(4)], axis=-1).reshape(rows.shape[0], 4 * nb)
    s = np.ascontiguousarray(rows[:, nb:]).view("<f4")[:, 0]
    return codes.astype(np.uint8), s


def dequantize_rotated(rows: np.ndarray) -> np.ndarray:
    """sigma * centroid[code] in fp64: the row's vector in the rotated domain."""
    codes, s = unpack_rows(rows)
    return CENTROIDS.astype(np.float64)[codes] * s.astype(np.float64)[:, None]


def decode_rows(rows: np.ndarray, signs) -> np.ndarray:
    """Cached rows -> reconstructed head vectors in the original domain (fp64)."""
    return unrotate(dequantize_rotated(rows), signs)


def paged_attention(query, cache, block_tables, seq_lens, query_start_loc, softmax_scale, signs,
                    seqs=None, kv_heads=None) -> np.ndarray:
    """Causal softmax attention in fp64 over the dequantised, un-rotated INT2 paged cache (the INT4
    oracle's attention with this module's row decoding)."""
    return _attention_over(query, cache, block_tables, seq_lens, query_start_loc, softmax_scale, signs,
                           seqs=seqs, kv_heads=kv_heads, row_decoder=decode_rows)
