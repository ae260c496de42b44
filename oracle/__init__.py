"""CPU oracle for the INT4 per-(token, head) KV cache and the paged attention that reads it.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package; the library under ``int4_token_head_kv_gb300`` never does, and the two share
no code.

* The write (rotation, quantisation, zero-point in the scale bits, nibble packing, paged store) is
  an encoding, so it is stated step by step in plain C (``kv_int4_oracle.c``) and called here
  through ctypes.
* The attention has a plain definition, written out here in fp64 numpy: dequantise every cached
  row in the rotated domain, un-rotate it (x = c * D * H_d * y with the exact 1/sqrt(d)), and run
  ordinary causal softmax attention with the original, un-rotated queries.  No split-dot, no
  rotation of Q, no segments: by the orthogonality of the rotation that is what the packed read
  path computes.

Pages followed (titles and sections): "[Feature] Triton INT4 / INT2 per-token-head KV cache
quantization" (PR #40633 description: rotation, asymmetric codes, zero-point in the scale,
score-side correction); "tests/quantization/test_per_token_kv_cache.py" (the INT4 dequant in
test_reshape_and_cache_per_token_head: lo/hi nibbles to even/odd elements, zp = bits & 0xF,
scale = bits & -16, (code - zp) * scale, inverse rotation; causal unified attention with
cu_seqlens_q and seqused_k in test_triton_unified_attention_per_token_head_scale); "PR #40835
report" (cache shape (num_blocks, 2, block_size, num_kv_heads, head_size // 2 + 4)).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build import LIB, build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = LIB if os.path.exists(LIB) else build_oracle()
        lib = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        lib.oracle_rotate_f32.argtypes = [f32p, f32p, ctypes.c_int, f32p]
        lib.oracle_rotate_f32.restype = ctypes.c_int
        lib.oracle_quantize_rotated.argtypes = [f32p, ctypes.c_int, u8p, ctypes.POINTER(ctypes.c_uint32)]
        lib.oracle_quantize_rotated.restype = ctypes.c_int
        lib.oracle_codes_division_form.argtypes = [f32p, ctypes.c_int, u8p]
        lib.oracle_codes_division_form.restype = ctypes.c_int
        lib.oracle_encode_row.argtypes = [f32p, f32p, ctypes.c_int, u8p]
        lib.oracle_encode_row.restype = ctypes.c_int
        lib.oracle_kv_int4_write.argtypes = [f32p, f32p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                             ctypes.POINTER(ctypes.c_int64), f32p, u8p,
                                             ctypes.c_int64, ctypes.c_int]
        lib.oracle_kv_int4_write.restype = ctypes.c_int64
        _lib = lib
    return _lib


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _as_f32_array(x) -> np.ndarray:
    """fp16 / bf16 / fp32 input (torch tensor or numpy array) -> its exact fp32 value."""
    if hasattr(x, "detach"):
        return np.ascontiguousarray(x.detach().cpu().float().numpy())
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def row_bytes(head_size: int) -> int:
    """Bytes per cached (token, head) row: head_size/2 code bytes then one fp32 scale."""
    return head_size // 2 + 4


def cache_shape(num_blocks: int, block_size: int, num_kv_heads: int, head_size: int):
    return (num_blocks, 2, block_size, num_kv_heads, row_bytes(head_size))


# ----------------------------------------------------------------------------- write side (C)

def rotate(x, signs) -> np.ndarray:
    """fp32 rotation y = c * H_d * (D x) of each row of x, in the fixed butterfly order."""
    lib = _load()
    x, _ = _f32(np.atleast_2d(_as_f32_array(x)))
    s, sp = _f32(signs)
    y = np.empty_like(x)
    for i in range(x.shape[0]):
        rc = lib.oracle_rotate_f32(x[i].ctypes.data_as(ctypes.POINTER(ctypes.c_float)), sp,
                                   x.shape[1], y[i].ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
        if rc != 0:
            raise ValueError("head size must be a power of two")
    return y


def quantize_rotated(y):
    """Codes [N, d] (uint8, 0..15) and scale words [N] (uint32) of already-rotated rows."""
    lib = _load()
    y, _ = _f32(np.atleast_2d(y))
    n, d = y.shape
    codes = np.empty((n, d), dtype=np.uint8)
    words = np.empty(n, dtype=np.uint32)
    for i in range(n):
        w = ctypes.c_uint32()
        lib.oracle_quantize_rotated(y[i].ctypes.data_as(ctypes.POINTER(ctypes.c_float)), d,
                                    codes[i].ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
                                    ctypes.byref(w))
        words[i] = w.value
    return codes, words


def codes_division_form(y) -> np.ndarray:
    """Codes formed as fp32 (y / s') + zp then rounded: the pages' reference form."""
    lib = _load()
    y, _ = _f32(np.atleast_2d(y))
    n, d = y.shape
    codes = np.empty((n, d), dtype=np.uint8)
    for i in range(n):
        lib.oracle_codes_division_form(y[i].ctypes.data_as(ctypes.POINTER(ctypes.c_float)), d,
                                       codes[i].ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    return codes


def encode_rows(x, signs) -> np.ndarray:
    """Cache rows [N, d/2 + 4] (uint8) of head vectors x [N, d]."""
    lib = _load()
    x = np.atleast_2d(_as_f32_array(x))
    n, d = x.shape
    s, sp = _f32(signs)
    rows = np.empty((n, row_bytes(d)), dtype=np.uint8)
    for i in range(n):
        rc = lib.oracle_encode_row(x[i].ctypes.data_as(ctypes.POINTER(ctypes.c_float)), sp, d,
                                   rows[i].ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
        if rc != 0:
            raise ValueError("head size must be a power of two")
    return rows


def write(key, value, slot_mapping, signs, cache: np.ndarray) -> int:
    """Write K/V [T, H, d] into ``cache`` (uint8 numpy, modified in place) at ``slot_mapping``.

    Returns the number of slots that were out of range (skipped)."""
    lib = _load()
    k, kp = _f32(_as_f32_array(key))
    v, vp = _f32(_as_f32_array(value))
    T, H, d = k.shape
    assert v.shape == k.shape
    slots = np.ascontiguousarray(np.asarray(slot_mapping, dtype=np.int64))
    s, sp = _f32(signs)
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    nb, two, bs, hh, rb = cache.shape
    assert two == 2 and hh == H and rb == row_bytes(d)
    bad = lib.oracle_kv_int4_write(kp, vp, T, H, d, slots.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                   sp, cache.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), nb, bs)
    if bad < 0:
        raise ValueError("head size must be a power of two")
    return int(bad)


# ------------------------------------------------------------------------ read side (fp64 numpy)

def unpack_rows(rows: np.ndarray):
    """rows [N, d/2+4] uint8 -> (codes [N, d] uint8, zp [N] int, truncated scale s' [N] float64)."""
    rows = np.atleast_2d(rows)
    d = (rows.shape[1] - 4) * 2
    data = rows[:, : d // 2]
    codes = np.empty((rows.shape[0], d), dtype=np.uint8)
    codes[:, 0::2] = data & 0xF
    codes[:, 1::2] = data >> 4
    word = np.ascontiguousarray(rows[:, d // 2: d // 2 + 4]).view("<u4")[:, 0]
    zp = (word & 0xF).astype(np.int64)
    scale = (word & np.uint32(0xFFFFFFF0)).view(np.float32).astype(np.float64)
    return codes, zp, scale


def dequantize_rotated(rows: np.ndarray) -> np.ndarray:
    """(code - zp) * s' in fp64: the row's vector in the rotated domain."""
    codes, zp, scale = unpack_rows(rows)
    return (codes.astype(np.float64) - zp[:, None]) * scale[:, None]


def hadamard(d: int) -> np.ndarray:
    """Natural-order (Sylvester) Hadamard matrix: H_1 = [1], H_2n = [[H, H], [H, -H]]."""
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def unrotate(yhat: np.ndarray, signs) -> np.ndarray:
    """x = c * D * H_d * y in fp64 with the exact c = 1/sqrt(d) (rows of yhat are vectors)."""
    d = yhat.shape[-1]
    hmat = hadamard(d)
    return (yhat @ hmat.T) * (np.asarray(signs, dtype=np.float64) / np.sqrt(d))


def decode_rows(rows: np.ndarray, signs) -> np.ndarray:
    """Cached rows -> reconstructed head vectors in the original domain (fp64)."""
    return unrotate(dequantize_rotated(rows), signs)


def gather_rows(cache: np.ndarray, block_table_row: np.ndarray, seq_len: int, plane: int, head: int):
    """The cached rows of positions 0..seq_len-1 of one sequence for one kv head and plane
    (0 = K, 1 = V); slot of position j = block_table[j // bs] * bs + j % bs."""
    bs = cache.shape[2]
    pos = np.arange(seq_len)
    blk = np.asarray(block_table_row)[pos // bs]
    return cache[blk, plane, pos % bs, head]


def paged_attention(query, cache, block_tables, seq_lens, query_start_loc, softmax_scale, signs,
                    seqs=None, kv_heads=None, window_left=-1, softcap=0.0, alibi_slopes=None,
                    row_decoder=None, qq_bias=None) -> np.ndarray:
    """Causal softmax attention over the dequantised, un-rotated paged cache, in fp64.

    query [Nq, Hq, d] (original domain); sequence b owns query rows
    query_start_loc[b] .. query_start_loc[b+1]-1, and its t-th query sits at position
    seq_len[b] - q_len[b] + t, seeing keys 0 .. that position.  Query head g reads kv head
    g // (Hq / H).  Returns fp64 [Nq, Hq, d]; rows of sequences or kv heads that are not selected
    (``seqs`` / ``kv_heads``) are NaN.  An empty key range gives a zero output.  ``row_decoder``
    (rows, signs) -> original-domain vectors reads another row format (default: the INT4 rows).

    Options of the unified-attention interface ("tests/quantization/test_per_token_kv_cache.py",
    ``window_size`` and ``softcap`` arguments; the PR #40633 description lists sliding window,
    softcap and ALiBi among the shared helpers), in this order on the scaled logit
    s_j = softmax_scale * q . k_j of key j for a query at position pos:
      softcap > 0:           s_j <- softcap * tanh(s_j / softcap)
      alibi_slopes [Hq]:     s_j <- s_j + slope_g * (j - pos)
      qq_bias [Q, Q]:        s_j <- s_j + qq_bias[t, j - c] for the keys of the query chunk itself
                             (c = seq_len - q_len <= j, j - c < Q), t the query's index in its chunk
      window_left >= 0:      key j is visible only if pos - j <= window_left (besides j <= pos).
    The page lists qq_bias among the shared helpers without defining it; this reading is the
    query-to-query bias of the unified-attention interface: one [Q, Q] matrix for every sequence and
    head, row t for the chunk's t-th query, column u for the chunk's u-th token as a key.
    """
    q = _as_f32_array(query).astype(np.float64)
    nq, hq, d = q.shape
    H = cache.shape[3]
    G = hq // H
    out = np.full((nq, hq, d), np.nan, dtype=np.float64)
    seqs = range(len(seq_lens)) if seqs is None else seqs
    kv_heads = range(H) if kv_heads is None else kv_heads
    dec = decode_rows if row_decoder is None else row_decoder
    for b in seqs:
        L = int(seq_lens[b])
        q0, q1 = int(query_start_loc[b]), int(query_start_loc[b + 1])
        qlen = q1 - q0
        if qlen == 0:
            continue
        for h in kv_heads:
            khat = dec(gather_rows(cache, block_tables[b], L, 0, h), signs)
            vhat = dec(gather_rows(cache, block_tables[b], L, 1, h), signs)
            for t in range(qlen):
                pos = L - qlen + t
                nkeys = max(0, min(pos + 1, L))
                first = max(0, pos - window_left) if window_left >= 0 else 0   # first visible key
                for g in range(h * G, (h + 1) * G):
                    if nkeys <= first:
                        out[q0 + t, g] = 0.0
                        continue
                    s = softmax_scale * (khat[first:nkeys] @ q[q0 + t, g])
                    if softcap > 0:
                        s = softcap * np.tanh(s / softcap)
                    if alibi_slopes is not None:
                        s = s + float(alibi_slopes[g]) * (np.arange(first, nkeys) - pos)
                    if qq_bias is not None:
                        bias = np.asarray(qq_bias, dtype=np.float64)
                        u = np.arange(first, nkeys) - (L - qlen)
                        inside = (u >= 0) & (u < bias.shape[1])
                        s = s + np.where(inside, bias[t, np.clip(u, 0, bias.shape[1] - 1)], 0.0)
                    w = np.exp(s - s.max())
                    out[q0 + t, g] = (w @ vhat[first:nkeys]) / w.sum()
    return out
