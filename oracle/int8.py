"""CPU oracle for the INT8 per-(token, head) KV cache (the comparator of the INT4 cache).

TEST INFRASTRUCTURE ONLY: the tests and the benchmark may import it; the library never does, and
the two share no code.

Pages followed (titles and sections): "tests/quantization/test_per_token_kv_cache.py"
(INT8_CONFIG: quant range [-128, 127], rounds before store; _quantize_per_token_head_ref: one
scale per token per head, absmax / quant_max clamped at 1e-6, data times the reciprocal of the
scale, rounding, clamp); "[Feature] Triton INT4 / INT2 per-token-head KV cache quantization"
(the INT8 reshape-kernel rounding fix in the PR conversation: round half away from zero, +0.5 /
-0.5 then to int32, where the old kernel truncated); "PR #40835 report", get_kv_cache_shape
(per-token-head rows hold head_size data bytes plus the float32 scale at the tail).  Where the
test helper rounds half to even and the kernel fix rounds half away, the kernel's reading is
taken; the two differ only at exact .5 ties (counted by codes_nearest_even_form).

The INT8 mode has no rotation and no zero-point: per (token, kv head, plane) vector x (upcast to
fp32, exact)

    s = max(fp32(max|x_i| / 127), 1e-6);  r = fp32(1 / s);  v_i = fp32(x_i * r)
    q_i = clamp(trunc(fp32(v_i + (v_i >= 0 ? 0.5 : -0.5))), -128, 127)

and the cache row is the d codes as two's-complement bytes followed by the 4 little-endian bytes of
s.  Reading: x_hat_i = q_i * s.  Every step is one IEEE fp32 operation (numpy float32 arithmetic),
written in the order above.
"""
from __future__ import annotations

import numpy as np

QMAX = 127
SCALE_FLOOR = np.float32(1e-6)


def row_bytes(head_size: int) -> int:
    """d int8 codes + the fp32 scale."""
    return head_size + 4


def cache_shape(num_blocks: int, block_size: int, num_kv_heads: int, head_size: int):
    return (num_blocks, 2, block_size, num_kv_heads, row_bytes(head_size))


def _f32(x) -> np.ndarray:
    import torch
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float32)
    return np.asarray(x, dtype=np.float32)


def quantize(x) -> tuple[np.ndarray, np.ndarray]:
    """x [..., d] -> (codes int8 [..., d], scale fp32 [...]) by the steps in the module docstring."""
    x = _f32(x)
    absmax = np.max(np.abs(x), axis=-1)
    s = (absmax / np.float32(QMAX)).astype(np.float32)
    s = np.where(s >= SCALE_FLOOR, s, SCALE_FLOOR).astype(np.float32)   # also catches NaN
    r = (np.float32(1.0) / s).astype(np.float32)
    v = (x * r[..., None]).astype(np.float32)
    half = np.where(v >= 0, np.float32(0.5), np.float32(-0.5)).astype(np.float32)
    t = np.trunc((v + half).astype(np.float32))
    q = np.clip(t, -128, QMAX).astype(np.int8)
    return q, s


def codes_nearest_even_form(x) -> np.ndarray:
    """Codes with round-half-to-even instead of half-away (the test helper's torch.round form);
    used only to count where the two readings differ (exact .5 ties)."""
    x = _f32(x)
    _, s = quantize(x)
    r = (np.float32(1.0) / s).astype(np.float32)
    v = (x * r[..., None]).astype(np.float32)
    return np.clip(np.rint(v), -128, QMAX).astype(np.int8)


def encode_rows(x) -> np.ndarray:
    """x [n, d] -> cache rows uint8 [n, d + 4]."""
    q, s = quantize(x)
    n, d = q.shape
    rows = np.empty((n, d + 4), dtype=np.uint8)
    rows[:, :d] = q.view(np.uint8)
    rows[:, d:] = s.astype("<f4").view(np.uint8).reshape(n, 4)
    return rows


def write(key, value, slot_mapping, cache: np.ndarray) -> int:
    """Paged store of K and V [T, H, d] at slot_mapping [T] (slot < 0: skipped).  Returns the
    number of tokens whose slot lies past the cache (skipped and counted)."""
    k, v = _f32(key), _f32(value)
    T, H, d = k.shape
    nb, _, bs, _, rb = cache.shape
    assert rb == row_bytes(d)
    bad = 0
    slots = np.asarray(slot_mapping).astype(np.int64)
    for p, x in ((0, k), (1, v)):
        rows = encode_rows(x.reshape(T * H, d)).reshape(T, H, rb)
        for t in range(T):
            sl = int(slots[t])
            if sl < 0:
                continue
            if sl >= nb * bs:
                bad += p == 0
                continue
            cache[sl // bs, p, sl % bs] = rows[t]
    return bad


def decode_rows(rows: np.ndarray) -> np.ndarray:
    """Cache rows [n, d + 4] -> x_hat = q * s in fp64."""
    rows = np.ascontiguousarray(rows)
    d = rows.shape[-1] - 4
    q = rows[..., :d].view(np.int8).astype(np.float64)
    s = rows[..., d:].copy().view("<f4").astype(np.float64)
    return q * s


def paged_attention(query, cache, block_tables, seq_lens, query_start_loc, softmax_scale,
                    seqs=None, kv_heads=None) -> np.ndarray:
    """Causal softmax attention in fp64 over the dequantised INT8 paged cache (same conventions as
    the INT4 oracle's paged_attention: query t of sequence b sits at seq_len - q_len + t; query
    head g reads kv head g // (Hq / H); unselected rows are NaN; no visible key gives zeros)."""
    q = _f32(query).astype(np.float64)
    nq, hq, d = q.shape
    H, bs = cache.shape[3], cache.shape[2]
    G = hq // H
    out = np.full((nq, hq, d), np.nan, dtype=np.float64)
    seqs = range(len(seq_lens)) if seqs is None else seqs
    kv_heads = range(H) if kv_heads is None else kv_heads
    for b in seqs:
        L = int(seq_lens[b])
        q0, q1 = int(query_start_loc[b]), int(query_start_loc[b + 1])
        if q1 == q0:
            continue
        pos = np.arange(L)
        blk = np.asarray(block_tables[b])[pos // bs]
        for h in kv_heads:
            khat = decode_rows(cache[blk, 0, pos % bs, h])
            vhat = decode_rows(cache[blk, 1, pos % bs, h])
            for t in range(q1 - q0):
                nkeys = max(0, min(L - (q1 - q0) + t + 1, L))
                for g in range(h * G, (h + 1) * G):
                    if nkeys == 0:
                        out[q0 + t, g] = 0.0
                        continue
                    sc = softmax_scale * (khat[:nkeys] @ q[q0 + t, g])
                    w = np.exp(sc - sc.max())
                    out[q0 + t, g] = (w @ vhat[:nkeys]) / w.sum()
    return out
