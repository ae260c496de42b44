"""Seeded synthetic inputs for the INT4 per-(token, head) KV-cache write and the paged attention
that reads it.

This module only draws random numbers and lays out index structures (sequence lengths, block
tables, slot mappings, query offsets).  It holds none of the method's arithmetic: no rotation,
no quantisation, no packing, no attention.  The CPU oracle and the CUDA path both consume exactly
what it returns, so both sides see identical input bits.

Recipe (all draws from numpy's PCG64 through ``np.random.SeedSequence``):

* Each component (structure, K, V, Q) gets its own child stream spawned from the workload seed,
  so that the draw of one never depends on the size of another.  Large tensors are drawn in
  chunks of about 4 M elements, chunk i from the i-th child of the component's stream, in
  parallel threads (the bits do not depend on the thread count).
* Gaussian draws are float32 ``standard_normal``; Student-t draws are ``Z * sqrt(nu / (2 G))``
  with ``G ~ Gamma(nu/2)`` (the textbook construction t = Z / sqrt(chi2_nu / nu)).
* The float32 draws are rounded to fp16 / bf16 with round-to-nearest-even (torch ``.to``).
* The Hadamard sign vector comes from SplitMix64 (Steele, Lea and Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014), seeded with 0: sign_i = -1 when the top bit of
  the i-th output is set, else +1.  One vector is shared by K, V and Q.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK_SIZE = 16

_MASK64 = (1 << 64) - 1


def splitmix64_signs(d: int, seed: int = 0) -> np.ndarray:
    """Return ``d`` float32 values, each exactly +1.0 or -1.0, from SplitMix64(seed)."""
    state = seed & _MASK64
    out = np.empty(d, dtype=np.float32)
    for i in range(d):
        state = (state + 0x9E3779B97F4A7C15) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        z = z ^ (z >> 31)
        out[i] = -1.0 if (z >> 63) else 1.0
    return out


def _to_half(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype)


def _children(seed: int, n: int) -> list[np.random.SeedSequence]:
    return np.random.SeedSequence(seed).spawn(n)


def _rng(seq: np.random.SeedSequence) -> np.random.Generator:
    return np.random.default_rng(seq)


_CHUNK_ELEMS = 1 << 22


def _fill_random(shape, dtype, seq, dist, row_scale=None):
    """Draw ``shape`` (rows first) into a torch CPU tensor of ``dtype``.

    The rows are cut into chunks of about 4 M elements; chunk i draws from the i-th child of ``seq``,
    so the result does not depend on how many threads draw the chunks (they run in parallel).
    ``row_scale`` (float32 [rows]) multiplies each row: it carries the per-token magnitudes of the
    write-throughput workload.  The multiplication is part of drawing the input, not of the method.
    """
    out = torch.empty(shape, dtype=dtype)
    rows = shape[0]
    inner = tuple(shape[1:])
    per_row = int(np.prod(inner)) if inner else 1
    chunk_rows = max(1, _CHUNK_ELEMS // max(1, per_row))
    starts = list(range(0, rows, chunk_rows))
    seqs = seq.spawn(len(starts))

    def one(i):
        r0 = starts[i]
        r1 = min(rows, r0 + chunk_rows)
        rng = np.random.default_rng(seqs[i])
        sub = (r1 - r0,) + inner
        if dist == "normal":
            x = rng.standard_normal(sub, dtype=np.float32)
        elif dist == "student_t3":
            nu = 3.0
            z = rng.standard_normal(sub, dtype=np.float32)
            g = rng.standard_gamma(nu / 2.0, sub, dtype=np.float32)
            x = z * np.sqrt(np.float32(nu) / (np.float32(2.0) * g))
        else:
            raise ValueError(dist)
        if row_scale is not None:
            x *= row_scale[r0:r1].reshape((-1,) + (1,) * len(inner))
        out[r0:r1] = _to_half(x, dtype)

    workers = min(len(starts), os.cpu_count() or 1, 16)
    if workers <= 1:
        for i in range(len(starts)):
            one(i)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(one, range(len(starts))))
    return out


@dataclass
class WriteWorkload:
    """Inputs of one cache write: ``num_tokens`` new K/V vectors and where they go."""

    name: str
    key: torch.Tensor            # [T, H, d] fp16/bf16, CPU
    value: torch.Tensor          # [T, H, d]
    slot_mapping: np.ndarray     # int64 [T]; < 0 = padding token, skipped
    num_blocks: int
    block_size: int
    signs: np.ndarray            # float32 [d], each +-1

    @property
    def num_tokens(self) -> int:
        return self.key.shape[0]

    @property
    def num_kv_heads(self) -> int:
        return self.key.shape[1]

    @property
    def head_size(self) -> int:
        return self.key.shape[2]


@dataclass
class AttentionWorkload:
    """A batch of sequences whose context lives in a paged cache, plus this step's queries.

    Tokens are stored sequence-major in ``key``/``value``: sequence ``b`` owns rows
    ``token_start[b] : token_start[b+1]`` (its positions 0 .. seq_len-1).  The last
    ``query_len[b]`` of them are this step's new tokens: a step writes them into the cache and
    then attends with ``query`` (the earlier ones are the history, written before the step).
    """

    name: str
    seq_lens: np.ndarray         # int32 [S]
    query_lens: np.ndarray       # int32 [S]
    block_tables: np.ndarray     # int32 [S, max_blocks_per_seq]
    num_blocks: int
    key: torch.Tensor            # [sum(seq_lens), H, d]
    value: torch.Tensor
    query: torch.Tensor          # [sum(query_lens), Hq, d]
    signs: np.ndarray            # float32 [d]
    num_q_heads: int
    segment_len: int = 0         # 0 = let the library choose
    block_size: int = BLOCK_SIZE
    token_start: np.ndarray = field(init=False)
    query_start_loc: np.ndarray = field(init=False)
    slot_mapping: np.ndarray = field(init=False)

    def __post_init__(self):
        self.token_start = np.concatenate([[0], np.cumsum(self.seq_lens, dtype=np.int64)])
        self.query_start_loc = np.concatenate(
            [[0], np.cumsum(self.query_lens, dtype=np.int64)]).astype(np.int32)
        slots = np.empty(int(self.token_start[-1]), dtype=np.int64)
        for b, L in enumerate(self.seq_lens.tolist()):
            pos = np.arange(L, dtype=np.int64)
            blk = self.block_tables[b, pos // self.block_size].astype(np.int64)
            slots[self.token_start[b]:self.token_start[b + 1]] = blk * self.block_size + pos % self.block_size
        self.slot_mapping = slots

    @property
    def num_kv_heads(self) -> int:
        return self.key.shape[1]

    @property
    def head_size(self) -> int:
        return self.key.shape[2]

    @property
    def softmax_scale(self) -> float:
        return float(self.head_size) ** -0.5

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if len(self.query_lens) else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if len(self.seq_lens) else 0

    def new_token_rows(self) -> np.ndarray:
        """Row indices (into key/value) of this step's new tokens, in query order."""
        idx = [np.arange(self.token_start[b + 1] - q, self.token_start[b + 1])
               for b, q in enumerate(self.query_lens.tolist())]
        return np.concatenate(idx).astype(np.int64) if idx else np.zeros(0, np.int64)

    def history_token_rows(self) -> np.ndarray:
        idx = [np.arange(self.token_start[b], self.token_start[b + 1] - q)
               for b, q in enumerate(self.query_lens.tolist())]
        return np.concatenate(idx).astype(np.int64) if idx else np.zeros(0, np.int64)


def make_attention_workload(name, seq_lens, query_lens, num_q_heads, num_kv_heads, head_size,
                            dtype=torch.bfloat16, kv_dist="normal", k_outlier_channels=0,
                            k_outlier_gain=10.0, seed=0, block_order="permuted", extra_blocks=0,
                            segment_len=0, block_size=BLOCK_SIZE):
    seq_lens = np.asarray(seq_lens, dtype=np.int32)
    query_lens = np.asarray(query_lens, dtype=np.int32)
    assert np.all(query_lens <= seq_lens)
    s_struct, r_k, r_v, r_q = _children(seed, 4)
    r_struct = _rng(s_struct)
    nblk = [(int(L) + block_size - 1) // block_size for L in seq_lens]
    total_blocks = sum(nblk) + extra_blocks
    maxb = max(nblk) if nblk else 1
    if block_order == "permuted":
        ids = r_struct.permutation(total_blocks).astype(np.int32)
    else:
        ids = np.arange(total_blocks, dtype=np.int32)
    tables = np.zeros((len(seq_lens), max(maxb, 1)), dtype=np.int32)
    pos = 0
    for b, n in enumerate(nblk):
        tables[b, :n] = ids[pos:pos + n]
        pos += n
    T = int(seq_lens.sum())
    H, d = num_kv_heads, head_size
    key = _fill_random((T, H, d), dtype, r_k, kv_dist)
    if k_outlier_channels:
        # per kv head, a fixed set of channels is louder for every token of K
        chans = np.stack([r_struct.choice(d, k_outlier_channels, replace=False) for _ in range(H)])
        gain = np.ones((H, d), dtype=np.float32)
        for h in range(H):
            gain[h, chans[h]] = k_outlier_gain
        for r0 in range(0, T, 65536):
            r1 = min(T, r0 + 65536)
            key[r0:r1] = _to_half(key[r0:r1].float().numpy() * gain[None], dtype)
    value = _fill_random((T, H, d), dtype, r_v, kv_dist)
    query = _fill_random((int(query_lens.sum()), num_q_heads, d), dtype, r_q, "normal")
    return AttentionWorkload(name=name, seq_lens=seq_lens, query_lens=query_lens,
                             block_tables=tables, num_blocks=total_blocks, key=key, value=value,
                             query=query, signs=splitmix64_signs(d, 0), num_q_heads=num_q_heads,
                             segment_len=segment_len, block_size=block_size)


# ---------------------------------------------------------------------------------------------
# The five named workloads.  Sizes follow the workloads the method is evaluated on; scaled-down
# variants (same structure, fewer tokens) serve as parity cases the oracle finishes in seconds.
# ---------------------------------------------------------------------------------------------

def tiny_write_decode(seed=0) -> AttentionWorkload:
    """Two sequences of 42 and 7 tokens, 4 q / 4 kv heads, head_size 64, fp16 N(0,1).

    Blocks are contiguous (sequence 0 owns blocks 0,1,2; sequence 1 owns block 3); every token is
    written, then each sequence runs one causal decode query.
    """
    return make_attention_workload("tiny_write_decode", [42, 7], [1, 1], 4, 4, 64,
                                   dtype=torch.float16, seed=seed, block_order="contiguous")


def gqa_decode_batch(seed=0, num_seqs=32, len_range=(512, 4096)) -> AttentionWorkload:
    """32 sequences with lengths uniform in [512, 4096], 32 q / 8 kv heads, d 128, bf16 N(0,1).

    Per kv head, 4 random K channels are 10x louder for every token; blocks are randomly permuted.
    """
    rng = _rng(_children(seed + 1000, 1)[0])
    lens = rng.integers(len_range[0], len_range[1] + 1, size=num_seqs)
    return make_attention_workload("gqa_decode_batch", lens, np.ones(num_seqs, np.int32), 32, 8, 128,
                                   dtype=torch.bfloat16, k_outlier_channels=4, seed=seed)


def long_context_decode(seed=0, num_seqs=8, seq_len=131072, segment_len=4096) -> AttentionWorkload:
    """8 sequences x 131072 tokens, 64 q / 8 kv heads, d 128, bf16 Student-t(3) K/V, N(0,1) Q.

    One decode query per sequence; split-KV segments of 4096 tokens.
    """
    return make_attention_workload("long_context_decode", [seq_len] * num_seqs, [1] * num_seqs, 64, 8,
                                   128, dtype=torch.bfloat16, kv_dist="student_t3", seed=seed,
                                   segment_len=segment_len)


def write_throughput(seed=0, num_tokens=65536, num_kv_heads=8, head_size=128,
                     num_blocks=8192, block_size=BLOCK_SIZE) -> WriteWorkload:
    """65536 new tokens, 8 kv heads, d 128, bf16: K, V = N(0,1) x m_t with m_t = 10^U(-2, 2) drawn
    per token (independently for K and V); slots are the first 65536 entries of a random
    permutation of the 8192 x 16 cache slots."""
    s_struct, r_k, r_v, s_mk, s_mv = _children(seed, 5)
    r_struct, r_mk, r_mv = _rng(s_struct), _rng(s_mk), _rng(s_mv)
    slots = r_struct.permutation(num_blocks * block_size)[:num_tokens].astype(np.int64)
    mk = np.power(np.float32(10.0), r_mk.uniform(-2.0, 2.0, num_tokens).astype(np.float32))
    mv = np.power(np.float32(10.0), r_mv.uniform(-2.0, 2.0, num_tokens).astype(np.float32))
    shape = (num_tokens, num_kv_heads, head_size)
    key = _fill_random(shape, torch.bfloat16, r_k, "normal", row_scale=mk.astype(np.float32))
    value = _fill_random(shape, torch.bfloat16, r_v, "normal", row_scale=mv.astype(np.float32))
    return WriteWorkload("write_throughput", key, value, slots, num_blocks, block_size,
                         splitmix64_signs(head_size, 0))


def mixed_prefill_decode(seed=0, num_prefill=4, prefill_cached=2048, prefill_chunk=2048,
                         num_decode=60, decode_len_max=32768) -> AttentionWorkload:
    """4 prefill sequences (2048 cached tokens + a 2048-token causal chunk, so seq_len 4096) and
    60 decode sequences with lengths uniform in [1, 32768]; 32 q / 8 kv heads, d 128, bf16 N(0,1).
    Prefill sequences come first in the batch."""
    rng = _rng(_children(seed + 2000, 1)[0])
    dec = rng.integers(1, decode_len_max + 1, size=num_decode)
    lens = [prefill_cached + prefill_chunk] * num_prefill + dec.tolist()
    qlens = [prefill_chunk] * num_prefill + [1] * num_decode
    return make_attention_workload("mixed_prefill_decode", lens, qlens, 32, 8, 128,
                                   dtype=torch.bfloat16, seed=seed)


def random_write(num_tokens, num_kv_heads, head_size, dtype=torch.bfloat16, seed=0,
                 num_blocks=None, block_size=BLOCK_SIZE, scale=1.0, negative_every=0):
    """Small write cases in the shape of the pages' cache-write tests: N(0,1) x ``scale`` K/V and
    slots sampled without replacement; optionally every ``negative_every``-th slot is -1."""
    s_struct, r_k, r_v = _children(seed, 3)
    r_struct = _rng(s_struct)
    if num_blocks is None:
        num_blocks = (num_tokens + block_size - 1) // block_size + 4
    slots = r_struct.permutation(num_blocks * block_size)[:num_tokens].astype(np.int64)
    if negative_every:
        slots[1::negative_every] = -1
    shape = (num_tokens, num_kv_heads, head_size)
    key = _fill_random(shape, dtype, r_k, "normal", row_scale=np.full(num_tokens, scale, np.float32))
    value = _fill_random(shape, dtype, r_v, "normal", row_scale=np.full(num_tokens, scale, np.float32))
    return WriteWorkload("random_write", key, value, slots, num_blocks, block_size,
                         splitmix64_signs(head_size, 0))
