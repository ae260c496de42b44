"""Time the oracle (as it stands) on a bounded sample of a workload; prints one JSON line.

TEST INFRASTRUCTURE: run by the benchmark's CPU-baseline leg and its reference arm, in a
subprocess whose BLAS threads the caller fixes through the environment.

  python -m oracle.timing long_decode <pairs> <seed> [--procs P]
      long-context decode workload (8 sequences x 131072 tokens, 64 q / 8 kv heads): the sample is
      <pairs> (sequence, kv head) pairs, each written in full (all 131072 tokens of that head) into
      the oracle's cache and then attended by that kv head's 8 query heads, one after the other on
      one thread.  With --procs P, P worker processes then take one further pair each at once (the
      all-cores leg), and the wall time from a common start to the last finish is reported.
  python -m oracle.timing decode <num_seqs_sample> <seed>   GQA decode batch, first sequences
  python -m oracle.timing write <num_tokens_sample> <seed>  write-throughput workload, first tokens

The reported bytes are the packed-KV (+ Q/O) bytes the sample covers (for the write: the input and
output bytes), so ``bytes / seconds`` is in the benchmark's unit.
"""
from __future__ import annotations

import json
import multiprocessing as mp
import os
import sys
import tempfile
import time

import numpy as np


def _one_pair(k, v, q, signs, softmax_scale):
    """Oracle write of one kv head's whole context [L, 1, d] and the attention of its query heads
    q [1, G, d]; returns (seconds, packed-KV + Q/O bytes)."""
    import oracle
    L, _, d = k.shape
    nb = (L + 15) // 16
    cache = np.zeros(oracle.cache_shape(nb, 16, 1, d), np.uint8)
    t0 = time.perf_counter()
    oracle.write(k, v, np.arange(L, dtype=np.int64), signs, cache)
    oracle.paged_attention(q, cache, np.arange(nb, dtype=np.int32)[None], np.array([L], np.int32),
                           np.array([0, 1], np.int32), softmax_scale, signs)
    dt = time.perf_counter() - t0
    return dt, L * 2 * (d // 2 + 4) + 2 * q.shape[1] * d * 2


def _long_pairs(seed, n, first=0):
    """(sequence, kv head) pairs first .. first + n - 1 of the long-context workload, in the order
    (pair i -> sequence i % 8, kv head (i // 8) % 8), as the 16-bit patterns of their bf16 K, V and
    query rows (half the bytes of fp32 to hand to the worker processes)."""
    import workloads
    wl = workloads.long_context_decode(seed=seed)
    S, H, Hq = len(wl.seq_lens), wl.num_kv_heads, wl.num_q_heads
    G = Hq // H
    out = []
    for i in range(first, first + n):
        b, h = i % S, (i // S) % H
        r0, r1 = int(wl.token_start[b]), int(wl.token_start[b + 1])
        out.append((_bits(wl.key[r0:r1, h:h + 1]), _bits(wl.value[r0:r1, h:h + 1]),
                    _bits(wl.query[b:b + 1, h * G:(h + 1) * G])))
    return out, wl.signs, wl.softmax_scale


def _bits(t):
    """bf16 tensor -> its 16-bit patterns (numpy uint16)."""
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f32_of_bits(u):
    """bf16 bit patterns -> the exact fp32 values."""
    return (np.asarray(u).astype(np.uint32) << 16).view(np.float32)


def _worker(path, idx, pairs, barrier, results):
    data = np.load(path, mmap_mode="r")
    signs, scale = np.array(data["signs"]), float(data["scale"])
    arrs = [(_f32_of_bits(data[f"k{idx}_{j}"]), _f32_of_bits(data[f"v{idx}_{j}"]), _f32_of_bits(data[f"q{idx}_{j}"]))
            for j in range(pairs)]
    barrier.wait()
    nbytes = 0
    for k, v, q in arrs:
        nbytes += _one_pair(k, v, q, signs, scale)[1]
    results.put((idx, time.perf_counter(), nbytes))


def _long_decode(pairs, seed, procs):
    """Single-threaded leg on ``pairs`` pairs, and (procs > 1) the all-cores leg: ``procs`` processes
    at once, one further pair each.  The workload is drawn once for both."""
    sample, signs, scale = _long_pairs(seed, pairs + (procs if procs > 1 else 0))
    secs, nbytes = 0.0, 0
    for k, v, q in sample[:pairs]:
        s_, b_ = _one_pair(_f32_of_bits(k), _f32_of_bits(v), _f32_of_bits(q), signs, scale)
        secs += s_
        nbytes += b_
    res = {"single": {"seconds": secs, "bytes": nbytes, "units": pairs, "threads": 1,
                      "what": f"{pairs} (sequence, kv head) pairs of the long-context decode, 131072 tokens each, "
                              f"written and attended by 8 query heads, one thread"}}
    if procs <= 1:
        return res
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    try:
        arrays = {"signs": signs, "scale": np.float64(scale)}
        for i in range(procs):
            k, v, q = sample[pairs + i]
            arrays[f"k{i}_0"], arrays[f"v{i}_0"], arrays[f"q{i}_0"] = k, v, q
        np.savez(path, **arrays)
        del sample, arrays
        ctx = mp.get_context("spawn")
        barrier = ctx.Barrier(procs + 1)
        results = ctx.Queue()
        ps = [ctx.Process(target=_worker, args=(path, i, 1, barrier, results)) for i in range(procs)]
        for p in ps:
            p.start()
        barrier.wait(timeout=600)
        t0 = time.perf_counter()
        done = [results.get(timeout=900) for _ in ps]
        for p in ps:
            p.join(timeout=60)
        t1 = max(t for _, t, _ in done)
        nbytes = sum(b for _, _, b in done)
    finally:
        os.unlink(path)
    res["all_cores"] = {"seconds": t1 - t0, "bytes": nbytes, "units": procs, "threads": procs,
                        "what": f"{procs} (sequence, kv head) pairs of the long-context decode, 131072 tokens "
                                f"each, one per process on {procs} processes at once"}
    return res


def _decode(nsample: int, seed: int):
    import workloads
    import oracle
    wl = workloads.gqa_decode_batch(seed=seed)
    seqs = list(range(min(nsample, len(wl.seq_lens))))
    rows = np.concatenate([np.arange(wl.token_start[b], wl.token_start[b + 1]) for b in seqs])
    cache = np.zeros(oracle.cache_shape(wl.num_blocks, 16, wl.num_kv_heads, wl.head_size), np.uint8)
    t0 = time.perf_counter()
    oracle.write(wl.key[rows], wl.value[rows], wl.slot_mapping[rows], wl.signs, cache)
    oracle.paged_attention(wl.query, cache, wl.block_tables, wl.seq_lens, wl.query_start_loc, wl.softmax_scale,
                           wl.signs, seqs=seqs)
    dt = time.perf_counter() - t0
    rb = wl.head_size // 2 + 4
    kv = sum(int(wl.seq_lens[b]) for b in seqs) * 2 * wl.num_kv_heads * rb
    qo = len(seqs) * wl.num_q_heads * wl.head_size * 2 * 2
    return {"seconds": dt, "bytes": kv + qo, "units": len(seqs), "threads": 1,
            "what": f"{len(seqs)} of {len(wl.seq_lens)} sequences"}


def _write(ntok: int, seed: int):
    import workloads
    import oracle
    wl = workloads.write_throughput(seed=seed)
    n = min(ntok, wl.num_tokens)
    cache = np.zeros(oracle.cache_shape(wl.num_blocks, 16, wl.num_kv_heads, wl.head_size), np.uint8)
    t0 = time.perf_counter()
    oracle.write(wl.key[:n], wl.value[:n], wl.slot_mapping[:n], wl.signs, cache)
    dt = time.perf_counter() - t0
    per_tok = 2 * wl.num_kv_heads * wl.head_size * 2 + 2 * wl.num_kv_heads * (wl.head_size // 2 + 4) + 8
    return {"seconds": dt, "bytes": n * per_tok, "units": n, "threads": 1, "what": f"{n} of {wl.num_tokens} tokens"}


def main(argv):
    procs = 1
    if "--procs" in argv:
        i = argv.index("--procs")
        procs = int(argv[i + 1])
        argv = argv[:i] + argv[i + 2:]
    kind, n, seed = argv[0], int(argv[1]), int(argv[2])
    if kind == "long_decode":
        res = _long_decode(n, seed, procs)
    elif kind == "decode":
        res = _decode(n, seed)
    else:
        res = _write(n, seed)
    print(json.dumps(res))


if __name__ == "__main__":
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    main(sys.argv[1:])
