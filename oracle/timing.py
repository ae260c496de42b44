"""Time the oracle (as it stands) on a bounded sample of a workload; prints one JSON line.

TEST INFRASTRUCTURE: run by the benchmark's CPU-baseline leg and its reference arm, in a
subprocess whose BLAS threads the caller fixes through the environment.

  python -m oracle.timing decode <num_seqs_sample> <seed>   GQA decode batch, first sequences
  python -m oracle.timing write <num_tokens_sample> <seed>  write-throughput workload, first tokens

A decode sample = write every token of the sampled sequences into the oracle's cache, then run the
oracle attention for their queries.  The reported bytes are the packed-KV (+ Q/O) bytes the sample
covers, so ``bytes / seconds`` is in the benchmark's unit.
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np


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
    return {"seconds": dt, "bytes": kv + qo, "units": len(seqs), "what": f"{len(seqs)} of {len(wl.seq_lens)} sequences"}


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
    return {"seconds": dt, "bytes": n * per_tok, "units": n, "what": f"{n} of {wl.num_tokens} tokens"}


def main(argv):
    kind, n, seed = argv[0], int(argv[1]), int(argv[2])
    res = _decode(n, seed) if kind == "decode" else _write(n, seed)
    res["threads"] = int(os.environ.get("OPENBLAS_NUM_THREADS", "0") or 0) or os.cpu_count()
    print(json.dumps(res))


if __name__ == "__main__":
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    main(sys.argv[1:])
