"""Shared plumbing of the GPU parity tests: run a workload through the CUDA library and through the
oracle on the same seeded inputs, and compare.

Agreement bars:
  * cache bytes (codes and scale words): bit-exact;
  * attention outputs (compared in fp32 against the fp64 oracle):
    |gpu - oracle| <= 2e-3 + 1e-2 * |oracle| elementwise.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL = 2e-3
RTOL = 1e-2


def dev():
    return torch.device("cuda:0")


def gpu_cache(num_blocks, block_size, H, d, fill=0):
    import int4_token_head_kv_gb300 as kv
    return torch.full(kv.kv_int4_cache_shape(num_blocks, block_size, H, d), fill, dtype=torch.uint8, device=dev())


def gpu_write(wl_key, wl_value, slots, signs, cache, rows=None):
    """Write K/V rows (all, or the given row indices) with the CUDA kernel."""
    import int4_token_head_kv_gb300 as kv
    k, v = (wl_key, wl_value) if rows is None else (wl_key[rows], wl_value[rows])
    s = slots if rows is None else slots[rows]
    kv.kv_int4_write(k.to(dev()).contiguous(), v.to(dev()).contiguous(),
                     torch.from_numpy(np.ascontiguousarray(s)).to(dev()),
                     torch.from_numpy(signs).to(dev()), cache)


def oracle_cache(wl, rows=None, fill=0):
    cache = np.full(oracle.cache_shape(wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_size), fill, np.uint8)
    if rows is None:
        oracle.write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    else:
        oracle.write(wl.key[rows], wl.value[rows], wl.slot_mapping[rows], wl.signs, cache)
    return cache


def gpu_attention(wl, cache, out_dtype=torch.float32, segment_len=None):
    import int4_token_head_kv_gb300 as kv
    seg = wl.segment_len if segment_len is None else segment_len
    return kv.kv_int4_paged_attention(
        wl.query.to(dev()), cache, torch.from_numpy(wl.block_tables).to(dev()),
        torch.from_numpy(wl.seq_lens).to(dev()), torch.from_numpy(wl.query_start_loc).to(dev()),
        wl.softmax_scale, torch.from_numpy(wl.signs).to(dev()), max_query_len=wl.max_query_len,
        max_seq_len=wl.max_seq_len, out_dtype=out_dtype, segment_len=seg)


def oracle_attention(wl, cache, seqs=None, kv_heads=None):
    return oracle.paged_attention(wl.query, cache, wl.block_tables, wl.seq_lens, wl.query_start_loc,
                                  wl.softmax_scale, wl.signs, seqs=seqs, kv_heads=kv_heads)


def assert_attention_close(got, ref, what=""):
    got = got.detach().float().cpu().numpy().astype(np.float64) if isinstance(got, torch.Tensor) else got
    mask = ~np.isnan(ref)
    assert mask.any(), "nothing to compare"
    g, r = got[mask], ref[mask]
    excess = np.abs(g - r) - (ATOL + RTOL * np.abs(r))
    worst = int(np.argmax(excess))
    assert excess[worst] <= 0, (f"{what}: attention out of tolerance at {worst}: got {g[worst]:.6g} "
                                f"ref {r[worst]:.6g} (max abs err {np.abs(g - r).max():.3g})")
    return float(np.abs(g - r).max())


def status():
    import int4_token_head_kv_gb300 as kv
    return kv.kv_int4_read_device_status()


def clear_status():
    import int4_token_head_kv_gb300 as kv
    kv.kv_int4_clear_device_status()
    torch.cuda.synchronize()
