"""GPU parity of kv_int4_write against the oracle: the whole cache, byte for byte.

Shapes follow the pages' cache-write tests ("tests/quantization/test_per_token_kv_cache.py":
tokens {1, 7, 42} x kv heads {1, 4, 8} x head size {64, 128}, block 16, random slots; the
round-trip case; the negative-slot case) plus the write-throughput workload at full size and
edge cases of the quantiser (constant, one-signed, tiny, huge and tied vectors).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gpu_helpers import clear_status
    clear_status()


def _check_write(wl, fill=0):
    from gpu_helpers import gpu_cache, gpu_write
    H, d = wl.num_kv_heads, wl.head_size
    ref = np.full(oracle.cache_shape(wl.num_blocks, wl.block_size, H, d), fill, np.uint8)
    bad = oracle.write(wl.key, wl.value, wl.slot_mapping, wl.signs, ref)
    cache = gpu_cache(wl.num_blocks, wl.block_size, H, d, fill)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    got = cache.cpu().numpy()
    if not np.array_equal(got, ref):
        diff = np.argwhere(got != ref)
        raise AssertionError(f"{len(diff)} cache bytes differ; first at {diff[0].tolist()}: "
                             f"gpu {got[tuple(diff[0])]:#x} oracle {ref[tuple(diff[0])]:#x}")
    return bad


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("head_size", [64, 128])
@pytest.mark.parametrize("num_heads", [1, 4, 8])
@pytest.mark.parametrize("num_tokens", [1, 7, 42])
def test_write_page_shapes_bit_exact(num_tokens, num_heads, head_size, dtype):
    wl = workloads.random_write(num_tokens, num_heads, head_size, dtype=dtype, seed=0)
    _check_write(wl, fill=0xA5)   # canary: untouched slots must keep it


@pytest.mark.parametrize("num_heads", [2, 3, 16, 64])
def test_write_other_head_counts(num_heads):
    # up to 64 kv heads: 3 takes the general vector index, 16 the grouped bulk stores at their
    # limit, 64 the per-thread stores
    wl = workloads.random_write(37, num_heads, 128, seed=50 + num_heads)
    _check_write(wl, fill=0x5A)


@pytest.mark.parametrize("num_tokens", [1, 16])
def test_write_round_trip_shape(num_tokens):
    wl = workloads.random_write(num_tokens, 4, 128, seed=42, scale=0.5)
    wl.slot_mapping = np.arange(num_tokens, dtype=np.int64)
    _check_write(wl)


def test_negative_slots_skipped():
    wl = workloads.random_write(4, 2, 64, seed=1, num_blocks=2)
    wl.slot_mapping = np.array([0, -1, 1, -1], np.int64)
    _check_write(wl, fill=0x5A)


def test_out_of_range_slots_counted_not_written():
    from gpu_helpers import status
    wl = workloads.random_write(40, 8, 128, seed=2, num_blocks=4)
    wl.slot_mapping[3] = wl.num_blocks * wl.block_size       # one past the end
    wl.slot_mapping[9] = 10 ** 9
    bad = _check_write(wl, fill=0x33)
    assert bad == 2
    assert status()["slot_out_of_range"] == 2


def test_write_throughput_workload_full_size():
    wl = workloads.write_throughput()
    _check_write(wl)


def test_tiny_workload_cache():
    wl = workloads.tiny_write_decode()
    _check_write(wl)


def _edge_vectors(d):
    rng = np.random.default_rng(11)
    rows = [
        np.zeros(d), np.full(d, 3.0), np.full(d, -1e-3),          # constant (floored scale)
        np.abs(rng.standard_normal(d)) + 5.0,                     # all positive -> zp clamps
        -np.abs(rng.standard_normal(d)) - 5.0,                    # all negative
        rng.standard_normal(d) * 1e-30,                           # tiny (subnormal after rotation)
        rng.standard_normal(d) * 1e30,                            # huge (bf16 only)
        np.eye(d)[3] * 7.0,                                        # one-hot
        rng.integers(-8, 9, d).astype(np.float64),                # small integers: exact sums, ties
        np.where(np.arange(d) % 2 == 0, 1.0, -1.0),
        rng.standard_normal(d) * np.where(rng.random(d) < 0.05, 100.0, 1.0),   # outliers
    ]
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("head_size", [64, 128])
def test_quantiser_edge_cases(dtype, head_size):
    x = _edge_vectors(head_size)
    if dtype == torch.float16:
        x = np.clip(x, -60000, 60000)
    n = x.shape[0]
    k = torch.from_numpy(x).to(dtype).reshape(n, 1, head_size)
    v = torch.from_numpy(x[::-1].copy()).to(dtype).reshape(n, 1, head_size)
    wl = workloads.WriteWorkload("edge", k, v, np.arange(n, dtype=np.int64), 2, 16,
                                 workloads.splitmix64_signs(head_size))
    _check_write(wl)


def test_random_magnitudes_many_tokens():
    # 4096 tokens with per-token magnitudes spanning 1e-6 .. 1e6
    r = np.random.default_rng(5)
    T, H, d = 4096, 2, 128
    x = r.standard_normal((T, H, d)).astype(np.float32) * (10.0 ** r.uniform(-6, 6, (T, 1, 1))).astype(np.float32)
    k = torch.from_numpy(x).to(torch.bfloat16)
    v = torch.from_numpy(x[:, ::-1].copy()).to(torch.bfloat16)
    slots = r.permutation(T * 2)[:T].astype(np.int64)
    wl = workloads.WriteWorkload("mags", k, v, slots, T * 2 // 16, 16, workloads.splitmix64_signs(d))
    _check_write(wl)


def test_write_is_deterministic():
    from gpu_helpers import gpu_cache, gpu_write
    wl = workloads.random_write(300, 8, 128, seed=9)
    a = gpu_cache(wl.num_blocks, 16, 8, 128)
    b = gpu_cache(wl.num_blocks, 16, 8, 128)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, a)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, b)
    assert torch.equal(a, b)
