"""GPU parity of kv_int8_write (the INT8 per-(token, head) comparator) against its oracle: the
whole cache, byte for byte, on the page-test shapes, the write-throughput workload at full size,
skipped and out-of-range slots, and quantiser edge cases (zero, constant, tiny, huge, exact ties)."""
import numpy as np
import pytest
import torch

from oracle import int8 as o8
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gpu_helpers import clear_status
    clear_status()


def _check(wl, fill=0):
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import dev
    H, d = wl.num_kv_heads, wl.head_size
    ref = np.full(o8.cache_shape(wl.num_blocks, wl.block_size, H, d), fill, np.uint8)
    bad = o8.write(wl.key, wl.value, wl.slot_mapping, ref)
    cache = torch.full(kv.kv_int8_cache_shape(wl.num_blocks, wl.block_size, H, d), fill, dtype=torch.uint8,
                       device=dev())
    kv.kv_int8_write(wl.key.to(dev()).contiguous(), wl.value.to(dev()).contiguous(),
                     torch.from_numpy(np.ascontiguousarray(wl.slot_mapping)).to(dev()), cache)
    got = cache.cpu().numpy()
    if not np.array_equal(got, ref):
        diff = np.argwhere(got != ref)
        raise AssertionError(f"{len(diff)} cache bytes differ; first at {diff[0].tolist()}: "
                             f"gpu {got[tuple(diff[0])]:#x} oracle {ref[tuple(diff[0])]:#x}")
    return bad


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("head_size", [64, 128])
@pytest.mark.parametrize("num_heads", [1, 2, 8])
@pytest.mark.parametrize("num_tokens", [1, 7, 42])
def test_int8_write_page_shapes_bit_exact(num_tokens, num_heads, head_size, dtype):
    wl = workloads.random_write(num_tokens, num_heads, head_size, dtype=dtype, seed=5)
    _check(wl, fill=0xA5)


def test_int8_write_throughput_workload_full_size():
    _check(workloads.write_throughput())


def test_int8_skipped_and_out_of_range_slots():
    from gpu_helpers import status
    wl = workloads.random_write(40, 8, 128, seed=6, num_blocks=4)
    wl.slot_mapping[3] = wl.num_blocks * wl.block_size
    wl.slot_mapping[9] = 10 ** 9
    wl.slot_mapping[11] = -1
    assert _check(wl, fill=0x33) == 2
    assert status()["slot_out_of_range"] == 2


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_int8_edge_vectors(dtype):
    d = 128
    rng = np.random.default_rng(7)
    rows = [np.zeros(d), np.full(d, 3.0), np.full(d, -1e-3), rng.standard_normal(d) * 1e-6,
            rng.standard_normal(d) * (1e4 if dtype == torch.float16 else 1e30),
            np.concatenate([[127.0], rng.integers(-126, 126, d - 1) + 0.5]),   # exact .5 ties at scale 1
            np.concatenate([[-254.0], np.arange(-63, 64)]),                       # scale 2: every x.5 tie
            np.eye(d)[5] * -9.0]
    x = np.stack(rows).astype(np.float32)
    T = x.shape[0]
    wl = workloads.random_write(T, 1, d, dtype=dtype, seed=8)
    wl.key = torch.from_numpy(x[:, None, :]).to(dtype)
    wl.value = torch.from_numpy(-x[:, None, :]).to(dtype)
    _check(wl, fill=0x11)
