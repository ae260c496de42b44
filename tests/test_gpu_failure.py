"""Failure detection on the GPU without a fault: every pipeline wait in the kernels is bounded; a
wait that runs out is recorded in the device status counters and the kernel winds down.  The
diagnostic entry point makes one wait run out (a barrier nothing completes) and the test checks the
counter and that the device still computes correctly afterwards."""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def test_bounded_wait_records_timeout_and_device_stays_usable():
    import int4_token_head_kv_gb300 as kv
    from gpu_helpers import assert_attention_close, gpu_attention, gpu_cache, gpu_write, oracle_attention, \
        oracle_cache
    kv.kv_int4_clear_device_status()
    kv.kv_int4_selftest_wait_timeout(5_000_000)
    st = kv.kv_int4_read_device_status()
    assert st["wait_timeout"] == 1
    kv.kv_int4_clear_device_status()
    wl = workloads.tiny_write_decode()
    cache = gpu_cache(wl.num_blocks, 16, wl.num_kv_heads, wl.head_size)
    gpu_write(wl.key, wl.value, wl.slot_mapping, wl.signs, cache)
    out = gpu_attention(wl, cache)
    ref_cache = oracle_cache(wl)
    assert np.array_equal(cache.cpu().numpy(), ref_cache)
    assert_attention_close(out, oracle_attention(wl, ref_cache), "after timeout")
    assert not any(kv.kv_int4_read_device_status().values())
