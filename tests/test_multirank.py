"""The multi-GPU benchmark path on CPU: two gloo ranks, each timing its own replica; the job's
time is the slowest rank's and its value counts every rank's bytes.  (Every run here has one GPU:
the path shards without any exchange, so N GPUs run N independent replicas.)"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [3.0, 5.0][rank]
    ms = bench.max_over_ranks(local_ms, "cpu")
    val = bench.whole_job_gbs(1_000_000, world, ms)
    w, r, _ = bench._dist()
    q.put((rank, ms, val, w, r))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, val, w, r in res:
        assert ms == 5.0 and w == 2 and r == rank
        assert val == pytest.approx(2 * 1_000_000 / 5e-3 / 1e9)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(4.5, "cpu") == 4.5
    assert bench.whole_job_gbs(2_000_000, 1, 2.0) == pytest.approx(1.0)
