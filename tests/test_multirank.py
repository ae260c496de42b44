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


def _bench_env():
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR",
                                                            "MASTER_PORT")}
    env["OPENBLAS_NUM_THREADS"] = "1"
    return env


def test_gpus_flag_starts_local_ranks():
    # `bench.py --gpus 2` without an outer launcher starts two local ranks itself; the reference arm
    # runs on CPU (rank 0 times the oracle and prints the line, rank 1 exits 0)
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                          "--warmup", "3", "--ref-budget-s", "2"], cwd=root, env=_bench_env(), capture_output=True,
                         text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0


def test_gpus_flag_must_match_an_outer_launcher():
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(_bench_env(), WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, "bench.py", "--gpus", "2"], cwd=root, env=env, capture_output=True,
                         text=True, timeout=120)
    assert res.returncode == 2 and "WORLD_SIZE" in res.stderr
