"""Benchmark of the INT4 per-(token, head) KV cache on GB300; prints ONE JSON line (rank 0).

Headline: the long-context decode workload (8 sequences x 131072 tokens, 64 q / 8 kv heads, head
size 128, block 16, bf16 Student-t(3) K/V, randomly permuted blocks).  A step is one pass of the
whole hot path over one batch: write the step's 8 new tokens (one per sequence) into the paged
INT4 cache (rotation, quantisation, packing), then run causal paged attention of the 8 queries over
the whole cache (query rotation, split-KV walker, segment combine).

  value     packed-KV GB/s of the step: bytes of packed K/V rows (codes + scales) the attention
            reads, plus Q and O, per step, over the device-timed step (write included).  The cache
            (1.14 GB) is larger than L2, so no flush is needed between steps.
  e2e       the same bytes over a step timed through the public API from pinned host buffers: each
            step copies its new K/V, slots, queries and tables host->device (one copy of the packed
            step inputs) and its output device->host.  The copies run on two copy streams beside the
            compute (one CUDA graph per step), double-buffered as a serving loop runs them;
            serial_value keeps the in-order figure.
  roofline  the attention call (query rotation + walker + combine) timed back to back on its stream,
            algorithmic bytes per call over its CUDA-event time, against MEASURED_PEAKS.json's HBM
            copy bandwidth; ``traffic`` is the ncu DRAM byte count per call from profiles/traffic.json,
            null when the kernel sources changed since it was taken.
  cpu_baseline  the oracle on a bounded sample of the same workload: single-threaded, and on all host
            cores (one process per core).

Sub-objects (each with its own roofline): ``gqa_decode_batch`` (32 sequences, lengths U[512, 4096],
32 q / 8 kv heads, steps rotated over cache replicas larger than 2x L2), ``write`` (65536 tokens,
8 kv heads), ``mixed_prefill_decode`` (4 prefill chunks of 2048 queries over 4096 keys + 60 decode
sequences: whole-call HBM fraction and the prefill part's dense-equivalent TFLOP/s against the
measured bf16 tensor peak), ``int8_comparator`` (the INT8 per-(token, head) cache write on the
write workload, and INT4 vs INT8 decode on the long-context workload), ``int2_lloyd_max`` (the INT2
mode's write and long-context decode, timed the same way).

Runs as N independent replicas under torchrun (the path does not shard across GPUs; no collective on
the data path); ``--gpus N`` without torchrun starts the N local ranks itself.  ``--impl reference``
times the CPU oracle on a bounded sample of the headline workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import socket
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode attn packed-KV GB/s (% HBM peak) at 1 GB300; write tokens/s"
L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
CSRC = os.path.join(ROOT, "int4_token_head_kv_gb300", "csrc")


def _peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, source) from MEASURED_PEAKS.json, else the fallback figures."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def sources_sha() -> str:
    """Digest of the CUDA sources: a committed ncu traffic figure is valid only for this digest."""
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def _traffic(key):
    """DRAM bytes per launch from profiles/traffic.json when taken on the current sources, else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        e = t.get(key)
        if isinstance(e, dict) and e.get("sources_sha") == sources_sha():
            return e.get("bytes")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, polled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value (the slowest rank's time); identity on one process."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job GB/s: every rank processes its own replica of the workload each step."""
    return bytes_per_rank_step * world / (ms_per_step * 1e-3) / 1e9


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_local_ranks(nproc: int, argv) -> int:
    """Run this script as ``nproc`` local ranks under torch.distributed.run (rendezvous on 127.0.0.1)
    and return the launcher's exit code."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={nproc}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.abspath(__file__)] + list(argv)
    return subprocess.call(cmd, cwd=ROOT)


# ----------------------------------------------------------------------------------- GPU arm

def _timed(torch, stream, fn, n):
    """Device time (ms) of ``n`` calls of fn(i), CUDA events on the launching stream, synchronised on
    both sides."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def _write_history(torch, kv, wl, dev, signs, cache, rows):
    step = 1 << 18
    for r0 in range(0, len(rows), step):
        idx = rows[r0:r0 + step]
        kv.kv_int4_write(wl.key[idx].to(dev), wl.value[idx].to(dev),
                         torch.from_numpy(wl.slot_mapping[idx]).to(dev), signs, cache)


def _decode_setup(torch, kv, wl, dev, replicas):
    """Cache replicas holding every sequence's history, and the step's device inputs (one packed
    device buffer filled from one pinned host buffer)."""
    H, d = wl.num_kv_heads, wl.head_size
    signs = torch.from_numpy(wl.signs).to(dev)
    hist = wl.history_token_rows()
    new = wl.new_token_rows()
    caches = []
    for _ in range(replicas):
        c = torch.zeros(kv.kv_int4_cache_shape(wl.num_blocks, wl.block_size, H, d), dtype=torch.uint8, device=dev)
        _write_history(torch, kv, wl, dev, signs, c, hist)
        caches.append(c)
    parts = {
        "k": wl.key[new].contiguous(),
        "v": wl.value[new].contiguous(),
        "slots": torch.from_numpy(wl.slot_mapping[new].copy()),
        "q": wl.query.contiguous(),
        "tables": torch.from_numpy(wl.block_tables.copy()),
        "lens": torch.from_numpy(wl.seq_lens.copy()),
        "qsl": torch.from_numpy(wl.query_start_loc.copy()),
    }
    offs, total = {}, 0
    for k, v in parts.items():
        offs[k] = total
        total += (v.numel() * v.element_size() + 255) // 256 * 256
    host = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device=dev)
    devt = {}
    for k, v in parts.items():
        n = v.numel() * v.element_size()
        host[offs[k]:offs[k] + n].copy_(v.reshape(-1).view(torch.uint8))
        devt[k] = dev_buf[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
    dev_buf.copy_(host)
    devt["signs"] = signs
    devt["_buf"] = dev_buf
    return caches, host, devt


def _decode_steps(torch, kv, wl, dev, args, replicas, world, with_e2e=False, sample_clocks=False, local=0):
    """Time decode steps (write the step's new tokens + attention) on ``wl``: whole steps, the
    attention call alone, the eager loop, and (optionally) end to end from host buffers."""
    stream = torch.cuda.current_stream()
    H, d, Hq = wl.num_kv_heads, wl.head_size, wl.num_q_heads
    rb = kv.kv_int4_row_bytes(d)
    caches, host, t = _decode_setup(torch, kv, wl, dev, replicas)
    S = len(wl.seq_lens)
    seg = kv.kv_int4_attention_segment_len(S, wl.max_seq_len, args.segment_len)
    ws = torch.empty(max(1, kv.kv_int4_attention_workspace_bytes(Hq, H, d, S, wl.max_seq_len, seg)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((wl.query.shape[0], Hq, d), dtype=wl.query.dtype, device=dev)
    kv_bytes = int(wl.seq_lens.sum()) * 2 * H * rb
    qo_bytes = 2 * wl.query.numel() * wl.query.element_size()
    attn_bytes = kv_bytes + qo_bytes

    def write(i):
        kv.kv_int4_write(t["k"], t["v"], t["slots"], t["signs"], caches[i % replicas])

    def attend(i):
        kv.kv_int4_paged_attention(t["q"], caches[i % replicas], t["tables"], t["lens"], t["qsl"], wl.softmax_scale,
                                   t["signs"], max_query_len=1, max_seq_len=wl.max_seq_len, out=out,
                                   segment_len=seg, workspace=ws)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup):
        write(i)
        attend(i)
    torch.cuda.synchronize()
    # One CUDA graph per cache replica holding a whole step (write + attention) and one holding the
    # attention call alone: decode steps replay as graphs, as a serving loop runs them.
    step_graphs, attn_graphs = [], []
    for r in range(replicas):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            write(r)
            attend(r)
        step_graphs.append(g)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2):
            attend(r)
        attn_graphs.append(g2)
    for i in range(args.warmup):
        step_graphs[i % replicas].replay()
        attn_graphs[i % replicas].replay()
    sampler = ClockSampler(local) if sample_clocks else None
    if sampler:
        sampler.start()
        time.sleep(0.06)
    barrier()
    ms_step = _timed(torch, stream, lambda i: step_graphs[i % replicas].replay(), args.steps) / args.steps
    barrier()
    clocks = sampler.stop() if sampler else None
    ms_step = max_over_ranks(ms_step, dev)
    attn_ms = _timed(torch, stream, lambda i: attn_graphs[i % replicas].replay(), args.steps) / args.steps

    def eager(i):
        write(i)
        attend(i)
    eager_ms = _timed(torch, stream, eager, args.steps) / args.steps
    res = {"ms_step": ms_step, "attn_ms": attn_ms, "eager_ms": eager_ms, "clocks": clocks, "seg": seg,
           "nseg": -(-wl.max_seq_len // seg), "kv_bytes": kv_bytes, "qo_bytes": qo_bytes, "attn_bytes": attn_bytes,
           "cache_bytes": wl.num_blocks * 2 * 16 * H * rb, "replicas": replicas}
    if with_e2e:
        h2d = host.numel()
        host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        d2h = host_out.numel() * host_out.element_size()

        def e2e_step(i):
            t["_buf"].copy_(host, non_blocking=True)
            write(i)
            attend(i)
            host_out.copy_(out, non_blocking=True)

        e2e_eager_ms = _timed(torch, stream, e2e_step, args.steps) / args.steps
        e2e_graphs = []
        for r in range(replicas):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                e2e_step(r)
            e2e_graphs.append(g)
        for i in range(args.warmup):
            e2e_graphs[i % replicas].replay()
        barrier()
        e2e_serial_ms = _timed(torch, stream, lambda i: e2e_graphs[i % replicas].replay(), args.steps) / args.steps
        barrier()
        del e2e_graphs
        e2e_ms = _pipelined_e2e(torch, kv, wl, t, caches, replicas, seg, ws, out, host, args, barrier)
        res.update(e2e_ms=max_over_ranks(e2e_ms, dev), e2e_serial_ms=max_over_ranks(e2e_serial_ms, dev),
                   e2e_eager_ms=e2e_eager_ms, h2d=h2d, d2h=d2h)
    del caches, ws, t
    torch.cuda.empty_cache()
    return res


def _pipelined_e2e(torch, kv, wl, t, caches, replicas, seg, ws, out, host, args, barrier):
    """End-to-end steps as a serving loop runs them: the inputs of a step go up on one copy stream and
    the output of the step before comes back on another while the current step computes (two device
    input buffers and two output buffers, pinned host buffers, the compute of each step one CUDA
    graph).  Every step's upload and read-back lies inside the timed region, which ends when the last
    read-back has landed.  Returns ms per step."""
    dev = out.device
    compute = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    base = t["_buf"]
    bufs = [base, torch.empty_like(base)]
    names = ("k", "v", "slots", "q", "tables", "lens", "qsl")
    views = []
    for b in bufs:
        vw = {}
        for n in names:
            off = t[n].data_ptr() - base.data_ptr()
            nb = t[n].numel() * t[n].element_size()
            vw[n] = b[off:off + nb].view(t[n].dtype).view(t[n].shape)
        views.append(vw)
    outs = [out, torch.empty_like(out)]
    host_outs = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    bufs[1].copy_(host)
    torch.cuda.synchronize()

    def step(r, b):
        v = views[b]
        kv.kv_int4_write(v["k"], v["v"], v["slots"], t["signs"], caches[r])
        kv.kv_int4_paged_attention(v["q"], caches[r], v["tables"], v["lens"], v["qsl"], wl.softmax_scale, t["signs"],
                                   max_query_len=1, max_seq_len=wl.max_seq_len, out=outs[b], segment_len=seg,
                                   workspace=ws)

    graphs = {}
    for r in range(replicas):
        for b in range(2):
            step(r, b)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(r, b)
            graphs[r, b] = g
    ev = lambda: torch.cuda.Event()   # noqa: E731
    uploaded, computed, landed = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(n, timed):
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if timed:
            start.record(compute)
        up.wait_stream(compute)
        down.wait_stream(compute)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(computed[b])          # step i - 2 has read input buffer b
                bufs[b].copy_(host, non_blocking=True)
                uploaded[b].record(up)
            compute.wait_event(uploaded[b])
            if i >= 2:
                compute.wait_event(landed[b])           # step i - 2's output has left buffer b
            graphs[i % replicas, b].replay()
            computed[b].record(compute)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                host_outs[b].copy_(outs[b], non_blocking=True)
                landed[b].record(down)
        compute.wait_stream(up)
        compute.wait_stream(down)
        if timed:
            end.record(compute)
        return start, end

    run(max(3, args.warmup), False)
    barrier()
    start, end = run(args.steps, True)
    end.synchronize()
    ms = start.elapsed_time(end) / args.steps
    barrier()
    del graphs
    return ms


def _gbs(nbytes, ms):
    return nbytes / (ms * 1e-3) / 1e9


def _roof(achieved, peak, kind, traffic, **extra):
    d = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
         "traffic": traffic, "peak_source": kind + " (MEASURED_PEAKS.json hbm_gbs)" if kind == "measured" else kind}
    d.update(extra)
    return d


def _gpu_arm(args):
    import torch

    import int4_token_head_kv_gb300 as kv
    import workloads

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    hbm, bf16, kind = _peaks()

    # ---- headline: long-context decode steps
    wl = workloads.long_context_decode(seed=args.seed)
    r = _decode_steps(torch, kv, wl, dev, args, replicas=1, world=world, with_e2e=True, sample_clocks=True,
                      local=local)
    attn_bytes = r["attn_bytes"]
    value = whole_job_gbs(attn_bytes, world, r["ms_step"])
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(r["ms_step"], 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4-kv/f16-mma/f32", "data": "synthetic",
        "config": {"workload": "long_context_decode: 8 seqs x 131072 tokens, 64 q / 8 kv heads, head 128, block 16, "
                               "bf16 Student-t(3) K/V, N(0,1) Q, permuted blocks; step = write 8 new tokens + "
                               "decode attention",
                   "segment_len": r["seg"], "segments_per_seq": r["nseg"], "packed_kv_bytes_per_step": r["kv_bytes"],
                   "qo_bytes_per_step": r["qo_bytes"],
                   "l2": f"inputs larger than L2 (cache {r['cache_bytes'] / 2**20:.0f} MiB > 129 MB)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": "steps replayed as one CUDA graph per step (write + attention)",
                   "eager_ms_per_step": round(r["eager_ms"], 5),
                   "eager_value": round(_gbs(attn_bytes * world, r["eager_ms"]), 2)},
        "e2e": {"value": round(_gbs(attn_bytes * world, r["e2e_ms"]), 2), "unit": "GB/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": round(r["e2e_ms"], 5),
                "serial_ms_per_step": round(r["e2e_serial_ms"], 5),
                "serial_value": round(_gbs(attn_bytes * world, r["e2e_serial_ms"]), 2),
                "timing": "serving loop: each step's packed inputs uploaded and the previous step's output read "
                          "back on two copy streams while the step (write + attention, one CUDA graph) computes; "
                          "double-buffered pinned host and device buffers; every copy inside the timed region. "
                          "serial_*: upload, write, attention and read-back in order in one graph per step",
                "eager_ms_per_step": round(r["e2e_eager_ms"], 5),
                "eager_value": round(_gbs(attn_bytes * world, r["e2e_eager_ms"]), 2)},
        "roofline": _roof(_gbs(attn_bytes, r["attn_ms"]), hbm, kind, _traffic("long_context_decode"),
                          kernel="attention call (query rotation + split-KV walker + combine), graph-replayed "
                                 "back to back", bytes_per_launch=attn_bytes, avg_ms=round(r["attn_ms"], 5)),
        "gpu_launches": 4 * args.steps,
        "clocks": r["clocks"],
    }
    del wl

    # ---- sub-objects (rank-local figures)
    if not args.headline_only:
        result["gqa_decode_batch"] = _gqa_bench(torch, kv, workloads, dev, args, world, hbm, kind)
        result["write"] = _write_bench(torch, kv, workloads, dev, args, hbm, kind)
        result["mixed_prefill_decode"] = _mixed_bench(torch, kv, workloads, dev, args, hbm, bf16, kind)
        result["int8_comparator"] = _int8_write_bench(torch, kv, workloads, dev, args, hbm)
        result["int8_comparator"]["decode"] = _int8_decode_bench(torch, kv, workloads, dev, args, hbm)
        result["int2_lloyd_max"] = _int2_bench(torch, kv, workloads, dev, args, hbm)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = _cpu_baseline(args)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def _gqa_bench(torch, kv, workloads, dev, args, world, hbm, kind):
    wl = workloads.gqa_decode_batch(seed=args.seed)
    rb = kv.kv_int4_row_bytes(wl.head_size)
    cache_bytes = wl.num_blocks * 2 * 16 * wl.num_kv_heads * rb
    replicas = max(2, -(-2 * L2_BYTES // cache_bytes))
    r = _decode_steps(torch, kv, wl, dev, args, replicas=replicas, world=world)
    return {"workload": "gqa_decode_batch: 32 seqs, seq_len U[512,4096] (sum %d), 32 q / 8 kv heads, head 128, "
                        "block 16, bf16 N(0,1) with 4 K channels x10 per kv head, permuted blocks; step = write 32 "
                        "new tokens + decode attention" % int(wl.seq_lens.sum()),
            "GB/s": round(_gbs(r["attn_bytes"], r["ms_step"]), 2), "ms_per_step": round(r["ms_step"], 5),
            "segment_len": r["seg"], "bytes_per_step": r["attn_bytes"],
            "l2": f"{replicas} cache replicas rotated per step ({replicas * cache_bytes / 2**20:.0f} MiB > 2 x 129 MB)",
            "roofline": _roof(_gbs(r["attn_bytes"], r["attn_ms"]), hbm, kind, _traffic("gqa_decode_batch"),
                              kernel="attention call, graph-replayed back to back over the replicas",
                              bytes_per_launch=r["attn_bytes"], avg_ms=round(r["attn_ms"], 5))}


def _write_bench(torch, kv, workloads, dev, args, hbm, kind):
    wl = workloads.write_throughput(seed=args.seed)
    H, d = wl.num_kv_heads, wl.head_size
    signs = torch.from_numpy(wl.signs).to(dev)
    k, v = wl.key.to(dev), wl.value.to(dev)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    cache = torch.zeros(kv.kv_int4_cache_shape(wl.num_blocks, 16, H, d), dtype=torch.uint8, device=dev)
    per_tok = 2 * H * d * k.element_size() + 2 * H * kv.kv_int4_row_bytes(d) + 8
    nbytes = wl.num_tokens * per_tok
    reps = max(50, min(2000, args.steps))
    for _ in range(max(3, args.warmup)):
        kv.kv_int4_write(k, v, slots, signs, cache)
    ms = _timed(torch, torch.cuda.current_stream(), lambda i: kv.kv_int4_write(k, v, slots, signs, cache), reps) / reps
    gbs = _gbs(nbytes, ms)
    return {"workload": "write_throughput: 65536 tokens, 8 kv heads, head 128, bf16, magnitudes 10^U(-2,2), "
                        "random slots over 8192 blocks of 16 (inputs 268 MB > L2)",
            "tokens_per_s": round(wl.num_tokens / (ms * 1e-3), 1), "GB/s": round(gbs, 1), "ms_per_call": round(ms, 5),
            "bytes_per_call": nbytes, "launches": reps,
            "roofline": _roof(gbs, hbm, kind, _traffic("write_throughput"), kernel="write_kernel",
                              bytes_per_launch=nbytes, avg_ms=round(ms, 5))}


def _attention_calls(torch, kv, wl, dev, reps, rows=None, segment_len=0, sub=None, bits=4):
    """Write every token of ``wl`` (untimed), then time ``reps`` back-to-back attention calls captured in
    one CUDA graph, over the whole batch or over the sequences ``sub`` (same cache).  Returns ms per call
    and the segment length.  bits=8 / 2: the INT8 comparator's or the INT2 mode's cache and decode call
    instead."""
    H, d = wl.num_kv_heads, wl.head_size
    signs = torch.from_numpy(wl.signs).to(dev)
    import numpy as np
    if bits == 4:
        cache = torch.zeros(kv.kv_int4_cache_shape(wl.num_blocks, 16, H, d), dtype=torch.uint8, device=dev)
        _write_history(torch, kv, wl, dev, signs, cache, np.arange(wl.key.shape[0]))
        row_bytes = kv.kv_int4_row_bytes(d)
    else:
        shape, write, row_bytes = ((kv.kv_int8_cache_shape, kv.kv_int8_write, kv.kv_int8_row_bytes(d)) if bits == 8
                                   else (kv.kv_int2_cache_shape, kv.kv_int2_write, kv.kv_int2_row_bytes(d)))
        cache = torch.zeros(shape(wl.num_blocks, 16, H, d), dtype=torch.uint8, device=dev)
        step = 1 << 18
        for r0 in range(0, wl.key.shape[0], step):
            extra = () if bits == 8 else (signs,)
            write(wl.key[r0:r0 + step].to(dev), wl.value[r0:r0 + step].to(dev),
                  torch.from_numpy(wl.slot_mapping[r0:r0 + step]).to(dev), *extra, cache)
    results = {}
    for name, seqs in (sub or {"all": None}).items():
        if seqs is None:
            seqs = list(range(len(wl.seq_lens)))
        qrows = np.concatenate([np.arange(wl.query_start_loc[b], wl.query_start_loc[b + 1]) for b in seqs])
        q = wl.query[qrows].to(dev)
        lens_np = wl.seq_lens[seqs]
        qlens = wl.query_lens[seqs]
        qsl = torch.from_numpy(np.concatenate([[0], np.cumsum(qlens)]).astype(np.int32)).to(dev)
        tables, lens = torch.from_numpy(wl.block_tables[seqs].copy()).to(dev), torch.from_numpy(lens_np).to(dev)
        max_len, max_q = int(lens_np.max()), int(qlens.max())
        seg = kv.kv_int4_attention_segment_len(len(seqs), max_len, segment_len)
        ws = torch.empty(max(1, kv.kv_int4_attention_workspace_bytes(wl.num_q_heads, H, d, len(seqs), max_len, seg)),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(q)

        def call():
            if bits == 4:
                kv.kv_int4_paged_attention(q, cache, tables, lens, qsl, wl.softmax_scale, signs, max_query_len=max_q,
                                           max_seq_len=max_len, out=out, segment_len=seg, workspace=ws)
            elif bits == 8:
                kv.kv_int8_paged_attention(q, cache, tables, lens, qsl, wl.softmax_scale, max_query_len=max_q,
                                           max_seq_len=max_len, out=out, segment_len=seg, workspace=ws)
            else:
                kv.kv_int2_paged_attention(q, cache, tables, lens, qsl, wl.softmax_scale, signs, max_query_len=max_q,
                                           max_seq_len=max_len, out=out, segment_len=seg, workspace=ws)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(reps):
                call()
        g.replay()
        ms = _timed(torch, torch.cuda.current_stream(), lambda i: g.replay(), 1) / reps
        kvb = int(lens_np.sum()) * 2 * H * row_bytes + 2 * q.numel() * q.element_size()
        results[name] = {"ms": ms, "seg": seg, "bytes": kvb, "seqs": seqs, "qlens": qlens, "lens": lens_np}
        del g, ws, out, q
    del cache
    torch.cuda.empty_cache()
    return results


def _prefill_flops(res, num_q_heads, d):
    """Dense-equivalent attention FLOPs of the prefill chunks: 4 d per visible (query, key) pair per q head."""
    pairs = sum(int(q) * (int(L) - int(q)) + int(q) * (int(q) + 1) // 2
                for L, q in zip(res["lens"], res["qlens"]) if q > 1)
    return 4 * d * pairs * num_q_heads


def _mixed_bench(torch, kv, workloads, dev, args, hbm, bf16, kind):
    wl = workloads.mixed_prefill_decode(seed=args.seed)
    nseq = len(wl.seq_lens)
    pre = [b for b in range(nseq) if wl.query_lens[b] > 1]
    dec = [b for b in range(nseq) if wl.query_lens[b] == 1]
    reps = 10
    res = _attention_calls(torch, kv, wl, dev, reps, sub={"all": None, "prefill": pre, "decode": dec})
    a, p, dd = res["all"], res["prefill"], res["decode"]
    flops = _prefill_flops(p, wl.num_q_heads, wl.head_size)
    tfs = flops / (p["ms"] * 1e-3) / 1e12
    return {"workload": "mixed_prefill_decode: 4 prefill seqs (2048 cached + 2048-query causal chunk) + 60 decode "
                        "seqs U[1,32768], 32 q / 8 kv heads, head 128, bf16 N(0,1); one attention call over the batch",
            "ms_per_call": round(a["ms"], 4), "GB/s": round(_gbs(a["bytes"], a["ms"]), 1), "bytes_per_call": a["bytes"],
            "segment_len": a["seg"],
            "roofline": _roof(_gbs(a["bytes"], a["ms"]), hbm, kind, _traffic("mixed_prefill_decode"),
                              kernel="whole attention call (decode kernels + prefill kernel), graph-replayed",
                              bytes_per_launch=a["bytes"], avg_ms=round(a["ms"], 4)),
            "prefill_part": {"ms": round(p["ms"], 4), "dense_equiv_TFLOP": round(flops / 1e12, 4),
                             "roofline": {"bound": "tensor", "achieved": round(tfs, 1), "peak": bf16,
                                          "unit": "TFLOP/s", "frac": round(tfs / bf16, 4), "traffic": None,
                                          "peak_source": "MEASURED_PEAKS.json bf16_tflops (burst; fp16 and bf16 "
                                                         "dense rates are equal)" if kind == "measured" else kind,
                                          "kernel": "prefill_kernel on the 4 prefill sequences alone"}},
            "decode_part": {"ms": round(dd["ms"], 4), "GB/s": round(_gbs(dd["bytes"], dd["ms"]), 1),
                            "frac": round(_gbs(dd["bytes"], dd["ms"]) / hbm, 4), "segment_len": dd["seg"]}}


def _int8_write_bench(torch, kv, workloads, dev, args, hbm):
    """The INT8 per-(token, head) comparator's write on the same workload (cache rows d + 4 bytes)."""
    wl = workloads.write_throughput(seed=args.seed)
    H, d = wl.num_kv_heads, wl.head_size
    k, v = wl.key.to(dev), wl.value.to(dev)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    cache = torch.zeros(kv.kv_int8_cache_shape(wl.num_blocks, 16, H, d), dtype=torch.uint8, device=dev)
    nbytes = wl.num_tokens * (2 * H * d * k.element_size() + 2 * H * kv.kv_int8_row_bytes(d) + 8)
    reps = max(50, min(2000, args.steps))
    for _ in range(5):
        kv.kv_int8_write(k, v, slots, cache)
    ms = _timed(torch, torch.cuda.current_stream(), lambda i: kv.kv_int8_write(k, v, slots, cache), reps) / reps
    gbs = _gbs(nbytes, ms)
    return {"write": {"tokens_per_s": round(wl.num_tokens / (ms * 1e-3), 1), "GB/s": round(gbs, 1),
                      "frac": round(gbs / hbm, 4), "ms_per_call": round(ms, 5), "bytes_per_call": nbytes},
            "cache_bytes_per_token": 2 * H * kv.kv_int8_row_bytes(d),
            "int4_cache_bytes_per_token": 2 * H * kv.kv_int4_row_bytes(d)}


def _int8_decode_bench(torch, kv, workloads, dev, args, hbm):
    """INT4 and INT8 decode attention on the long-context workload, timed the same way (one CUDA graph
    of back-to-back calls over a cache larger than L2) on the same box."""
    wl = workloads.long_context_decode(seed=args.seed)
    reps = 50
    res = {}
    for bits in (4, 8):
        r = _attention_calls(torch, kv, wl, dev, reps=reps, segment_len=args.segment_len, bits=bits)["all"]
        rb = kv.kv_int4_row_bytes(wl.head_size) if bits == 4 else kv.kv_int8_row_bytes(wl.head_size)
        gbs = _gbs(r["bytes"], r["ms"])
        res[f"int{bits}"] = {"ms_per_call": round(r["ms"], 5), "GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                             "decode_tokens_per_s": round(len(wl.seq_lens) / (r["ms"] * 1e-3), 1),
                             "context_tokens_per_s": round(float(wl.seq_lens.sum()) / (r["ms"] * 1e-3), 1),
                             "kv_bytes_per_token_per_layer": 2 * wl.num_kv_heads * rb, "segment_len": r["seg"]}
    res["workload"] = ("long_context_decode: 8 seqs x 131072 tokens, 64 q / 8 kv heads, head 128; one decode "
                       "attention call per step (no write), graph-replayed %d times back to back" % reps)
    res["int8_over_int4_time"] = round(res["int8"]["ms_per_call"] / res["int4"]["ms_per_call"], 3)
    res["int4_kv_bytes_saving_vs_int8"] = round(1 - res["int4"]["kv_bytes_per_token_per_layer"] /
                                                res["int8"]["kv_bytes_per_token_per_layer"], 4)
    return res


def _int2_bench(torch, kv, workloads, dev, args, hbm):
    """The INT2 Lloyd-Max mode: its write on the write-throughput workload and its decode attention on
    the long-context workload, timed as the INT4 and INT8 figures are."""
    wl = workloads.write_throughput(seed=args.seed)
    H, d = wl.num_kv_heads, wl.head_size
    k, v = wl.key.to(dev), wl.value.to(dev)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    signs = torch.from_numpy(wl.signs).to(dev)
    cache = torch.zeros(kv.kv_int2_cache_shape(wl.num_blocks, 16, H, d), dtype=torch.uint8, device=dev)
    nbytes = wl.num_tokens * (2 * H * d * k.element_size() + 2 * H * kv.kv_int2_row_bytes(d) + 8)
    reps = max(50, min(2000, args.steps))
    for _ in range(5):
        kv.kv_int2_write(k, v, slots, signs, cache)
    ms = _timed(torch, torch.cuda.current_stream(), lambda i: kv.kv_int2_write(k, v, slots, signs, cache), reps) / reps
    gbs = _gbs(nbytes, ms)
    res = {"write": {"tokens_per_s": round(wl.num_tokens / (ms * 1e-3), 1), "GB/s": round(gbs, 1),
                     "frac": round(gbs / hbm, 4), "ms_per_call": round(ms, 5), "bytes_per_call": nbytes,
                     "workload": "write_throughput: 65536 tokens, 8 kv heads, head 128, bf16"},
           "cache_bytes_per_token": 2 * H * kv.kv_int2_row_bytes(d)}
    del k, v, cache
    wl = workloads.long_context_decode(seed=args.seed)
    reps = 50
    r = _attention_calls(torch, kv, wl, dev, reps=reps, segment_len=args.segment_len, bits=2)["all"]
    gbs = _gbs(r["bytes"], r["ms"])
    res["decode"] = {"ms_per_call": round(r["ms"], 5), "GB/s": round(gbs, 1), "frac": round(gbs / hbm, 4),
                     "decode_tokens_per_s": round(len(wl.seq_lens) / (r["ms"] * 1e-3), 1),
                     "context_tokens_per_s": round(float(wl.seq_lens.sum()) / (r["ms"] * 1e-3), 1),
                     "kv_bytes_per_token_per_layer": 2 * wl.num_kv_heads * kv.kv_int2_row_bytes(wl.head_size),
                     "segment_len": r["seg"],
                     "workload": "long_context_decode: 8 seqs x 131072 tokens, 64 q / 8 kv heads, head 128; one "
                                 "decode attention call per step, graph-replayed %d times back to back" % reps}
    return res


# ------------------------------------------------------------------------------- CPU oracle

def _oracle_timing(argv):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    res = subprocess.run([sys.executable, "-m", "oracle.timing"] + argv, cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=1200)
    if res.returncode != 0:
        raise RuntimeError(res.stderr[-600:])
    return json.loads(res.stdout.strip().splitlines()[-1])


def _cpu_baseline(args):
    """The oracle on a bounded sample of the headline workload: single-threaded (a few (sequence,
    kv head) pairs) and on all host cores (one process per core, one pair each)."""
    ncpu = os.cpu_count() or 1
    try:
        r = _oracle_timing(["long_decode", str(args.cpu_pairs), str(args.seed), "--procs", str(ncpu)])
    except Exception as e:   # report, do not fail the GPU measurement
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "error": str(e)[-400:]}
    one = r["single"]
    out = {"value": round(one["bytes"] / one["seconds"] / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": one["what"] + f"; {one['seconds']:.1f} s", "nproc": ncpu}
    if "all_cores" in r:
        a = r["all_cores"]
        out["all_cores"] = {"value": round(a["bytes"] / a["seconds"] / 1e9, 6), "unit": "GB/s", "cores": a["threads"],
                            "kind": "oracle", "sample": a["what"] + f"; {a['seconds']:.1f} s wall"}
    return out


def _reference_arm(args):
    """The CPU oracle, as it stands, on the GPU arm's headline workload and metric.  Each step is a
    bounded sample: one (sequence, kv head) pair of the long-context decode batch, round-robin,
    truncated to its first n tokens so that warm-up + steps take about ``--ref-budget-s`` seconds
    whatever --steps is.  A step writes the sample's tokens into the oracle's cache and runs the oracle
    attention for that kv head's query heads; its bytes are the packed K/V rows (+ Q/O) it covers."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np

    import oracle
    import workloads

    t_start = time.perf_counter()
    wl = workloads.long_context_decode(seed=args.seed)
    S, H, G, d = len(wl.seq_lens), wl.num_kv_heads, wl.num_q_heads // wl.num_kv_heads, wl.head_size
    rb = d // 2 + 4

    def one(i, ntok):
        b, h = i % S, (i // S) % H
        L = min(int(wl.seq_lens[b]), ntok)
        rows = slice(int(wl.token_start[b]), int(wl.token_start[b]) + L)
        nb = (L + 15) // 16
        table = np.arange(nb, dtype=np.int32)[None]
        cache = np.zeros(oracle.cache_shape(nb, 16, 1, d), np.uint8)
        k, v = wl.key[rows, h:h + 1], wl.value[rows, h:h + 1]
        q = wl.query[b:b + 1, h * G:(h + 1) * G]
        t0 = time.perf_counter()
        oracle.write(k, v, np.arange(L, dtype=np.int64), wl.signs, cache)
        oracle.paged_attention(q, cache, table, np.array([L], np.int32), np.array([0, 1], np.int32),
                               wl.softmax_scale, wl.signs)
        return time.perf_counter() - t0, L * 2 * rb + 2 * G * d * 2

    dt, _ = one(0, 4096)
    per_tok = dt / 4096
    budget = args.ref_budget_s / max(1, args.steps + args.warmup)
    ntok = int(max(16, min(int(wl.seq_lens[0]), budget / max(per_tok, 1e-9))))
    for i in range(args.warmup):
        one(i, ntok)
    secs, nbytes = 0.0, 0
    for i in range(args.steps):
        s_, b_ = one(i, ntok)
        secs += s_
        nbytes += b_
    value = nbytes / secs / 1e9
    sample = f"1 (sequence, kv head) pair of the long-context decode batch per step, first {ntok} tokens, round-robin"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 write / f64 attention",
            "data": "synthetic",
            "config": {"workload": "long_context_decode (the GPU arm's headline workload); oracle on a bounded "
                                   "sample per step", "sample_tokens": ntok},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - t_start, 2)}
    print(json.dumps(line))


def _only(args):
    """One workload's attention call (or the write), timed as in the sub-objects, on its own: a small
    program for profiling one kernel."""
    import torch

    import int4_token_head_kv_gb300 as kv
    import workloads

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    hbm, _, _ = _peaks()
    if args.only == "write_throughput":
        r = _write_bench(torch, kv, workloads, dev, args, hbm, "measured")
        print(json.dumps({"only": args.only, "ms": r["ms_per_call"], "GB/s": r["GB/s"]}))
        return
    wl = getattr(workloads, args.only)(seed=args.seed)
    res = _attention_calls(torch, kv, wl, dev, reps=args.steps, segment_len=args.segment_len)["all"]
    print(json.dumps({"only": args.only, "ms": round(res["ms"], 4), "GB/s": round(_gbs(res["bytes"], res["ms"]), 1),
                      "frac": round(_gbs(res["bytes"], res["ms"]) / hbm, 4), "bytes": res["bytes"],
                      "segment_len": res["seg"]}))


def main(argv=None):
    argv = sys.argv[1:] if argv is None else argv
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--segment-len", type=int, default=0,
                    help="split-KV segment length in tokens (multiple of 16); 0 = the library's choice")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--headline-only", action="store_true", help="skip the sub-object workloads")
    ap.add_argument("--cpu-pairs", type=int, default=8,
                    help="(sequence, kv head) pairs in the single-threaded oracle sample")
    ap.add_argument("--ref-budget-s", type=float, default=120.0,
                    help="reference arm: seconds of oracle work over warm-up + steps")
    ap.add_argument("--only", choices=["long_context_decode", "mixed_prefill_decode", "gqa_decode_batch",
                                       "write_throughput"],
                    help="time just this workload's attention call (or the write) and print its own line")
    args = ap.parse_args(argv)
    world = os.environ.get("WORLD_SIZE")
    if world is None and args.gpus > 1:
        return launch_local_ranks(args.gpus, argv)
    if world is not None and int(world) != args.gpus:
        print(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
        return 2
    if args.only:
        _only(args)
        return 0
    if args.impl == "reference":
        # the oracle runs single-threaded; fix BLAS threads before numpy loads
        for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        _reference_arm(args)
    else:
        _gpu_arm(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
