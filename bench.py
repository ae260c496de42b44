"""Benchmark of the INT4 per-(token, head) KV cache on GB300; prints ONE JSON line (rank 0).

A step is one pass of the whole hot path over one batch of the GQA decode workload
(32 sequences with lengths uniform in [512, 4096], 32 q / 8 kv heads, head size 128, block 16,
bf16, 4 loud K channels per kv head): write the step's 32 new tokens into the paged INT4 cache
(rotation, quantisation, packing), then run causal paged attention of the 32 queries over the
whole cache.

  value   packed-KV GB/s of the decode step: bytes of packed K/V rows (codes + scales) the
          attention reads, plus Q and O, per step, over the device-timed step (write included).
  e2e     the same bytes over a step timed through the public API from pinned host buffers:
          each step copies its new K/V, slots, queries and tables host->device (one copy of the
          packed step inputs) and the output device->host; the step (copies included) is replayed
          as a CUDA graph, as a serving loop runs decode steps (the eager Python loop is reported
          beside it).
  write   the write-throughput workload (65536 tokens, 8 kv heads, d 128, bf16, per-token
          magnitudes 10^U(-2,2), random slots over 8192 blocks): tokens/s and GB/s.
  roofline  for the dominant kernel call (the attention: query rotation + decode kernel + segment combine), bytes
          per launch over its CUDA-event time on the launching stream, against the measured HBM
          copy bandwidth; ``traffic`` is the ncu DRAM byte count of the decode kernel when a
          summary with it is committed under profiles/, else null.

L2 (129 MB) is defeated by rotating the steps over several independent cache replicas whose total
exceeds twice the L2 size.  Runs as N independent replicas under torchrun (the path does not
shard across GPUs; each rank runs the same workload, no collective on the data path).
``--impl reference`` times the CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
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


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary (profiles/traffic.json), if present."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)
        return t.get(kernel_key)
    except Exception:
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


# ----------------------------------------------------------------------------------- GPU arm

def _decode_setup(torch, kv, wl, dev, replicas):
    """Cache replicas holding every sequence's history, and the step's device inputs."""
    H, d = wl.num_kv_heads, wl.head_size
    signs = torch.from_numpy(wl.signs).to(dev)
    hist = wl.history_token_rows()
    new = wl.new_token_rows()
    caches = []
    for _ in range(replicas):
        c = torch.zeros(kv.kv_int4_cache_shape(wl.num_blocks, wl.block_size, H, d), dtype=torch.uint8, device=dev)
        kv.kv_int4_write(wl.key[hist].to(dev), wl.value[hist].to(dev),
                         torch.from_numpy(wl.slot_mapping[hist]).to(dev), signs, c)
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
    # A step's inputs live in one pinned host buffer and one device buffer (256-byte aligned
    # slices), so a step uploads them with a single copy.
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
    stream = torch.cuda.current_stream()

    wl = workloads.gqa_decode_batch(seed=args.seed)
    H, d, Hq = wl.num_kv_heads, wl.head_size, wl.num_q_heads
    rb = kv.kv_int4_row_bytes(d)
    cache_bytes = wl.num_blocks * 2 * 16 * H * rb
    replicas = max(2, -(-2 * L2_BYTES // cache_bytes))
    caches, host, t = _decode_setup(torch, kv, wl, dev, replicas)
    seg = kv.kv_int4_attention_segment_len(len(wl.seq_lens), wl.max_seq_len, args.segment_len)
    nseg = -(-wl.max_seq_len // seg)
    ws = torch.empty(max(1, kv.kv_int4_attention_workspace_bytes(Hq, H, d, len(wl.seq_lens), wl.max_seq_len, seg)),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((wl.query.shape[0], Hq, d), dtype=wl.query.dtype, device=dev)
    kv_bytes = int(wl.seq_lens.sum()) * 2 * H * rb
    qo_bytes = 2 * wl.query.numel() * wl.query.element_size()
    attn_bytes = kv_bytes + qo_bytes
    launches_per_step = 4   # write; query rotation; split-KV walker; combine

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
    # One CUDA graph per cache replica holding one whole step (write + attention), and one holding
    # the attention call alone; decode steps are replayed as graphs, which takes the Python and
    # launch overhead of the four kernel launches per step off the GPU's critical path.
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
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # ---- device-timed steps (the headline)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.06)
    barrier()
    e0.record(stream)
    for i in range(args.steps):
        step_graphs[i % replicas].replay()
    e1.record(stream)
    barrier()
    clocks = sampler.stop()
    ms_step = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    value = whole_job_gbs(attn_bytes, world, ms_step)
    # ---- the attention call alone, back to back (roofline of the dominant kernel call)
    barrier()
    e0.record(stream)
    for i in range(args.steps):
        attn_graphs[i % replicas].replay()
    e1.record(stream)
    barrier()
    attn_avg_ms = e0.elapsed_time(e1) / args.steps
    # ---- the same steps issued eagerly through the Python API (no graph)
    barrier()
    e0.record(stream)
    for i in range(args.steps):
        write(i)
        attend(i)
    e1.record(stream)
    barrier()
    eager_ms = e0.elapsed_time(e1) / args.steps

    # ---- end to end through the public API from pinned host buffers: every step uploads its
    # packed inputs, runs the write and the attention and reads the output back.  Timed eagerly
    # (Python issuing each step) and, as a serving loop would run decode steps, as one CUDA graph
    # per cache replica holding the whole step including both copies.
    h2d = host.numel()
    host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    d2h = host_out.numel() * host_out.element_size()

    def e2e_step(i):
        t["_buf"].copy_(host, non_blocking=True)
        write(i)
        attend(i)
        host_out.copy_(out, non_blocking=True)

    barrier()
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    barrier()
    e2e_eager_ms = e0.elapsed_time(e1) / args.steps
    e2e_graphs = []
    for r in range(replicas):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e2e_step(r)
        e2e_graphs.append(g)
    for i in range(args.warmup):
        e2e_graphs[i % replicas].replay()
    barrier()
    e0.record(stream)
    for i in range(args.steps):
        e2e_graphs[i % replicas].replay()
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    e2e_value = attn_bytes * world / (e2e_ms * 1e-3) / 1e9

    # ---- write-throughput workload
    wres = _write_bench(torch, kv, workloads, dev, stream, args)

    peak, peak_kind = _peaks()
    roof_achieved = attn_bytes / (attn_avg_ms * 1e-3) / 1e9
    traffic = _traffic("decode_gqa_batch")
    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int4-kv/f16-mma/f32", "data": "synthetic",
        "config": {"workload": "gqa_decode_batch: 32 seqs, seq_len U[512,4096] (sum %d), 32 q / 8 kv heads, "
                               "head 128, block 16, bf16 N(0,1) with 4 K channels x10 per kv head, "
                               "permuted blocks; step = write 32 new tokens + decode attention"
                               % int(wl.seq_lens.sum()),
                   "segment_len": seg, "segments_max": nseg, "packed_kv_bytes_per_step": kv_bytes,
                   "qo_bytes_per_step": qo_bytes,
                   "l2": f"{replicas} cache replicas rotated per step ({replicas * cache_bytes / 2**20:.0f} MiB "
                         f"> 2 x 129 MB L2)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "timing": "steps replayed as one CUDA graph per step (write + attention)",
                   "eager_ms_per_step": round(eager_ms, 5),
                   "eager_value": round(attn_bytes * world / (eager_ms * 1e-3) / 1e9, 2)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5), "timing": "one CUDA graph per step: packed input upload, write, "
                "attention, output read-back", "eager_ms_per_step": round(e2e_eager_ms, 5),
                "eager_value": round(attn_bytes * world / (e2e_eager_ms * 1e-3) / 1e9, 2)},
        "roofline": {"bound": "hbm", "achieved": round(roof_achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(roof_achieved / peak, 4), "traffic": traffic,
                     "kernel": "attention call (query rotation + decode kernel + segment combine), graph-replayed back to back",
                     "peak_source": peak_kind,
                     "bytes_per_launch": attn_bytes, "avg_ms": round(attn_avg_ms, 5)},
        "write": wres,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if args.extra:
        result["extra"] = _extra(torch, kv, workloads, dev, args)
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = _cpu_baseline("decode", args)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(result))


def _write_bench(torch, kv, workloads, dev, stream, args):
    wl = workloads.write_throughput(seed=args.seed)
    H, d = wl.num_kv_heads, wl.head_size
    signs = torch.from_numpy(wl.signs).to(dev)
    k, v = wl.key.to(dev), wl.value.to(dev)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    cache = torch.zeros(kv.kv_int4_cache_shape(wl.num_blocks, 16, H, d), dtype=torch.uint8, device=dev)
    per_tok = 2 * H * d * k.element_size() + 2 * H * kv.kv_int4_row_bytes(d) + 8
    nbytes = wl.num_tokens * per_tok
    reps = max(3, args.steps // 4)
    for _ in range(max(3, args.warmup)):
        kv.kv_int4_write(k, v, slots, signs, cache)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        kv.kv_int4_write(k, v, slots, signs, cache)   # inputs (268 MB) exceed L2
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    peak, kind = _peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": "write_throughput: 65536 tokens, 8 kv heads, head 128, bf16, magnitudes 10^U(-2,2), "
                        "random slots over 8192 blocks of 16",
            "tokens_per_s": round(wl.num_tokens / (ms * 1e-3), 1), "GB/s": round(gbs, 1), "ms_per_call": round(ms, 5),
            "bytes_per_call": nbytes, "launches": reps,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(gbs / peak, 4), "traffic": _traffic("write_throughput"),
                         "peak_source": kind}}


def _int8_write_bench(torch, kv, workloads, dev, args):
    """The INT8 per-(token, head) comparator's write on the same workload (cache rows d + 4 bytes)."""
    wl = workloads.write_throughput(seed=args.seed)
    H, d = wl.num_kv_heads, wl.head_size
    k, v = wl.key.to(dev), wl.value.to(dev)
    slots = torch.from_numpy(wl.slot_mapping).to(dev)
    cache = torch.zeros(kv.kv_int8_cache_shape(wl.num_blocks, 16, H, d), dtype=torch.uint8, device=dev)
    nbytes = wl.num_tokens * (2 * H * d * k.element_size() + 2 * H * kv.kv_int8_row_bytes(d) + 8)
    reps = 200
    for _ in range(5):
        kv.kv_int8_write(k, v, slots, cache)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        kv.kv_int8_write(k, v, slots, cache)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    peak, _ = _peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"tokens_per_s": round(wl.num_tokens / (ms * 1e-3), 1), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
            "ms_per_call": round(ms, 5), "bytes_per_call": nbytes,
            "cache_bytes_per_token": 2 * H * kv.kv_int8_row_bytes(d),
            "int4_cache_bytes_per_token": 2 * H * kv.kv_int4_row_bytes(d)}


# ------------------------------------------------------------------------------- CPU oracle

def _attention_only(torch, kv, wl, dev, reps, rows=None, segment_len=0):
    """Write every token of ``wl`` (untimed), then time ``reps`` back-to-back attention calls
    (captured in one CUDA graph) over the whole batch.  Returns ms per call."""
    H, d = wl.num_kv_heads, wl.head_size
    signs = torch.from_numpy(wl.signs).to(dev)
    cache = torch.zeros(kv.kv_int4_cache_shape(wl.num_blocks, 16, H, d), dtype=torch.uint8, device=dev)
    step = 1 << 18
    for r0 in range(0, wl.key.shape[0], step):
        r1 = min(wl.key.shape[0], r0 + step)
        kv.kv_int4_write(wl.key[r0:r1].to(dev), wl.value[r0:r1].to(dev),
                         torch.from_numpy(wl.slot_mapping[r0:r1]).to(dev), signs, cache)
    q = wl.query.to(dev)
    tables, lens = torch.from_numpy(wl.block_tables).to(dev), torch.from_numpy(wl.seq_lens).to(dev)
    qsl = torch.from_numpy(wl.query_start_loc).to(dev)
    seg = kv.kv_int4_attention_segment_len(len(wl.seq_lens), wl.max_seq_len, segment_len)
    ws = torch.empty(max(1, kv.kv_int4_attention_workspace_bytes(wl.num_q_heads, H, d, len(wl.seq_lens),
                                                                 wl.max_seq_len, seg)), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)

    def call():
        kv.kv_int4_paged_attention(q, cache, tables, lens, qsl, wl.softmax_scale, signs,
                                   max_query_len=wl.max_query_len, max_seq_len=wl.max_seq_len, out=out,
                                   segment_len=seg, workspace=ws)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            call()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    g.replay()
    e1.record()
    torch.cuda.synchronize()
    del cache
    return e0.elapsed_time(e1) / reps, seg


def _extra(torch, kv, workloads, dev, args):
    """The long-context and mixed workloads, attention call only (their caches exceed L2)."""
    peak, _ = _peaks()
    res = {}
    wl = workloads.long_context_decode(seed=args.seed)
    ms, seg = _attention_only(torch, kv, wl, dev, reps=20)
    rb = kv.kv_int4_row_bytes(wl.head_size)
    kvb = int(wl.seq_lens.sum()) * 2 * wl.num_kv_heads * rb + 2 * wl.query.numel() * 2
    res["long_context_decode"] = {"ms": round(ms, 4), "GB/s": round(kvb / ms / 1e6, 1),
                                  "frac": round(kvb / ms / 1e6 / peak, 4), "bytes": kvb, "segment_len": seg}
    del wl
    wl = workloads.mixed_prefill_decode(seed=args.seed)
    ms, seg = _attention_only(torch, kv, wl, dev, reps=10)
    kvb = int(wl.seq_lens.sum()) * 2 * wl.num_kv_heads * rb + 2 * wl.query.numel() * 2
    # dense-equivalent attention FLOPs of the prefill chunks: 4 d per visible (query, key) pair per q head
    pairs = sum(int(q) * (int(L) - int(q)) + int(q) * (int(q) + 1) // 2
                for L, q in zip(wl.seq_lens, wl.query_lens) if q > 1)
    flops = 4 * wl.head_size * pairs * wl.num_q_heads
    res["mixed_prefill_decode"] = {"ms": round(ms, 4), "GB/s_packed_kv": round(kvb / ms / 1e6, 1),
                                   "prefill_TFLOP": round(flops / 1e12, 4), "bytes": kvb, "segment_len": seg}
    pre = workloads.make_attention_workload("prefill_only", wl.seq_lens[:4], wl.query_lens[:4], 32, 8, 128,
                                            seed=args.seed)
    ms_p, _ = _attention_only(torch, kv, pre, dev, reps=10)
    res["mixed_prefill_decode"]["prefill_part_ms"] = round(ms_p, 4)
    res["mixed_prefill_decode"]["prefill_part_TFLOP/s"] = round(flops / ms_p / 1e9, 1)
    res["int8_write_comparator"] = _int8_write_bench(torch, kv, workloads, dev, args)
    return res


def _only(args):
    """One workload's attention call, timed as in --extra, on its own (no decode-batch steps)."""
    import torch

    import int4_token_head_kv_gb300 as kv
    import workloads

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    peak, _ = _peaks()
    wl = getattr(workloads, args.only)(seed=args.seed)
    ms, seg = _attention_only(torch, kv, wl, dev, reps=10)
    kvb = int(wl.seq_lens.sum()) * 2 * wl.num_kv_heads * kv.kv_int4_row_bytes(wl.head_size) + 2 * wl.query.numel() * 2
    print(json.dumps({"only": args.only, "ms": round(ms, 4), "GB/s": round(kvb / ms / 1e6, 1),
                      "frac": round(kvb / ms / 1e6 / peak, 4), "bytes": kvb, "segment_len": seg}))


def _cpu_baseline(kind, args, nsample=None):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    n = nsample if nsample is not None else (2 if kind == "decode" else 2048)
    res = subprocess.run([sys.executable, "-m", "oracle.timing", kind, str(n), str(args.seed)], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=900)
    if res.returncode != 0:
        return {"value": None, "unit": "GB/s", "cores": 1, "kind": "oracle", "error": res.stderr[-400:]}
    r = json.loads(res.stdout.strip().splitlines()[-1])
    return {"value": round(r["bytes"] / r["seconds"] / 1e9, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{r['what']} of the GQA decode workload (write their tokens + attention), "
                      f"{r['seconds']:.2f} s single-threaded" if kind == "decode" else r["what"],
            "seconds": round(r["seconds"], 3)}


def _reference_arm(args):
    """The CPU oracle, as it stands, on the GPU arm's workload and metric.  Each step is a bounded
    sample: one (sequence, kv head) of the GQA decode batch, round-robin, truncated to the first n
    tokens so that warm-up + steps take about two minutes whatever --steps is.  A step writes the
    sample's tokens into the oracle's cache and runs the oracle attention for that kv head's query
    heads; its bytes are the packed K/V rows (+ Q/O) it covers."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np

    import oracle
    import workloads

    wl = workloads.gqa_decode_batch(seed=args.seed)
    S, H, G, d = len(wl.seq_lens), wl.num_kv_heads, wl.num_q_heads // wl.num_kv_heads, wl.head_size
    rb = d // 2 + 4

    def one(i, ntok):
        b, h = i % S, (i // S) % H
        L = min(int(wl.seq_lens[b]), ntok)
        rows = np.arange(wl.token_start[b], wl.token_start[b] + L)
        nb = (L + 15) // 16
        table = np.arange(nb, dtype=np.int32)[None]
        cache = np.zeros(oracle.cache_shape(nb, 16, 1, d), np.uint8)
        q = wl.query[b:b + 1, h * G:(h + 1) * G]
        t0 = time.perf_counter()
        oracle.write(wl.key[rows, h:h + 1], wl.value[rows, h:h + 1], np.arange(L, dtype=np.int64), wl.signs, cache)
        oracle.paged_attention(q, cache, table, np.array([L], np.int32), np.array([0, 1], np.int32),
                               wl.softmax_scale, wl.signs)
        return time.perf_counter() - t0, L * 2 * rb + 2 * G * d * 2

    t_start = time.perf_counter()
    dt, _ = one(0, 4096)
    per_tok = dt / min(int(wl.seq_lens[0]), 4096)
    budget = 120.0 / max(1, args.steps + args.warmup)
    ntok = int(max(16, min(4096, budget / max(per_tok, 1e-9))))
    for i in range(args.warmup):
        one(i, ntok)
    secs, nbytes = 0.0, 0
    for i in range(args.steps):
        s_, b_ = one(i, ntok)
        secs += s_
        nbytes += b_
    value = nbytes / secs / 1e9
    sample = f"1 (sequence, kv head) of the GQA decode batch per step, first {ntok} tokens, round-robin"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 write / f64 attention",
            "data": "synthetic",
            "config": {"workload": "gqa_decode_batch (the GPU arm's workload); oracle on a bounded sample per step",
                       "sample_tokens": ntok},
            "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(time.perf_counter() - t_start, 2)}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--segment-len", type=int, default=0,
                    help="split-KV segment length in tokens (multiple of 16); 0 = the library's choice")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra", action="store_true",
                    help="also time the long-context and mixed prefill+decode workloads (attention call only)")
    ap.add_argument("--only", choices=["long_context_decode", "mixed_prefill_decode"],
                    help="time just this workload's attention call and print its own JSON line (for profiling)")
    args = ap.parse_args()
    if args.only:
        _only(args)
        return
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


if __name__ == "__main__":
    main()
