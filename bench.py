#!/usr/bin/env python
"""Benchmark of split-KV paged-attention decode on GB300.

A step is one decode call over the whole batch: the partition kernel and the
log-sum-exp reduce, through the library's C ABI, with q, the K/V pool, the
block tables and the sequence lengths already resident in HBM.  The default
workload is the 100K-token long-context decode: batch 1, seq_len 102400
(the library's plan: one wave of 38 partitions x 4 kv heads), 24 query /
4 kv heads, head_dim 256, block_size 16,
fp16 N(0,1) data, scale 1/16; its 419 MB of K/V exceed the 129 MB L2, so
back-to-back steps read from HBM.

Prints one JSON line: KV-cache GB/s read (sum_b L_b * 4096 B per call / time),
with the fraction of the measured HBM peak, calls/s, tokens/s, a roofline
entry for the partition kernel, the float64 oracle timed on the host cores as
a CPU baseline, an end-to-end figure through the public call with host
buffers, and the SM clocks sampled during the timed region.

`--impl reference` times the float64 CPU oracle on the same workload instead
(the only reference implementation of this method).  Under torchrun the
GPU arm runs one replica per rank (the path needs no exchange between GPUs:
replicas only) and reports the aggregate.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_308_gb300 import workloads as W  # noqa: E402

METRIC = "decode-attention KV-cache GB/s"
DEFAULT_WORKLOAD = "b1_l102400"
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic_partition_b1_l102400.json")
KERNEL_SRC = os.path.join(ROOT, "paged_kv_cache_308_gb300", "csrc", "pa_kernels.cu")

WORKLOAD_TEXT = {
    "b1_l2048": "batch 1, seq_len 2048, heads 24/4, head_dim 256, block_size 16",
    "b8_u8192": "batch 8, seq_lens uniform [1, 8192], heads 24/4, head_dim 256, block_size 16, pool 8192 blocks",
    "b4_l32768_peaked": "batch 4, seq_len 32768, 1% of keys x8, heads 24/4, head_dim 256, block_size 16",
    "b1_l102400": "batch 1, seq_len 102400, heads 24/4, head_dim 256, block_size 16",
    "b64_loguniform": "batch 64, seq_lens log-uniform [16, 65536], heads 24/4, head_dim 256, block_size 16, "
                      "pool 98304 blocks",
}


def parse():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.CONFIG_NAMES)
    ap.add_argument("--all-configs", action="store_true",
                    help="longer per-workload timing (500 calls instead of 200); the other workloads are always timed")
    ap.add_argument("--no-per-config", action="store_true", help="time the headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU work budget of the oracle baseline")
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken during the timed region."""

    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        if which == 0:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        time.sleep(0.15)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.06 <= r[0] <= self.t1 + 0.06]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        mhz = [float(p[1]) for _, p in use if p[1].replace(".", "", 1).isdigit()]
        mx = [float(p[2]) for _, p in use if p[2].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for _, p in use for n, v in zip(names, p[5:9]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use), "in_region": bool(inside)}


def max_over_ranks(x: float, dist, device) -> float:
    """The slowest rank's time: every rank passes its own, all get the max."""
    t = torch.tensor([x], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_step: int, steps: int, world: int, elapsed_max: float) -> float:
    """Whole-job K/V GB/s: every rank runs the same workload (replicas)."""
    return world * bytes_per_step * steps / elapsed_max / 1e9


def kernel_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_308_gb300", "csrc")
    for p in (KERNEL_SRC, os.path.join(csrc, "pa_partition_block.cuh"), os.path.join(csrc, "pa_device.cuh"),
              os.path.join(csrc, "pa_internal.h")):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload):
    """DRAM bytes per partition-kernel launch from the committed ncu summary,
    or None when the kernel source changed since it was captured."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        if d.get("kernel_sha") == kernel_hash() and d.get("workload") == workload:
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def host_bits(t):
    import numpy as np
    a = t.detach().cpu().contiguous().numpy()
    return a.view(np.uint16) if a.dtype == np.float16 else a


def cpu_baseline(w, budget_s: float):
    """The float64 oracle as it stands, on the host cores, over whole decode
    calls of the workload: repeated until `budget_s` of work (at least one)."""
    import oracle
    q, k, v = host_bits(w.q), host_bits(w.k_cache), host_bits(w.v_cache)
    bt, sl = host_bits(w.block_tables), host_bits(w.seq_lens)
    cores = os.cpu_count() or 1
    oracle.build()
    calls = 0
    t0 = time.perf_counter()
    while True:
        oracle.paged_decode(q, k, v, bt, sl, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                            threads=cores)
        calls += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (calls >= 1 and el * (calls + 1) / calls > 3 * budget_s):
            break
    gbs = w.kv_bytes * calls / el / 1e9
    # the same oracle on one thread, over one call
    t1 = time.perf_counter()
    oracle.paged_decode(q, k, v, bt, sl, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale, threads=1)
    el1 = time.perf_counter() - t1
    return {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{calls} whole decode call(s) of {w.name} ({w.total_tokens} tokens, {w.num_heads} heads), "
                      f"{el:.1f} s, float64, OpenMP over (seq, head) pairs",
            "value_1_thread": w.kv_bytes / el1 / 1e9}, calls / el


def flushed_latency_us(fn, stream, dev, n=50):
    """Median device time of `n` single calls, each after a write of twice
    the L2 size on the same stream, so every call starts from a cold L2."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size or (129 << 20)
    scratch = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for e0, e1 in evs:
        scratch.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    del scratch
    return statistics.median(e0.elapsed_time(e1) for e0, e1 in evs) * 1e3


def graph_calls_per_s(pb, w, dev, per_graph=20, replays=25):
    """Calls/s with the calls captured once in a CUDA graph and replayed
    (caller workspace, no allocation in the captured region)."""
    out = torch.empty_like(w.q)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len)
    ws = pb.alloc_workspace(plan, dev)

    def call(s):
        pb.pa_decode_ex(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                        w.head_dim, w.block_size, w.scale, s, max_seq_len=w.max_seq_len, workspace=ws)

    call(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(per_graph):
            call(torch.cuda.current_stream())
    g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(replays):
        g.replay()
    e1.record(s)
    e1.synchronize()
    return per_graph * replays / (e0.elapsed_time(e1) / 1e3)


def queue_ahead(stream, calls):
    """Queue a GPU spin on `stream` long enough for the host to queue the
    next `calls` calls behind it (about 15 us of host time each, 0.3-50 ms),
    so a timed region that starts after it opens on a full queue: the
    region then holds the calls' device time, not the host's launch latency
    of its first call.  (The host's costs are in the end-to-end figure.)"""
    if hasattr(torch.cuda, "_sleep"):
        with torch.cuda.stream(stream):
            torch.cuda._sleep(int(min(50e-3, max(3e-4, calls * 15e-6)) * 2.0e9))  # ~2 GHz SM clock


def time_steps(fn, steps, stream):
    """Seconds of device time for `steps` back-to-back calls of `fn`."""
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    queue_ahead(stream, steps)
    s.record(stream)
    for _ in range(steps):
        fn()
    e.record(stream)
    e.synchronize()
    return s.elapsed_time(e) / 1e3


def time_e2e(pb, w, stream, dev, steps, nbuf=2):
    """Seconds for `steps` decode calls through the public call, each with
    its own host->device input copy and device->host output copy (pinned
    host memory), pipelined over `nbuf` buffer sets; returns (seconds, steps,
    h2d bytes per step, d2h bytes per step).  A step's inputs (q, block
    table, sequence lengths) are packed in one buffer, so one copy brings
    them, as a serving loop would stage them."""
    parts = [w.q, w.block_tables, w.seq_lens]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs = [0]
    for n in sizes:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    h_in = torch.empty(offs[-1], dtype=torch.uint8, pin_memory=True)
    for t, o, n in zip(parts, offs, sizes):
        h_in[o:o + n].copy_(t.contiguous().view(-1).view(torch.uint8).cpu())
    d_in = [torch.empty(offs[-1], dtype=torch.uint8, device=dev) for _ in range(nbuf)]

    def view(buf, i):
        t = parts[i]
        return buf[offs[i]:offs[i] + sizes[i]].view(t.dtype).view(t.shape)

    d_q = [view(d, 0) for d in d_in]
    d_bt = [view(d, 1) for d in d_in]
    d_sl = [view(d, 2) for d in d_in]
    h_out = [torch.empty(w.q.shape, dtype=w.q.dtype, pin_memory=True) for _ in range(nbuf)]
    d_out = [torch.empty_like(w.q) for _ in range(nbuf)]
    h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]    # inputs of set k landed
    ev_done = [torch.cuda.Event() for _ in range(nbuf)]  # the call on set k finished
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]   # output of set k is back on the host
    count = [0]

    def e2e_step():
        k = count[0] % nbuf
        with torch.cuda.stream(h2d):
            h2d.wait_event(ev_done[k])  # the call two steps back has read set k
            d_in[k].copy_(h_in, non_blocking=True)
            ev_in[k].record(h2d)
        stream.wait_event(ev_in[k])
        stream.wait_event(ev_out[k])  # set k's previous output has been copied back
        pb.pa_decode(d_out[k], d_q[k], w.k_cache, w.v_cache, d_bt[k], d_sl[k], w.num_heads, w.num_kv_heads,
                     w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len)
        ev_done[k].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(ev_done[k])
            h_out[k].copy_(d_out[k], non_blocking=True)
            ev_out[k].record(d2h)
        count[0] += 1

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    h2d.wait_event(start)
    for _ in range(steps):
        e2e_step()
    stream.wait_event(ev_out[(count[0] - 1) % nbuf])  # the last output is on the host
    end.record(stream)
    end.synchronize()
    torch.cuda.synchronize()
    # the pipelined calls agree with a plain call on the resident inputs (to
    # the rounding of the partial sums: a pooled plan's partials cover
    # timing-dependent blocks)
    ref = torch.empty_like(w.q)
    pb.pa_decode(ref, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                 w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    got, want = h_out[(count[0] - 1) % nbuf].float(), ref.cpu().float()
    if not bool(((got - want).abs() <= 2e-3 + 1e-2 * want.abs()).all()):
        raise RuntimeError("pipelined end-to-end output differs from the direct call")
    return (start.elapsed_time(end) / 1e3, steps, h_in.numel(), h_out[0].numel() * 2)


def measure_workload(pb, w, stream, dev, peak, n):
    """Back-to-back, cold-L2 and graph-replayed figures of the library's own
    plan (pa_decode, AUTO) on one workload."""
    out = torch.empty_like(w.q)
    fn = lambda: pb.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                              w.num_kv_heads, w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len)
    for _ in range(20):
        fn()
    torch.cuda.synchronize()
    el = time_steps(fn, n, stream)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len)
    return {"kv_bytes": w.kv_bytes, "us_per_call": el / n * 1e6, "GB_per_s": w.kv_bytes * n / el / 1e9,
            "pct_of_hbm_peak": 100 * w.kv_bytes * n / el / 1e9 / peak, "calls_per_s": n / el,
            "tokens_per_s": w.num_seqs * n / el,
            "plan": {"mode": "split" if plan["launch_reduce"] else "single", "partition_size": plan["partition_size"],
                     "cta": f"{plan['threads'] // 32}x{plan['stages']}", "grid": [plan["grid_x"], plan["grid_y"],
                                                                                   plan["grid_z"]],
                     "pooled": bool(plan["pooled"])},
            "l2": "larger than L2" if w.kv_bytes > 129e6 else "fits in L2 (warm)",
            "latency_us_l2_flushed": flushed_latency_us(fn, stream, dev),
            "graph_calls_per_s": graph_calls_per_s(pb, w, dev)}


def measure_variant(pb, w, stream, dev, peak, n, **opt):
    """Back-to-back figure of one explicitly requested plan (pa_decode_ex with a
    caller workspace kept across calls)."""
    out = torch.empty_like(w.q)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len, **opt)
    ws = pb.alloc_workspace(plan, dev)
    fn = lambda: pb.pa_decode_ex(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                                 w.num_kv_heads, w.head_dim, w.block_size, w.scale, stream,
                                 max_seq_len=w.max_seq_len, workspace=ws, **opt)
    for _ in range(20):
        fn()
    torch.cuda.synchronize()
    el = time_steps(fn, n, stream)
    return {"us_per_call": el / n * 1e6, "GB_per_s": w.kv_bytes * n / el / 1e9,
            "pct_of_hbm_peak": 100 * w.kv_bytes * n / el / 1e9 / peak, "calls_per_s": n / el,
            "partition_size": plan["partition_size"], "partitions": plan["max_partitions"],
            "cta": f"{plan['threads'] // 32}x{plan['stages']}", "pooled": bool(plan["pooled"])}


def measure_split_kv(pb, w, stream, dev, peak, n, sources=2, partition_size=512):
    """Split-KV across devices, kernel side, emulated on this one GPU: the
    partials of each source's range of partitions (one pa_decode_partials
    call per source into its slot of the gathered buffer), then
    pa_merge_partials.  No exchange between devices takes place."""
    from paged_kv_cache_308_gb300 import split_kv
    ranges = [split_kv.partition_range(r, sources, w.max_seq_len, partition_size) for r in range(sources)]
    count = ranges[0][1]
    gm, gl, gacc = split_kv.alloc_partials(w.num_seqs, w.num_heads, w.head_dim, count, dev, sources=sources)
    out = torch.empty_like(w.q)

    def fn():
        for r, (b, c) in enumerate(ranges):
            pb.pa_decode_partials(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                                  w.num_kv_heads, w.head_dim, w.block_size, w.scale, partition_size, b, c, gm[r],
                                  gl[r], gacc[r], stream, max_seq_len=w.max_seq_len)
        pb.pa_merge_partials(out, gm, gl, gacc, w.seq_lens, w.num_heads, w.head_dim, partition_size, sources, count,
                             stream, max_seq_len=w.max_seq_len)

    for _ in range(20):
        fn()
    torch.cuda.synchronize()
    el = time_steps(fn, n, stream)
    return {"us_per_call": el / n * 1e6, "GB_per_s": w.kv_bytes * n / el / 1e9,
            "pct_of_hbm_peak": 100 * w.kv_bytes * n / el / 1e9 / peak, "sources": sources,
            "partition_size": partition_size, "partitions_per_source": count,
            "launches_per_call": sources + 1,
            "note": "all sources on this one GPU, one after another; no exchange between devices"}


def run_reference(args):
    """The float64 oracle on the host cores.  Each step is a bounded sample of
    the workload: every (sequence, head) pair over the first L' tokens of its
    sequence, L' calibrated so that the whole run ends within a few minutes;
    the step is credited with the K/V bytes of those tokens (4096 B each)."""
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    w = W.make_config(args.workload, device="cpu", seed=args.seed)
    oracle.build()
    q, k, v = host_bits(w.q), host_bits(w.k_cache), host_bits(w.v_cache)
    bt = host_bits(w.block_tables)
    lens = np.array(w.seq_lens_host, dtype=np.int32)
    cores = os.cpu_count() or 1
    per_token = w.num_kv_heads * w.head_dim * 2 * 2

    def call(cap):
        sl = np.minimum(lens, cap).astype(np.int32)
        oracle.paged_decode(q, k, v, bt, sl, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                            threads=cores)
        return int(sl.sum())

    target = max(0.002, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    cap, t = 16, 0.0
    while cap < int(lens.max()):
        t0 = time.perf_counter()
        call(cap)
        t = time.perf_counter() - t0
        if t >= target:
            break
        cap = min(int(lens.max()), cap * 2)
    if t > target and cap > 16:
        cap = max(16, int(cap * target / t))
    for _ in range(args.warmup):
        call(cap)
    tokens = 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        tokens += call(cap)
    el = time.perf_counter() - t0
    gbs = tokens * per_token / el / 1e9
    sample = (f"each step: all {w.num_seqs}x{w.num_heads} (seq, head) pairs of {args.workload} over the first "
              f"{cap} tokens of each sequence ({tokens // max(1, args.steps)} of {w.total_tokens} cache tokens), "
              f"float64, OpenMP over pairs")
    line = {
        "metric": METRIC, "value": gbs, "unit": "GB/s", "impl": "reference", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}", "parallelism": "none (CPU)"},
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (use --impl reference for the CPU oracle)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    from paged_kv_cache_308_gb300 import binding as pb

    w = W.make_config(args.workload, device=dev, seed=args.seed)
    out = torch.empty_like(w.q)
    stream = torch.cuda.current_stream()
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len)
    launches_per_step = 1 + plan["launch_reduce"]

    def step():
        pb.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                     w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len)

    step()  # the first warm-up step sets the kernels' attributes and allocates the workspace
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0

    sampler = ClockSampler(local)
    sampler.start()
    # the other warm-up steps run right before the timed region: starting the
    # clock sampler leaves the GPU idle for a moment, and the first calls
    # after an idle spell run slower
    for _ in range(max(args.warmup, 3) - 1):
        step()
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    sampler.mark(0)
    elapsed = time_steps(step, args.steps, stream)
    torch.cuda.synchronize()
    sampler.mark(1)
    if pg:
        pg.barrier()
    sampler.stop()
    if pg:
        elapsed = max_over_ranks(elapsed, pg, dev)
    assert pb.pa_get_device_status() == 0

    peak, peak_kind = hbm_peak()
    kv = w.kv_bytes
    value = aggregate_gbs(kv, args.steps, world, elapsed)
    per_gpu = kv * args.steps / elapsed / 1e9

    # roofline: the partition kernel alone, timed by events the library records
    # on this stream around its launch
    ws = pb.alloc_workspace(plan, dev)
    nrep = max(20, min(args.steps, 500))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(nrep)]
    for e0, e1 in evs:  # torch creates the CUDA event on its first record
        e0.record(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    for e0, e1 in evs:
        pb.pa_decode_ex(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                        w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len, workspace=ws,
                        events=(e0, e1))
    torch.cuda.synchronize()
    part_s = statistics.mean(e0.elapsed_time(e1) for e0, e1 in evs) / 1e3
    achieved = kv / part_s / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": profiled_traffic(args.workload), "kernel": f"pa_partition_kernel<{w.head_dim}, {plan['threads'] // 32}, {plan['stages']}"
                + (", pooled>" if plan["pooled"] else ">"),
                "algorithmic_bytes_per_launch": kv, "launch_us": part_s * 1e6,
                "peak_kind": f"{peak_kind} HBM copy bandwidth (burst)"}

    # end to end through the public call with host buffers: per step the
    # step's inputs (q, block tables, sequence lengths) go host->device from
    # pinned memory, the call runs, and its output comes back to pinned host
    # memory; the K/V cache stays resident in HBM.  As in a serving loop the
    # copies overlap the previous step's call: two sets of device buffers,
    # inputs on one copy stream and outputs on another, ordered by events.
    e2e_el, e2e_steps, h2d_bytes, d2h_bytes = time_e2e(pb, w, stream, dev, max(10, min(args.steps, 2000)))
    e2e = {"value": world * kv * e2e_steps / e2e_el / 1e9, "unit": "GB/s",
           "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
           "ms_per_step": e2e_el / e2e_steps * 1e3,
           "pipelining": "step i's copies overlap step i-1's call (2 buffer sets, separate copy streams); "
                         "the step's inputs packed in one pinned buffer, one copy"}

    # single-call latency from a cold L2 (median of 50) and CUDA-graph-replayed calls/s
    lat_flushed = flushed_latency_us(step, stream, dev)
    graph_cps = graph_calls_per_s(pb, w, dev)

    # the same workload under two other plans: the pages' 512-token partitions
    # (fixed split), and the one-wave plan with fixed partitions (deterministic);
    # and the split-KV-across-devices kernels with two sources on this GPU
    n_var = 500 if args.all_configs else 200
    variants = None
    if rank == 0 and not args.no_per_config:
        variants = {"split_p512": measure_variant(pb, w, stream, dev, peak, n_var, mode="split", partition_size=512),
                    "auto_deterministic": measure_variant(pb, w, stream, dev, peak, n_var,
                                                          flags=pb.PA_FLAG_DETERMINISTIC),
                    "split_kv_2_sources_1gpu": measure_split_kv(pb, w, stream, dev, peak, n_var)}

    per_config = None
    if rank == 0 and not args.no_per_config:
        per_config = {}
        for name in W.CONFIG_NAMES:
            if name == args.workload:
                continue
            wc = W.make_config(name, device=dev, seed=args.seed)
            per_config[name] = measure_workload(pb, wc, stream, dev, peak, n_var)
            if name == "b8_u8192":  # both decode modes of this workload
                per_config[name]["single"] = measure_variant(pb, wc, stream, dev, peak, n_var, mode="single")
                per_config[name]["split_p512"] = measure_variant(pb, wc, stream, dev, peak, n_var, mode="split",
                                                                 partition_size=512)
            if name == "b4_l32768_peaked":  # equal lengths: the caller may say so (one-wave plan)
                per_config[name]["uniform_lengths_flag"] = measure_variant(pb, wc, stream, dev, peak, n_var,
                                                                           flags=pb.PA_FLAG_UNIFORM_LENGTHS)
            del wc
            torch.cuda.empty_cache()
        # chunked prefill over the paged cache (both kernels), TFLOP/s
        from paged_kv_cache_308_gb300 import prefix_bench
        per_config["prefix"] = prefix_bench.measure(W.PREFIX_CONFIG_NAMES, list(prefix_bench.IMPLS), 20, 3, dev)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu, _ = cpu_baseline(W.make_config(args.workload, device="cpu", seed=args.seed), args.cpu_seconds)

    if rank == 0:
        clocks = sampler.summary()
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": f"{args.workload}: {WORKLOAD_TEXT[args.workload]}",
                       "kv_bytes_per_step": kv, "tokens_in_cache": w.total_tokens,
                       "mode": "split" if plan["launch_reduce"] else "single",
                       "partition_size": plan["partition_size"],
                       "pooled": bool(plan["pooled"]),
                       "l2": f"inputs larger than L2 ({kv / 1e6:.0f} MB of K/V vs 129 MB L2), no flush",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "pct_of_hbm_peak": 100 * per_gpu / peak,
            "calls_per_s": world * args.steps / elapsed,
            "tokens_per_s": world * w.num_seqs * args.steps / elapsed,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "latency_us_l2_flushed": lat_flushed,
            "graph_calls_per_s": graph_cps,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
        }
        if variants is not None:
            line["variants"] = variants
        if per_config is not None:
            line["per_config"] = per_config
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
