"""Measure every compiled partition CTA shape at several partition sizes.

For each named workload, times back-to-back decode calls (pa_decode_ex with
a caller workspace, so consecutive calls overlap their launches as in
serving) for every (partition size, warps x stages) pair, interleaved over
three rounds; prints the median time per call and the K/V GB/s.  These are
the measurements the host's CTA-shape model was fitted to.

    python -m paged_kv_cache_308_gb300.tune [--parts 128,256,512,1024] [workload ...]
"""
from __future__ import annotations

import argparse
import statistics

import torch

from . import binding as pb
from . import workloads as W

SHAPES = [(2, 2), (1, 2), (1, 3), (4, 2)]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--parts", default="128,256,512,1024")
    ap.add_argument("--rounds", type=int, default=3)
    ap.add_argument("workloads", nargs="*", default=W.CONFIG_NAMES)
    args = ap.parse_args()
    parts = [int(x) for x in args.parts.split(",")]
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream()
    for name in args.workloads:
        w = W.make_config(name, device=dev)
        out = torch.empty_like(w.q)
        calls = {}
        for P in parts:
            for nw, ns in SHAPES:
                opt = dict(mode="split", partition_size=P, warps=nw, stages=ns)
                plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                                         w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                                         max_seq_len=w.max_seq_len, **opt)
                ws = pb.alloc_workspace(plan, dev)
                calls[(P, nw, ns)] = (lambda opt=opt, ws=ws: pb.pa_decode_ex(
                    out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                    w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len, workspace=ws, **opt))
        auto = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                                 w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len)
        times = {k: [] for k in calls}
        n = 300 if w.kv_bytes > 1e8 else 1000
        for _ in range(args.rounds):
            for k, fn in calls.items():
                for _ in range(10):
                    fn()
                s = torch.cuda.Event(enable_timing=True)
                e = torch.cuda.Event(enable_timing=True)
                s.record(stream)
                for _ in range(n):
                    fn()
                e.record(stream)
                e.synchronize()
                times[k].append(s.elapsed_time(e) / n * 1e3)
        print(f"{name}: library choice at P={auto['partition_size']}: "
              f"{auto['threads'] // 32} warp(s) x {auto['stages']} stages")
        for (P, nw, ns), v in times.items():
            t = statistics.median(v)
            print(f"  P={P:5d} {nw}x{ns}  {t:9.2f} us  {w.kv_bytes / t / 1e3:7.0f} GB/s", flush=True)
        del w, calls
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
