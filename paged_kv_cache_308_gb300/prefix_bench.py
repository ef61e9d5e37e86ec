"""Time the chunked-prefill (prefix) attention kernels on the named workloads.

For each workload and kernel, runs back-to-back pa_prefix_ex calls on one
stream (after warm-up), times them with CUDA events and prints one JSON line:
microseconds per call, useful TFLOP/s (score and P.V multiply-adds over the
visible keys only, see workloads.PrefixWorkload.flops) and the fraction of
the measured dense 16-bit tensor-core peak.

    python -m paged_kv_cache_308_gb300.prefix_bench [--impl NAME|all] [--iters N] [workload ...]

tcgen05_split is pa_prefix_split (the last round's query tiles split by key
range) under the library's plan; both run the tcgen05 kernel's default
persistent form, the _grid variants its grid form (PA_FLAG_PREFIX_GRID).
"""
from __future__ import annotations

import argparse
import json
import os

import torch

from . import binding as pb
from . import workloads as W

# name: (option flags, through pa_prefix_split)
IMPLS = {"tcgen05": (0, False), "tcgen05_split": (0, True),
         "tcgen05_grid": (pb.PA_FLAG_PREFIX_GRID, False),
         "tcgen05_split_grid": (pb.PA_FLAG_PREFIX_GRID, True),
         "warp_mma": (pb.PA_FLAG_PREFIX_WARP_MMA, False)}
FALLBACK_TENSOR_TFLOPS = 1900.0


def tensor_peak():
    """Dense 16-bit tensor-core TFLOP/s: the measured burst figure when present."""
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_TENSOR_TFLOPS, "fallback"


def time_prefix(w, flags: int, iters: int, warmup: int, stream=None, split: bool = False) -> float:
    """Mean seconds per call over `iters` back-to-back calls: pa_prefix_ex, or
    with `split` pa_prefix_split under the library's plan (workspace kept)."""
    stream = stream or torch.cuda.current_stream()
    out = torch.empty_like(w.q)
    if split:
        ws = torch.empty(max(1, pb.prefix_split_workspace_size(w)), dtype=torch.uint8, device=out.device)
        call = lambda: pb.prefix_split_workload(w, out, stream=stream, workspace=ws, flags=flags)
    else:
        call = lambda: pb.prefix_workload(w, out, stream=stream, flags=flags)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    if pb.pa_get_device_status() != 0:
        raise RuntimeError("prefix kernel reported a device error")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(iters):
        call()
    e1.record(stream)
    e1.synchronize()
    if pb.pa_get_device_status() != 0:
        raise RuntimeError("prefix kernel reported a device error")
    return e0.elapsed_time(e1) / iters / 1e3


def measure(names, impls, iters: int, warmup: int, device) -> list:
    peak, kind = tensor_peak()
    rows = []
    for name in names:
        w = W.make_prefix_config(name, device=device)
        for impl in impls:
            flags, split = IMPLS[impl]
            t = time_prefix(w, flags, iters, warmup, split=split)
            tf = w.flops / t / 1e12
            rows.append({"workload": name, "kernel": impl, "us_per_call": t * 1e6, "tflops": tf,
                         "frac_of_tensor_peak": tf / peak, "peak_tflops": peak, "peak_kind": kind,
                         "tokens": w.num_tokens, "flops_per_call": w.flops})
        del w
        torch.cuda.empty_cache()
    return rows


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--impl", choices=list(IMPLS) + ["all"], default="all")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("workloads", nargs="*", default=W.PREFIX_CONFIG_NAMES)
    args = ap.parse_args()
    impls = list(IMPLS) if args.impl == "all" else [args.impl]
    for row in measure(args.workloads, impls, args.iters, args.warmup, torch.device("cuda:0")):
        print(json.dumps(row), flush=True)


if __name__ == "__main__":
    main()
