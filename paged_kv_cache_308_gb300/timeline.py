"""Per-CTA timeline of the partition kernel (diagnostics).

Rebuilds the library with -DPA_TRACE, runs one decode call of a named
workload after a few warm-up calls, and reports from the per-CTA records
(SM id; globaltimer at entry, first staged block, end of the main loop and
exit): start-up, streaming and epilogue times, CTAs per SM, and how many CTAs
are resident / streaming over the launch.  The default library is rebuilt
afterwards.

    python -m paged_kv_cache_308_gb300.timeline b1_l102400:512 [name:partition[:warps:stages] ...]

A partition of 0 takes the library's own plan; `name:persistent` runs the
persistent schedule with its default plan (its "main loop done" is the end of
the CTA's first item); `name:pooled` the library's plan with PA_FLAG_POOLED.
"""
from __future__ import annotations

import collections
import ctypes
import sys

import numpy as np
import torch


def _analyse(pb, W, name: str, partition: int, warps: int = 0, stages: int = 0, out=print, special=""):
    dev = torch.device("cuda:0")
    w = W.make_config(name, device=dev)
    res = torch.empty_like(w.q)
    opt = dict(mode="split", partition_size=partition, warps=warps, stages=stages) if partition else dict()
    if special == "persistent":
        opt = dict(mode="persistent")
    elif special == "pooled":
        opt = dict(flags=pb.PA_FLAG_POOLED)
    plan = pb.pa_decode_plan(res, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len, **opt)
    ncta = plan["grid_x"] * plan["grid_y"] * plan["grid_z"]
    buf = torch.zeros(ncta * 5, dtype=torch.int64, device=dev)
    ws = pb.alloc_workspace(plan, dev) if opt else None  # kept: the pooled counters are armed by a call
    for _ in range(5):
        pb.decode_workload(w, workspace=ws, **opt)
    torch.cuda.synchronize()
    pb.lib.pa_debug_set_trace.argtypes = [ctypes.c_void_p]
    pb.lib.pa_debug_set_trace(buf.data_ptr())
    pb.decode_workload(w, workspace=ws, **opt)
    torch.cuda.synchronize()
    pb.lib.pa_debug_set_trace(None)
    t = buf.view(ncta, 5).cpu().numpy()
    t = t[(t[:, 4] > 0) & (t[:, 2] > 0)]
    sm, t0 = t[:, 0], t[:, 1].min()
    e, f, l, x = [(t[:, k] - t0) / 1e3 for k in (1, 2, 3, 4)]
    q = lambda a: np.percentile(a, [0, 10, 50, 90, 100]).round(2).tolist()
    out(f"== {name} P={plan['partition_size']}, CTA {plan['threads'] // 32} warp(s) x {plan['stages']} stages: "
        f"{len(t)} working CTAs of {ncta}; span {x.max():.2f} us = {w.kv_bytes / x.max() / 1e3:.0f} GB/s in-kernel")
    out(f"  start-up (entry -> first block)  us, pct 0/10/50/90/100: {q(f - e)}")
    out(f"  streaming (first block -> loop end): {q(l - f)}")
    out(f"  epilogue (loop end -> exit):         {q(x - l)}")
    per = collections.defaultdict(list)
    for i in range(len(sm)):
        per[int(sm[i])].append(x[i])
    out(f"  CTAs per SM: {dict(sorted(collections.Counter(len(v) for v in per.values()).items()))}; "
        f"per-SM last exit us: {q(np.array([max(v) for v in per.values()]))}")
    grid = np.linspace(0, x.max(), 24)
    out(f"  resident CTAs over the launch:  {[int(((e <= g) & (x > g)).sum()) for g in grid]}")
    out(f"  streaming CTAs over the launch: {[int(((f <= g) & (l > g)).sum()) for g in grid]}")


def main(argv):
    from . import build
    build.build(force=True, extra_flags=["-DPA_TRACE"])
    try:
        from . import binding as pb
        from . import workloads as W
        for spec in (argv or ["b1_l102400:512"]):
            name, *rest = spec.split(":")
            if rest in (["persistent"], ["pooled"]):
                _analyse(pb, W, name, 0, special=rest[0])
                continue
            nums = [int(v) for v in rest] + [0] * (3 - len(rest))
            _analyse(pb, W, name, *nums[:3])
    finally:
        build.build(force=True)


if __name__ == "__main__":
    main(sys.argv[1:])
