"""Per-CTA phases of the tcgen05 chunked-prefill kernel (diagnostics).

Rebuilds the library with -DPA_TRACE, runs one prefix call of a named
workload (or of `ctx:ql:count`, count sequences of ctx cached and ql new
tokens) after a few warm-up calls, and reports from the per-CTA global-timer
records: setup (entry to barriers and tensor memory ready), Q into tensor
memory, the tile loop, the epilogue (loop end to O stored), and the gap
between one CTA's exit and the next one's entry on an SM.  The default
library is rebuilt afterwards.

    python -m paged_kv_cache_308_gb300.prefix_timeline prefix_b4_c8192_q512 [0:1024:8 ...]
"""
from __future__ import annotations

import collections
import ctypes
import sys

import numpy as np
import torch

ITERS = 256  # trace records per CTA (kPrefixTraceIters); the last holds the phases


def _workload(W, spec, dev):
    if spec in W.PREFIX_CONFIG_NAMES:
        return W.make_prefix_config(spec, device=dev)
    ctx, ql, n = (int(v) for v in spec.split(":"))
    return W.make_prefix_workload(f"ctx{ctx}_q{ql}_x{n}", [ctx] * n, [ql] * n, seed=1, device=dev)


def _analyse(pb, W, spec: str, out=print):
    dev = torch.device("cuda:0")
    w = _workload(W, spec, dev)
    res = torch.empty_like(w.q)
    for _ in range(3):
        pb.prefix_workload(w, res)
    torch.cuda.synchronize()
    g = w.num_heads // w.num_kv_heads
    tiles = (max(w.query_lens_host) + 128 // g - 1) // (128 // g)
    ncta = len(w.query_lens_host) * w.num_kv_heads * tiles
    buf = torch.zeros(ncta * ITERS * 16, dtype=torch.int64, device=dev)
    pb.lib.pa_debug_set_trace.argtypes = [ctypes.c_void_p]
    pb.lib.pa_debug_set_trace(buf.data_ptr())
    pb.prefix_workload(w, res)
    torch.cuda.synchronize()
    pb.lib.pa_debug_set_trace(None)
    ph = buf.view(ncta, ITERS, 16)[:, ITERS - 1, :8].cpu().numpy()
    ph = ph[(ph[:, 0] > 0) & (ph[:, 5] > 0)]  # CTAs with a query tile (the others return at once)
    q = lambda a: np.percentile(a, [0, 10, 50, 90, 100]).round(2).tolist()
    us = lambda a, b: (ph[:, b] - ph[:, a]) / 1e3
    out(f"== {w.name}: {len(ph)} working CTAs of {ncta}; span {(ph[:, 5].max() - ph[:, 0].min()) / 1e3:.1f} us")
    out(f"  us, pct 0/10/50/90/100")
    out(f"  setup (entry -> barriers, tensor memory)  {q(us(0, 1))}")
    out(f"  Q into tensor memory                     {q(us(1, 2))}")
    out(f"  tile loop                                {q(us(2, 3))}")
    out(f"  epilogue (loop end -> O stored)          {q(us(3, 4))}")
    out(f"  CTA total                                {q(us(0, 5))}")
    per = collections.defaultdict(list)
    for r in ph:
        per[int(r[7])].append((r[0], r[5]))
    gaps = []
    for v in per.values():
        v.sort()
        gaps += [(v[i + 1][0] - v[i][1]) / 1e3 for i in range(len(v) - 1)]
    out(f"  CTAs per SM {q([len(v) for v in per.values()])}; exit -> next entry on an SM {q(gaps) if gaps else None}")


def main(argv):
    from . import build
    build.build(force=True, extra_flags=["-DPA_TRACE"])
    try:
        from . import binding as pb
        from . import workloads as W
        for spec in (argv or ["prefix_b4_c8192_q512"]):
            _analyse(pb, W, spec)
    finally:
        build.build(force=True)


if __name__ == "__main__":
    main(sys.argv[1:])
