"""Split-KV across devices, host side, on CPU: the partition ranges and the
exchange of partials between ranks (gloo, world sizes 2 and 3).

Each rank computes the partials of its own range with the float64 oracle
(standing in for pa_decode_partials, which needs a GPU), converted to the
library's base-2 convention; split_kv.gather_partials exchanges them; rank 0
merges the gathered set, locating partition p at slot p % count of source
p // count as pa_merge_partials does, with the oracle's log-sum-exp combine,
and must reproduce the oracle's unsplit decode."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_cache_308_gb300 import split_kv
from paged_kv_cache_308_gb300 import workloads as W

LOG2E = 1.0 / math.log(2.0)
LENS = [0, 1, 37, 700, 1500, 1029]
P = 128


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem():
    w = W.make_workload("dist", LENS, num_heads=6, num_kv_heads=2, head_dim=32, num_blocks=250, seed=41,
                        device="cpu", scale=1 / math.sqrt(32))
    bits = lambda t: t.numpy().view(np.uint16) if t.dtype == torch.float16 else t.numpy()
    args = (bits(w.q), bits(w.k_cache), bits(w.v_cache), bits(w.block_tables), bits(w.seq_lens), w.num_heads,
            w.num_kv_heads, w.head_dim, w.block_size, w.scale)
    return w, args


def _local_partials(oracle, w, args, begin, count):
    # the library's buffer shapes, in float64 so that the check can stay at 1e-12
    m, l, acc = (torch.zeros_like(t, dtype=torch.float64)
                 for t in split_kv.alloc_partials(w.num_seqs, w.num_heads, w.head_dim, count, "cpu"))
    m.fill_(-math.inf)
    for b in range(w.num_seqs):
        for h in range(w.num_heads):
            om, ol, oacc = oracle.partition_partials(*args, b, h, P, 16)
            for j in range(count):
                if begin + j < len(om):
                    m[b, h, j] = om[begin + j] * LOG2E  # the library's base-2 max
                    l[b, h, j] = ol[begin + j]
                    acc[b, h, j] = torch.from_numpy(oacc[begin + j])
    return m, l, acc


def _worker(rank, world, port, q):
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, args = _problem()
        begin, count = split_kv.partition_range(rank, world, w.max_seq_len, P)
        m, l, acc = _local_partials(oracle, w, args, begin, count)
        gm, gl, gacc = split_kv.gather_partials(m, l, acc)
        assert gm.shape == (world,) + tuple(m.shape) and gacc.shape == (world,) + tuple(acc.shape)
        # this rank's own partials arrive at its own source slot, unchanged
        assert torch.equal(gm[rank], m) and torch.equal(gacc[rank], acc)
        ref = oracle.paged_decode(*args)
        got = np.zeros_like(ref)
        for b, L in enumerate(LENS):
            n = (L + P - 1) // P
            for h in range(w.num_heads):
                loc = [(p // count, p % count) for p in range(n)]
                mm = np.array([gm[r, b, h, j].item() for r, j in loc]) / LOG2E
                ll = np.array([gl[r, b, h, j].item() for r, j in loc])
                aa = np.array([gacc[r, b, h, j].numpy() for r, j in loc]).reshape(n, w.head_dim)
                got[b, h] = oracle.combine_lse(mm, ll, aa)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
        q.put((rank, "ok"))
    except Exception as e:  # reported to the parent
        q.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_and_merge_with_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    assert got == [(r, "ok") for r in range(world)]


@pytest.mark.parametrize("n_tokens,P_,world", [(102400, 512, 2), (102400, 512, 3), (1, 16, 4), (8000, 512, 8),
                                              (0, 512, 2)])
def test_ranges_cover_every_partition_once_in_rank_order(n_tokens, P_, world):
    n = split_kv.num_partitions(n_tokens, P_)
    ranges = [split_kv.partition_range(r, world, n_tokens, P_) for r in range(world)]
    counts = {c for _, c in ranges}
    assert len(counts) == 1  # every rank sends the same number of bytes
    count = counts.pop()
    covered = [p for b, c in ranges for p in range(b, b + c)]
    assert covered == list(range(world * count))  # consecutive, rank order, no overlap
    assert world * count >= n and (count - 1) * world < n  # the fewest per rank that cover n
    with pytest.raises(ValueError):
        split_kv.partition_range(world, world, n_tokens, P_)
