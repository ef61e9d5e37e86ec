"""Split-KV decode across devices: each device computes the partials of its own
range of partitions, the devices exchange them, and each merges all of them.

The pages split one long sequence into partitions of 512 tokens ("docs"
commit page, GQA-aware grid and partition paragraphs: 200 partitions for
100K tokens) and merge the per-partition partials (max score, exp sum,
weighted V) in a second pass.  Spreading those partitions over several
devices needs exactly one exchange: an all-gather of the partials, about
num_heads * partitions * (head_dim + 2) * 4 bytes per sequence and device.

Host logic only (ranges, buffers, the collective); every step of the
arithmetic runs in the library's kernels through ``pa_decode_partials`` and
``pa_merge_partials``.  The collective is ``torch.distributed`` on local
buffers: NCCL between GPUs (``all_gather_into_tensor``), gloo on the CPU;
no kernel ever reads another device's memory.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch
import torch.distributed as dist


def num_partitions(max_seq_len: int, partition_size: int) -> int:
    """Partitions of the longest sequence (at least one)."""
    if partition_size <= 0:
        raise ValueError("partition_size must be positive")
    return max(1, (int(max_seq_len) + partition_size - 1) // partition_size)


def partition_range(rank: int, world: int, max_seq_len: int, partition_size: int) -> Tuple[int, int]:
    """(begin, count) of the partitions device `rank` of `world` computes:
    equal runs of ceil(n / world) consecutive partitions, in rank order, so
    that source r of the merge holds partitions [r * count, (r + 1) * count).
    A rank whose run lies past the longest sequence still produces (empty)
    partials, so every rank sends the same number of bytes."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    per = (num_partitions(max_seq_len, partition_size) + world - 1) // world
    return rank * per, per


def alloc_partials(num_seqs: int, num_heads: int, head_dim: int, count: int, device, sources: Optional[int] = None):
    """(max_logits, exp_sums, tmp_out) float32 buffers of one source
    ([B, H, count], [B, H, count], [B, H, count, D]) or, with `sources`,
    of the gathered set with a leading source dimension."""
    lead = () if sources is None else (int(sources),)
    m = torch.empty(lead + (num_seqs, num_heads, count), dtype=torch.float32, device=device)
    l = torch.empty_like(m)
    acc = torch.empty(lead + (num_seqs, num_heads, count, head_dim), dtype=torch.float32, device=device)
    return m, l, acc


def gather_partials(m: torch.Tensor, l: torch.Tensor, acc: torch.Tensor, group=None):
    """All-gather of the local partials along a new leading source dimension
    (rank order): the layout pa_merge_partials reads."""
    world = dist.get_world_size(group)
    out = []
    for t in (m, l, acc):
        t = t.contiguous()
        g = torch.empty((world,) + tuple(t.shape), dtype=t.dtype, device=t.device)
        if dist.get_backend(group) == "nccl":
            dist.all_gather_into_tensor(g, t, group=group)
        else:
            dist.all_gather(list(g.unbind(0)), t, group=group)
        out.append(g)
    return tuple(out)


def split_kv_decode(out, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                    block_size, scale, partition_size: int, *, max_seq_len: int, group=None, stream=None,
                    **opt) -> None:
    """One decode call whose partitions are spread over the ranks of `group`.

    Every rank passes the same q, block tables and lengths; its K/V pool must
    hold the blocks of its own partition range (entries of the block table
    outside that range are never read).  Every rank ends with the full output
    in `out`."""
    from paged_kv_cache_308_gb300 import binding as pb

    rank, world = dist.get_rank(group), dist.get_world_size(group)
    begin, count = partition_range(rank, world, max_seq_len, partition_size)
    s = torch.cuda.current_stream(q.device) if stream is None else stream
    # the collective orders itself after the current stream's work, so the
    # three steps run with `s` as the current stream
    with torch.cuda.stream(s):
        m, l, acc = alloc_partials(int(seq_lens.shape[0]), num_heads, head_dim, count, q.device)
        pb.pa_decode_partials(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                              block_size, scale, partition_size, begin, count, m, l, acc, s, max_seq_len=max_seq_len,
                              **opt)
        gm, gl, gacc = gather_partials(m, l, acc, group)
        pb.pa_merge_partials(out, gm, gl, gacc, seq_lens, num_heads, head_dim, partition_size, world, count, s,
                             max_seq_len=max_seq_len)
