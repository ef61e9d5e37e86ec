"""Seeded synthetic decode workloads (inputs only; no attention arithmetic).

This module is shared by the tests, the benchmark and the smoke check.  It
builds the inputs of one decode call -- q, a block-tabled K/V pool, block
tables and sequence lengths -- and nothing else: it imports neither the CUDA
binding nor the oracle.

Cache layout (both K and V): ``[num_blocks, num_kv_heads, block_size, head_dim]``
fp16, so one (block, kv head) is ``block_size * head_dim`` contiguous halves.

Recipes of the five named workloads (heads 24 query / 4 kv, head_dim 256,
block_size 16, q/K/V fp16 ~ N(0, 1), scale 1/16, partition 512 tokens):

* ``b1_l2048``            1 sequence of 2048 tokens; pool of exactly 128 blocks,
                          block table = a seeded permutation of them.
* ``b8_u8192``            8 sequences, lengths uniform on [1, 8192]; pool of
                          8192 blocks, disjoint random blocks per sequence.
* ``b4_l32768_peaked``    4 x 32768 tokens, pool of 8192 blocks; 1% of the
                          token positions of every sequence (drawn without
                          replacement) have their key multiplied by 8 in every
                          kv head (exact in fp16), making the softmax peaked.
* ``b1_l102400``          1 sequence of 102400 tokens (200 partitions of 512);
                          pool of exactly 6400 blocks in a seeded permutation.
* ``b64_loguniform``      64 sequences, lengths round(exp(U(ln 16, ln 65536)));
                          shared pool of 1.5 * 2^20 tokens = 98304 blocks,
                          disjoint random blocks per sequence.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional

import torch

NUM_HEADS = 24
NUM_KV_HEADS = 4
HEAD_DIM = 256
BLOCK_SIZE = 16
PARTITION_SIZE = 512
SCALE = 1.0 / 16.0


@dataclass
class Workload:
    name: str
    q: torch.Tensor              # fp16 [B, H, D]
    k_cache: torch.Tensor        # fp16 [NB, Hkv, bs, D]
    v_cache: torch.Tensor        # fp16 [NB, Hkv, bs, D]
    block_tables: torch.Tensor   # int32 [B, max_blocks_per_seq]
    seq_lens: torch.Tensor       # int32 [B]
    seq_lens_host: List[int]
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    partition_size: int = PARTITION_SIZE
    peaked_positions: Optional[List[List[int]]] = field(default=None, repr=False)

    @property
    def num_seqs(self) -> int:
        return len(self.seq_lens_host)

    @property
    def max_seq_len(self) -> int:
        return max(self.seq_lens_host) if self.seq_lens_host else 0

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_lens_host))

    @property
    def kv_bytes(self) -> int:
        """K and V bytes one call must read: sum_b L_b * Hkv * D * 2 B * 2."""
        return self.total_tokens * self.num_kv_heads * self.head_dim * 2 * 2

    def to(self, device) -> "Workload":
        mv = lambda t: t.to(device)
        return Workload(self.name, mv(self.q), mv(self.k_cache), mv(self.v_cache),
                        mv(self.block_tables), mv(self.seq_lens), list(self.seq_lens_host),
                        self.num_heads, self.num_kv_heads, self.head_dim, self.block_size,
                        self.scale, self.partition_size, self.peaked_positions)


def _normal_fp16(shape, gen: torch.Generator, device) -> torch.Tensor:
    """N(0,1) rounded to fp16, drawn in chunks so large pools need little scratch."""
    out = torch.empty(shape, dtype=torch.float16, device=device)
    flat = out.view(-1)
    chunk = 1 << 26
    for s in range(0, flat.numel(), chunk):
        e = min(flat.numel(), s + chunk)
        flat[s:e] = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32).to(torch.float16)
    return out


def _device_generator(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_workload(name: str, seq_lens: List[int], *, num_heads: int = NUM_HEADS,
                  num_kv_heads: int = NUM_KV_HEADS, head_dim: int = HEAD_DIM,
                  block_size: int = BLOCK_SIZE, num_blocks: Optional[int] = None,
                  scale: float = SCALE, partition_size: int = PARTITION_SIZE, seed: int = 0,
                  device="cpu", peaked_fraction: float = 0.0, peak_factor: float = 8.0,
                  tail_fill: Optional[float] = None, extra_table_cols: int = 0) -> Workload:
    """Build one workload.

    Blocks are handed out disjointly from a seeded permutation of the pool;
    the unused tail of every block-table row holds -1.  ``tail_fill`` writes a
    value (e.g. NaN) into the slots of each sequence's last block that lie
    past its length, to check that they are excluded.
    """
    host = torch.Generator().manual_seed(seed)
    seq_lens = [int(x) for x in seq_lens]
    nblk = [(L + block_size - 1) // block_size for L in seq_lens]
    need = sum(nblk)
    if num_blocks is None:
        num_blocks = max(need, 1)
    if need > num_blocks:
        raise ValueError(f"pool of {num_blocks} blocks cannot hold {need}")
    mbps = max(max(nblk, default=0), 1) + extra_table_cols
    perm = torch.randperm(num_blocks, generator=host)
    bt = torch.full((len(seq_lens), mbps), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n].to(torch.int32)
        off += n
    dev_gen = _device_generator(device, seed + 1)
    q = _normal_fp16((len(seq_lens), num_heads, head_dim), dev_gen, device)
    k = _normal_fp16((num_blocks, num_kv_heads, block_size, head_dim), dev_gen, device)
    v = _normal_fp16((num_blocks, num_kv_heads, block_size, head_dim), dev_gen, device)
    peaked = None
    if peaked_fraction > 0:
        peaked = []
        for b, L in enumerate(seq_lens):
            n = int(round(peaked_fraction * L))
            pos = torch.randperm(L, generator=host)[:n].sort().values
            peaked.append(pos.tolist())
            if n == 0:
                continue
            phys = bt[b, (pos // block_size).long()].long().to(device)
            slot = (pos % block_size).long().to(device)
            k[phys, :, slot, :] = k[phys, :, slot, :] * peak_factor
    if tail_fill is not None:
        for b, L in enumerate(seq_lens):
            if L % block_size:
                phys = int(bt[b, L // block_size])
                k[phys, :, L % block_size:, :] = tail_fill
                v[phys, :, L % block_size:, :] = tail_fill
    return Workload(name, q, k, v, bt.to(device), torch.tensor(seq_lens, dtype=torch.int32, device=device),
                    seq_lens, num_heads, num_kv_heads, head_dim, block_size, scale, partition_size, peaked)


def config_seq_lens(name: str, seed: int = 0) -> List[int]:
    g = torch.Generator().manual_seed(seed)
    if name == "b1_l2048":
        return [2048]
    if name == "b8_u8192":
        return torch.randint(1, 8192 + 1, (8,), generator=g).tolist()
    if name == "b4_l32768_peaked":
        return [32768] * 4
    if name == "b1_l102400":
        return [102400]
    if name == "b64_loguniform":
        u = torch.rand(64, generator=g, dtype=torch.float64)
        lo, hi = math.log(16.0), math.log(65536.0)
        return [int(round(math.exp(lo + (hi - lo) * float(x)))) for x in u]
    raise KeyError(name)


CONFIG_NAMES = ["b1_l2048", "b8_u8192", "b4_l32768_peaked", "b1_l102400", "b64_loguniform"]

_POOL = {"b1_l2048": None, "b8_u8192": 8192, "b4_l32768_peaked": 8192, "b1_l102400": None,
         "b64_loguniform": 98304}


def make_config(name: str, device="cpu", seed: int = 0, **kw) -> Workload:
    """One of the five named workloads (see the module docstring)."""
    lens = config_seq_lens(name, seed)
    peaked = 0.01 if name == "b4_l32768_peaked" else 0.0
    return make_workload(name, lens, num_blocks=_POOL[name], seed=seed, device=device,
                         peaked_fraction=peaked, **kw)


@dataclass
class PrefixWorkload:
    """Inputs of one chunked-prefill call: per sequence, context_lens[b]
    cached tokens (paged, as for decode) and a chunk of new tokens packed
    in q / k_new / v_new at rows query_start_loc[b] .. [b+1]-1."""
    name: str
    q: torch.Tensor                # fp16 [T, H, D]
    k_new: torch.Tensor            # fp16 [T, Hkv, D]
    v_new: torch.Tensor            # fp16 [T, Hkv, D]
    k_cache: torch.Tensor          # fp16 [NB, Hkv, bs, D]
    v_cache: torch.Tensor
    block_tables: torch.Tensor     # int32 [B, max_blocks_per_seq]
    context_lens: torch.Tensor     # int32 [B]
    query_start_loc: torch.Tensor  # int32 [B + 1]
    context_lens_host: List[int]
    query_lens_host: List[int]
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float

    @property
    def num_tokens(self) -> int:
        return int(sum(self.query_lens_host))

    @property
    def max_context_len(self) -> int:
        return max(self.context_lens_host) if self.context_lens_host else 0

    @property
    def max_query_len(self) -> int:
        return max(self.query_lens_host) if self.query_lens_host else 0

    @property
    def flops(self) -> int:
        """Score and P.V multiply-adds x 2: per new token i of a sequence with
        context C, (C + i + 1) keys x heads x head_dim x 2 products x 2."""
        keys = sum(C * L + L * (L + 1) // 2 for C, L in zip(self.context_lens_host, self.query_lens_host))
        return 4 * keys * self.num_heads * self.head_dim


def make_prefix_workload(name: str, context_lens: List[int], query_lens: List[int], *, num_heads: int = NUM_HEADS,
                         num_kv_heads: int = NUM_KV_HEADS, head_dim: int = HEAD_DIM, block_size: int = BLOCK_SIZE,
                         num_blocks: Optional[int] = None, scale: float = SCALE, seed: int = 0, device="cpu",
                         tail_fill: Optional[float] = None) -> PrefixWorkload:
    base = make_workload(name, context_lens, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                         block_size=block_size, num_blocks=num_blocks, scale=scale, seed=seed, device=device,
                         tail_fill=tail_fill)
    gen = _device_generator(device, seed + 7)
    T = int(sum(query_lens))
    qs = [0]
    for L in query_lens:
        qs.append(qs[-1] + int(L))
    q = _normal_fp16((T, num_heads, head_dim), gen, device)
    kn = _normal_fp16((T, num_kv_heads, head_dim), gen, device)
    vn = _normal_fp16((T, num_kv_heads, head_dim), gen, device)
    return PrefixWorkload(name, q, kn, vn, base.k_cache, base.v_cache, base.block_tables, base.seq_lens,
                          torch.tensor(qs, dtype=torch.int32, device=device), list(base.seq_lens_host),
                          [int(x) for x in query_lens], num_heads, num_kv_heads, head_dim, block_size, scale)


PREFIX_CONFIG_NAMES = ["prefix_b4_c8192_q512", "prefix_b16_mixed"]


def make_prefix_config(name: str, device="cpu", seed: int = 0) -> PrefixWorkload:
    """Chunked-prefill workloads (24/4 heads, head_dim 256, block_size 16):

    * ``prefix_b4_c8192_q512``  4 sequences, 8192 cached tokens each, chunks of 512;
    * ``prefix_b16_mixed``      16 sequences, cached lengths log-uniform on
                                [16, 32768] (0 for two of them), chunks uniform
                                on [1, 1024]."""
    if name == "prefix_b4_c8192_q512":
        return make_prefix_workload(name, [8192] * 4, [512] * 4, seed=seed, device=device)
    if name == "prefix_b16_mixed":
        g = torch.Generator().manual_seed(seed)
        u = torch.rand(16, generator=g, dtype=torch.float64)
        lo, hi = math.log(16.0), math.log(32768.0)
        ctx = [int(round(math.exp(lo + (hi - lo) * float(x)))) for x in u]
        ctx[3] = ctx[11] = 0
        ql = torch.randint(1, 1025, (16,), generator=g).tolist()
        return make_prefix_workload(name, ctx, ql, seed=seed, device=device)
    raise KeyError(name)

