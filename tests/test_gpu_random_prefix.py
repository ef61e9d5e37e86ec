"""Seeded random sweep of chunked-prefill shapes on the GPU against the float64 oracle.

Each case draws a batch of sequences with context lengths (0, inside a block,
on a block boundary, a few blocks) and chunk lengths (1 to a few query
tiles), a GQA ratio and a head_dim, and runs both prefix kernels (tcgen05 and
warp-level MMA) through the C ABI; every output element is compared with the
oracle.  A second sweep runs the key split (pa_prefix_split) with random
forced splits.  The draws come from a fixed seed.
"""
import os
import random

import pytest
import torch

import oracle
from paged_kv_cache_308_gb300 import binding as pb
from paged_kv_cache_308_gb300 import workloads as W
from parity_helpers import assert_parity, host_bits

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1


def draw_case(i):
    r = random.Random(2000 + i)
    hkv = r.choice([1, 2, 4])
    g = r.choice([1, 2, 4, 6, 8])
    d = r.choice([64, 128, 256])
    b = r.choice([1, 2, 3, 5])
    ctx = [r.choice([0, 1, 15, 16, 17, 64, 200, r.randint(1, 900)]) for _ in range(b)]
    ql = [r.choice([1, 2, 21, 22, 64, r.randint(1, 160)]) for _ in range(b)]
    return dict(ctx=ctx, ql=ql, num_heads=hkv * g, num_kv_heads=hkv, head_dim=d, seed=i)


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.mark.parametrize("flags", [0, pb.PA_FLAG_PREFIX_WARP_MMA], ids=["tcgen05", "warp_mma"])
@pytest.mark.parametrize("i", range(16))
def test_random_prefix_case(dev, i, flags):
    c = draw_case(i)
    w = W.make_prefix_workload(f"prand{i}", c["ctx"], c["ql"], num_heads=c["num_heads"],
                               num_kv_heads=c["num_kv_heads"], head_dim=c["head_dim"], seed=c["seed"], device=dev)
    out = pb.prefix_workload(w, flags=flags)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    ref = oracle.prefix_attention(host_bits(w.q), host_bits(w.k_new), host_bits(w.v_new), host_bits(w.k_cache),
                                  host_bits(w.v_cache), host_bits(w.block_tables), host_bits(w.context_lens),
                                  host_bits(w.query_start_loc), w.num_heads, w.num_kv_heads, w.head_dim,
                                  w.block_size, w.scale, threads=THREADS)
    assert_parity(out, ref, f"prefix case {i}: {c}")


@pytest.mark.parametrize("i", range(12))
def test_random_prefix_split_case(dev, i):
    # the key split (pa_prefix_split) on the same kind of draws, with a forced
    # split: a random number of key ranges for a random run of trailing tiles
    c = draw_case(100 + i)
    r = random.Random(3000 + i)
    w = W.make_prefix_workload(f"psplit{i}", c["ctx"], c["ql"], num_heads=c["num_heads"],
                               num_kv_heads=c["num_kv_heads"], head_dim=c["head_dim"], seed=c["seed"], device=dev,
                               tail_fill=float("nan"))
    tile_tokens = 128 // (w.num_heads // w.num_kv_heads)
    n = -(-w.max_query_len // tile_tokens) * w.num_kv_heads * len(c["ql"])
    parts, units = r.randint(1, 9), r.randint(1, n)
    out = pb.prefix_split_workload(w, parts=parts, units=units)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    ref = oracle.prefix_attention(host_bits(w.q), host_bits(w.k_new), host_bits(w.v_new), host_bits(w.k_cache),
                                  host_bits(w.v_cache), host_bits(w.block_tables), host_bits(w.context_lens),
                                  host_bits(w.query_start_loc), w.num_heads, w.num_kv_heads, w.head_dim,
                                  w.block_size, w.scale, threads=THREADS)
    assert_parity(out, ref, f"prefix split case {i}: {c} parts={parts} units={units} of {n}")
