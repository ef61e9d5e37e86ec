"""GPU parity of chunked-prefill (prefix) attention against the float64 oracle.

Small shapes cover several query tiles, context lengths that are and are not
multiples of the block size, chunks without context, every GQA group size up
to 8 and head_dim 64/128/256; the two named prefix workloads run at full size
and are checked on sampled rows.  Gather exactness (permuted pool) must be
bit-identical; device-side bad lengths and the forced timeout are exercised
without faulting.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_308_gb300 import binding as pb
from paged_kv_cache_308_gb300 import workloads as W
from parity_helpers import assert_parity, host_bits

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


# the tcgen05 (tensor-memory) kernel is the default (its persistent form), its
# grid form and the warp-level MMA kernel on request
IMPLS = {"tcgen05": {}, "tcgen05_grid": {"flags": pb.PA_FLAG_PREFIX_GRID},
         "warp_mma": {"flags": pb.PA_FLAG_PREFIX_WARP_MMA}}


@pytest.fixture(params=list(IMPLS))
def impl(request):
    return IMPLS[request.param]


def _oracle(w, threads=THREADS):
    return oracle.prefix_attention(host_bits(w.q), host_bits(w.k_new), host_bits(w.v_new), host_bits(w.k_cache),
                                   host_bits(w.v_cache), host_bits(w.block_tables), host_bits(w.context_lens),
                                   host_bits(w.query_start_loc), w.num_heads, w.num_kv_heads, w.head_dim,
                                   w.block_size, w.scale, threads=threads)


def _run(w, impl=None, **opt):
    out = pb.prefix_workload(w, **{**(impl or {}), **opt})
    torch.cuda.synchronize()
    st = pb.pa_get_device_status()
    assert st == 0, f"device status {st}"
    return out


@pytest.mark.parametrize("ctx,ql", [
    ([0], [1]), ([0], [70]), ([16], [16]), ([17], [33]), ([100, 0, 31], [5, 64, 11]),
    ([511, 512, 513], [1, 2, 130]), ([2048], [200]),
])
def test_small_gqa6_d256(dev, impl, ctx, ql):
    w = W.make_prefix_workload("p", ctx, ql, num_blocks=sum((c + 15) // 16 for c in ctx) + 5, seed=sum(ctx) + sum(ql),
                               device=dev, tail_fill=float("nan"))
    assert_parity(_run(w, impl), _oracle(w), f"ctx={ctx} ql={ql} {impl}")


@pytest.mark.parametrize("H,Hkv,D", [(4, 4, 64), (8, 4, 128), (16, 2, 256), (12, 4, 64), (7, 1, 256), (5, 5, 128)])
def test_group_sizes_and_head_dims(dev, impl, H, Hkv, D):
    w = W.make_prefix_workload("p", [300, 0, 45], [40, 17, 100], num_heads=H, num_kv_heads=Hkv, head_dim=D,
                               num_blocks=40, seed=H * D, device=dev, scale=1 / math.sqrt(D), tail_fill=float("inf"))
    assert_parity(_run(w, impl), _oracle(w), f"H={H} Hkv={Hkv} D={D} {impl}")


def test_single_new_token_matches_decode_over_the_extended_cache(dev, impl):
    # prefix attention of one new token == decode once that token is in the cache
    ctx = [40, 16, 1000]
    w = W.make_prefix_workload("p", ctx, [1, 1, 1], num_blocks=200, seed=3, device=dev)
    pre = _run(w, impl)
    k2, v2, bt2 = w.k_cache.clone(), w.v_cache.clone(), torch.cat(
        [w.block_tables, torch.full((3, 1), -1, dtype=torch.int32, device=dev)], 1)
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    free = [i for i in range(w.k_cache.shape[0]) if i not in used]
    for b, C in enumerate(ctx):
        if int(bt2[b, C // 16]) < 0:
            bt2[b, C // 16] = free.pop()
        k2[int(bt2[b, C // 16]), :, C % 16] = w.k_new[b]
        v2[int(bt2[b, C // 16]), :, C % 16] = w.v_new[b]
    d = W.Workload("d", w.q, k2, v2, bt2, torch.tensor([c + 1 for c in ctx], dtype=torch.int32, device=dev),
                   [c + 1 for c in ctx], w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale)
    dec = pb.decode_workload(d, mode="single")
    torch.cuda.synchronize()
    assert (pre.float() - dec.float()).abs().max().item() < 2e-3


@pytest.mark.parametrize("name", W.PREFIX_CONFIG_NAMES)
def test_named_prefix_workload_sampled(dev, impl, name):
    w = W.make_prefix_config(name, device=dev)
    out = _run(w, impl)
    assert torch.isfinite(out).all()
    hq, hkn, hvn = host_bits(w.q), host_bits(w.k_new), host_bits(w.v_new)
    hk, hv = host_bits(w.k_cache), host_bits(w.v_cache)
    hbt, hcl, hqs = host_bits(w.block_tables), host_bits(w.context_lens), host_bits(w.query_start_loc)
    rng = np.random.default_rng(0)
    toks = set()
    for b in range(len(w.query_lens_host)):
        a, e = int(hqs[b]), int(hqs[b + 1])
        if e > a:
            toks.update({a, e - 1, int(rng.integers(a, e))})
    ref, got = [], []
    for tok in sorted(toks):
        for h in (0, 5, 13, 23):
            ref.append(oracle.prefix_attention_one(hq, hkn, hvn, hk, hv, hbt, hcl, hqs, w.num_heads, w.num_kv_heads,
                                                   w.head_dim, w.block_size, w.scale, tok, h))
            got.append(out[tok, h])
    assert_parity(torch.stack(got), np.stack(ref), f"{name} sampled")


def test_permuted_pool_is_bit_identical(dev, impl):
    w = W.make_prefix_workload("p", [700, 33, 0], [50, 20, 9], num_blocks=120, seed=5, device=dev)
    a = _run(w, impl)
    g = torch.Generator(device=dev).manual_seed(2)
    perm = torch.randperm(w.k_cache.shape[0], generator=g, device=dev)
    k2, v2 = torch.empty_like(w.k_cache), torch.empty_like(w.v_cache)
    k2[perm], v2[perm] = w.k_cache, w.v_cache
    bt = w.block_tables.long()
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).to(torch.int32)
    w2 = W.PrefixWorkload(w.name, w.q, w.k_new, w.v_new, k2, v2, bt2, w.context_lens, w.query_start_loc,
                          w.context_lens_host, w.query_lens_host, w.num_heads, w.num_kv_heads, w.head_dim,
                          w.block_size, w.scale)
    assert torch.equal(a, _run(w2, impl))


def test_bad_context_length_sets_status(dev):
    w = W.make_prefix_workload("p", [40, 10], [4, 4], num_blocks=10, seed=6, device=dev)
    pb.pa_get_device_status()
    w.context_lens[0] = 41  # above the max_context_len bound of 40
    pb.prefix_workload(w)
    assert pb.pa_get_device_status() & pb.PA_DEV_BAD_SEQ_LEN


def test_forced_timeout_returns_status_and_context_survives(dev, impl):
    w = W.make_prefix_workload("p", [300, 20], [40, 9], num_blocks=40, seed=7, device=dev)
    pb.pa_get_device_status()
    pb.prefix_workload(w, flags=pb.PA_FLAG_FORCE_TIMEOUT | impl.get("flags", 0))
    assert pb.pa_get_device_status() & pb.PA_DEV_TIMEOUT
    assert_parity(_run(w, impl), _oracle(w), "after forced timeout")


def test_both_kernels_agree(dev):
    w = W.make_prefix_workload("p", [1000, 0, 77], [300, 129, 64], num_blocks=80, seed=8, device=dev)
    a = _run(w, IMPLS["tcgen05"])
    b = _run(w, IMPLS["warp_mma"])
    assert (a.float() - b.float()).abs().max().item() < 2e-3
