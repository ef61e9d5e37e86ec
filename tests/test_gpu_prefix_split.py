"""GPU parity of the key-split chunked prefill (pa_prefix_split) against the
float64 oracle.

pa_prefix_split runs the trailing query tiles of the grid as several CTAs,
each walking one range of the tile's key tiles, and merges their per-row
online-softmax states in a second kernel.  Forced splits (every part count
from 1 up, parts with no key tile at all, every tile split, ragged batches,
chunks without context, other group sizes and head dims, a negative scale)
are compared element by element with the oracle and with the unsplit call;
the library's own plan is checked on the named 4 x 8192 workload; repeats
and a permuted pool must be bit-identical; bad workspaces are refused.
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


def _oracle(w):
    return oracle.prefix_attention(host_bits(w.q), host_bits(w.k_new), host_bits(w.v_new), host_bits(w.k_cache),
                                   host_bits(w.v_cache), host_bits(w.block_tables), host_bits(w.context_lens),
                                   host_bits(w.query_start_loc), w.num_heads, w.num_kv_heads, w.head_dim,
                                   w.block_size, w.scale, threads=THREADS)


def _units(w):
    """Query tiles of the tensor-core kernel's grid (tile, kv head, sequence)."""
    tile_tokens = 128 // (w.num_heads // w.num_kv_heads)
    return -(-w.max_query_len // tile_tokens) * w.num_kv_heads * len(w.query_lens_host)


def _check(out):
    torch.cuda.synchronize()
    st = pb.pa_get_device_status()
    assert st == 0, f"device status {st}"
    return out


def _split(w, **kw):
    return _check(pb.prefix_split_workload(w, **kw))


def _plain(w, **opt):
    return _check(pb.prefix_workload(w, **opt))


@pytest.mark.parametrize("ctx,ql,parts,units", [
    ([2048], [200], 3, "all"),                       # every tile in three ranges
    ([511, 512, 513], [1, 2, 130], 2, 5),            # the five trailing tiles
    ([0], [70], 4, "all"),                           # chunk only: parts without any key tile
    ([100, 0, 31], [5, 64, 11], 5, "all"),
    ([700, 33, 0], [50, 20, 9], 1, "all"),           # one part: the partial and merge path alone
    ([3000, 17], [300, 41], 7, 30),
    ([16], [16], 64, "all"),                         # more parts than key tiles
])
def test_forced_split_matches_the_oracle(dev, ctx, ql, parts, units):
    w = W.make_prefix_workload("s", ctx, ql, num_blocks=sum((c + 15) // 16 for c in ctx) + 5,
                               seed=sum(ctx) + 7 * sum(ql), device=dev, tail_fill=float("nan"))
    n = _units(w)
    u = n if units == "all" else min(units, n)
    out = _split(w, parts=parts, units=u)
    assert_parity(out, _oracle(w), f"ctx={ctx} ql={ql} parts={parts} units={u}")
    assert (out.float() - _plain(w).float()).abs().max().item() < 2e-3


@pytest.mark.parametrize("H,Hkv,D", [(8, 4, 128), (4, 4, 64), (7, 1, 256), (16, 2, 256)])
def test_forced_split_group_sizes_and_head_dims(dev, H, Hkv, D):
    w = W.make_prefix_workload("s", [300, 0, 45], [40, 17, 100], num_heads=H, num_kv_heads=Hkv, head_dim=D,
                               num_blocks=40, seed=H * D + 1, device=dev, scale=1 / math.sqrt(D),
                               tail_fill=float("inf"))
    n = _units(w)
    assert_parity(_split(w, parts=2, units=max(1, n // 2)), _oracle(w), f"H={H} Hkv={Hkv} D={D}")


def test_forced_split_negative_scale(dev):
    w = W.make_prefix_workload("s", [900, 5], [60, 30], num_blocks=70, seed=11, device=dev, scale=-1 / 16)
    assert_parity(_split(w, parts=3, units=_units(w)), _oracle(w), "negative scale")


def test_split_repeats_and_permuted_pool_are_bit_identical(dev):
    w = W.make_prefix_workload("s", [1500, 33, 0], [90, 20, 9], num_blocks=120, seed=12, device=dev)
    kw = dict(parts=3, units=_units(w))
    a = _split(w, **kw)
    assert torch.equal(a, _split(w, **kw))
    g = torch.Generator(device=dev).manual_seed(4)
    perm = torch.randperm(w.k_cache.shape[0], generator=g, device=dev)
    k2, v2 = torch.empty_like(w.k_cache), torch.empty_like(w.v_cache)
    k2[perm], v2[perm] = w.k_cache, w.v_cache
    bt = w.block_tables.long()
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).to(torch.int32)
    w2 = W.PrefixWorkload(w.name, w.q, w.k_new, w.v_new, k2, v2, bt2, w.context_lens, w.query_start_loc,
                          w.context_lens_host, w.query_lens_host, w.num_heads, w.num_kv_heads, w.head_dim,
                          w.block_size, w.scale)
    assert torch.equal(a, _split(w2, **kw))


def test_library_plan_on_the_named_workload(dev):
    w = W.make_prefix_config("prefix_b4_c8192_q512", device=dev)
    # 400 tiles on the GPU's SMs: the last round is partly empty, so the plan splits
    assert pb.prefix_split_workspace_size(w) > 0
    out = _split(w)
    assert torch.isfinite(out).all()
    assert (out.float() - _plain(w).float()).abs().max().item() < 2e-3
    hq, hkn, hvn = host_bits(w.q), host_bits(w.k_new), host_bits(w.v_new)
    hk, hv = host_bits(w.k_cache), host_bits(w.v_cache)
    hbt, hcl, hqs = host_bits(w.block_tables), host_bits(w.context_lens), host_bits(w.query_start_loc)
    rng = np.random.default_rng(1)
    ref, got = [], []
    # the last sequence holds the split tiles; sample it and the others
    for tok in sorted({0, 511, 1024, 1535, 1536, 2047} | set(rng.integers(1536, 2048, 6).tolist())):
        for h in (0, 7, 23):
            ref.append(oracle.prefix_attention_one(hq, hkn, hvn, hk, hv, hbt, hcl, hqs, w.num_heads, w.num_kv_heads,
                                                   w.head_dim, w.block_size, w.scale, tok, h))
            got.append(out[tok, h])
    assert_parity(torch.stack(got), np.stack(ref), "prefix_b4_c8192_q512 split, sampled")


def test_mixed_workload_under_the_library_plan(dev):
    w = W.make_prefix_config("prefix_b16_mixed", device=dev)
    # 3136 tiles, about 21 rounds of a ragged batch: the plan splits nothing
    assert pb.prefix_split_workspace_size(w) == 0
    out = _split(w)
    assert torch.isfinite(out).all()
    assert (out.float() - _plain(w).float()).abs().max().item() < 2e-3


def test_no_split_planned_needs_no_workspace(dev):
    w = W.make_prefix_workload("s", [40], [5], num_blocks=5, seed=13, device=dev)
    assert pb.prefix_split_workspace_size(w) == 0
    assert torch.equal(_split(w), _plain(w))


def test_warp_mma_flag_splits_nothing(dev):
    w = W.make_prefix_workload("s", [300, 20], [40, 9], num_blocks=40, seed=14, device=dev)
    a = _split(w, parts=3, units=_units(w), flags=pb.PA_FLAG_PREFIX_WARP_MMA)
    assert torch.equal(a, _plain(w, flags=pb.PA_FLAG_PREFIX_WARP_MMA))


def test_bad_workspace_and_split_are_refused(dev):
    w = W.make_prefix_workload("s", [300, 20], [40, 9], num_blocks=40, seed=15, device=dev)
    n = _units(w)
    need = pb.prefix_split_workspace_size(w, parts=2, units=n)
    assert need > 0
    ws = torch.empty(need + 512, dtype=torch.uint8, device=dev)
    for bad in (dict(workspace=ws[: need - 1]), dict(workspace=ws[16: 16 + need])):
        with pytest.raises(pb.PaDecodeError) as e:
            pb.prefix_split_workload(w, parts=2, units=n, **bad)
        assert e.value.code == pb.PA_ERR_INVALID_ARG
    for parts, units in ((65, 1), (-1, 1), (2, n + 1), (2, -1)):
        with pytest.raises(pb.PaDecodeError) as e:
            pb.prefix_split_workload(w, parts=parts, units=units, workspace=ws)
        assert e.value.code == pb.PA_ERR_INVALID_ARG
    # the exact size is enough
    assert_parity(_split(w, parts=2, units=n, workspace=ws[:need]), _oracle(w), "exact workspace")


def test_forced_timeout_in_a_split_returns_status_and_context_survives(dev):
    w = W.make_prefix_workload("s", [600, 20], [40, 9], num_blocks=60, seed=16, device=dev)
    kw = dict(parts=3, units=_units(w))
    pb.pa_get_device_status()
    pb.prefix_split_workload(w, flags=pb.PA_FLAG_FORCE_TIMEOUT, **kw)
    assert pb.pa_get_device_status() & pb.PA_DEV_TIMEOUT
    assert_parity(_split(w, **kw), _oracle(w), "after forced timeout")


def test_split_replays_from_a_cuda_graph(dev):
    w = W.make_prefix_workload("s", [1200, 300], [100, 64], num_blocks=120, seed=17, device=dev)
    kw = dict(parts=3, units=_units(w))
    ws = torch.empty(pb.prefix_split_workspace_size(w, **kw), dtype=torch.uint8, device=dev)
    out = torch.full_like(w.q, float("nan"))
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        pb.prefix_split_workload(w, out=out, stream=s, workspace=ws, **kw)  # warm-up (kernel attributes)
    s.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pb.prefix_split_workload(w, out=out, stream=s, workspace=ws, **kw)
    g.replay()
    _check(out)
    assert_parity(out, _oracle(w), "graph replay")
