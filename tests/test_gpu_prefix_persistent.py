"""GPU parity of the tcgen05 prefill kernel's persistent form (the default)
against the float64 oracle and the grid form (PA_FLAG_PREFIX_GRID).

In the persistent form a grid of the CTAs the SMs hold at once claims the
query tiles (and key-split parts) from a device counter, carrying its copy
rings and barrier phases from one tile to the next.  Each tile is computed
by the same arithmetic, so the output must be bit-identical to the grid
form's, whatever CTA took the tile: ragged batches with tiles past a
sequence's new tokens, chunks without context, other group sizes and head
dims, forced key splits, the named workloads at full size.  The counter must
be re-armed by every call (repeats, a call after a forced timeout, a CUDA
graph replayed several times).
"""
import math
import os

import pytest
import torch

import oracle
from paged_kv_cache_308_gb300 import binding as pb
from paged_kv_cache_308_gb300 import workloads as W
from parity_helpers import assert_parity, host_bits

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1
GRID = pb.PA_FLAG_PREFIX_GRID


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


def _plain(w, **opt):
    return _check(pb.prefix_workload(w, **opt))


def _split(w, **kw):
    return _check(pb.prefix_split_workload(w, **kw))


@pytest.mark.parametrize("ctx,ql", [
    ([0], [1]), ([0], [70]), ([17], [33]), ([100, 0, 31], [5, 64, 11]),
    ([511, 512, 513], [1, 2, 130]), ([2048], [200]), ([3000, 17, 250, 0, 64], [300, 41, 1, 129, 7]),
])
def test_persistent_matches_the_oracle_and_the_grid_form(dev, ctx, ql):
    w = W.make_prefix_workload("p", ctx, ql, num_blocks=sum((c + 15) // 16 for c in ctx) + 5,
                               seed=3 * sum(ctx) + sum(ql), device=dev, tail_fill=float("nan"))
    out = _plain(w)
    assert_parity(out, _oracle(w), f"ctx={ctx} ql={ql} persistent")
    assert torch.equal(out, _plain(w, flags=GRID))


@pytest.mark.parametrize("H,Hkv,D", [(4, 4, 64), (8, 4, 128), (16, 2, 256), (12, 4, 64), (7, 1, 256), (5, 5, 128)])
def test_persistent_group_sizes_and_head_dims(dev, H, Hkv, D):
    w = W.make_prefix_workload("p", [300, 0, 45, 1200], [40, 17, 100, 260], num_heads=H, num_kv_heads=Hkv,
                               head_dim=D, num_blocks=120, seed=H * D + 5, device=dev, scale=1 / math.sqrt(D),
                               tail_fill=float("inf"))
    out = _plain(w)
    assert_parity(out, _oracle(w), f"H={H} Hkv={Hkv} D={D} persistent")
    assert torch.equal(out, _plain(w, flags=GRID))


@pytest.mark.parametrize("ctx,ql,parts,units", [
    ([2048], [200], 3, "all"),
    ([0], [70], 4, "all"),                 # parts without any key tile
    ([3000, 17], [300, 41], 7, 30),
    ([16], [16], 64, "all"),               # more parts than key tiles
    ([900, 0, 33], [129, 64, 1], 2, 4),
])
def test_persistent_forced_split(dev, ctx, ql, parts, units):
    w = W.make_prefix_workload("s", ctx, ql, num_blocks=sum((c + 15) // 16 for c in ctx) + 5,
                               seed=sum(ctx) + 11 * sum(ql), device=dev, tail_fill=float("nan"))
    n = _units(w)
    u = n if units == "all" else min(units, n)
    out = _split(w, parts=parts, units=u)
    assert_parity(out, _oracle(w), f"ctx={ctx} ql={ql} parts={parts} units={u} persistent")
    assert torch.equal(out, _split(w, parts=parts, units=u, flags=GRID))


@pytest.mark.parametrize("name", W.PREFIX_CONFIG_NAMES)
def test_named_workloads_bit_identical_to_the_grid_form(dev, name):
    w = W.make_prefix_config(name, device=dev)
    assert torch.equal(_plain(w), _plain(w, flags=GRID))
    assert torch.equal(_split(w), _split(w, flags=GRID))


def test_repeats_and_a_forced_timeout_rearm_the_counter(dev):
    w = W.make_prefix_workload("p", [1500, 33, 0, 400], [90, 20, 9, 200], num_blocks=150, seed=21, device=dev)
    ref = _plain(w, flags=GRID)
    for _ in range(3):
        assert torch.equal(_plain(w), ref)
    pb.pa_get_device_status()
    pb.prefix_workload(w, flags=pb.PA_FLAG_FORCE_TIMEOUT)
    assert pb.pa_get_device_status() & pb.PA_DEV_TIMEOUT
    assert torch.equal(_plain(w), ref)
    n = _units(w)
    pb.prefix_split_workload(w, parts=3, units=n, flags=pb.PA_FLAG_FORCE_TIMEOUT)
    assert pb.pa_get_device_status() & pb.PA_DEV_TIMEOUT
    assert torch.equal(_split(w, parts=3, units=n), _split(w, parts=3, units=n, flags=GRID))


def test_persistent_replays_from_a_cuda_graph(dev):
    w = W.make_prefix_workload("p", [1200, 300, 0], [100, 64, 150], num_blocks=120, seed=22, device=dev)
    ref = _plain(w, flags=GRID)
    out = torch.full_like(w.q, float("nan"))
    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        pb.prefix_workload(w, out=out, stream=s)  # allocates the counter, sets kernel attributes
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pb.prefix_workload(w, out=out, stream=s)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        _check(out)
        assert torch.equal(out, ref)


_CAPTURE_FIRST = r"""
import sys, torch
sys.path.insert(0, {root!r})
from paged_kv_cache_308_gb300 import binding as pb, workloads as W
dev = torch.device("cuda:0")
w = W.make_prefix_workload("p", [900, 40], [70, 33], num_blocks=80, seed=23, device=dev)
ref = pb.prefix_workload(w, flags=pb.PA_FLAG_PREFIX_GRID)  # kernel attributes set; no counter yet
torch.cuda.synchronize()
out = torch.full_like(w.q, float("nan"))
s = torch.cuda.Stream(device=dev)
s.wait_stream(torch.cuda.current_stream(dev))
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g, stream=s):
    pb.prefix_workload(w, out=out, stream=s)  # captured before the counter exists: the grid form
g.replay()
torch.cuda.synchronize()
assert pb.pa_get_device_status() == 0
assert torch.equal(out, ref)
fresh = pb.prefix_workload(w)  # outside a capture: allocates the counter, persistent form
torch.cuda.synchronize()
assert torch.equal(fresh, ref)
print("ok")
"""


def test_capture_before_the_counter_exists_keeps_the_grid_form(dev):
    # a fresh process: the counter is per process and device, and this one has it already
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _CAPTURE_FIRST.format(root=root)], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]


def test_concurrent_calls_on_two_streams(dev):
    # each stream has its own counter: two persistent calls in flight at once,
    # on different workloads, both give the grid form's bits
    a = W.make_prefix_workload("a", [3000, 17, 250], [300, 41, 129], num_blocks=240, seed=31, device=dev)
    b = W.make_prefix_workload("b", [900, 0, 4000, 64], [64, 200, 90, 7], num_blocks=340, seed=32, device=dev)
    ref_a, ref_b = _plain(a, flags=GRID), _plain(b, flags=GRID)
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    out_a, out_b = torch.empty_like(a.q), torch.empty_like(b.q)
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream(dev))
    for _ in range(5):
        out_a.fill_(float("nan"))
        out_b.fill_(float("nan"))
        s1.wait_stream(torch.cuda.current_stream(dev))
        s2.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s1):
            pb.prefix_workload(a, out=out_a, stream=s1)
        with torch.cuda.stream(s2):
            pb.prefix_workload(b, out=out_b, stream=s2)
        torch.cuda.synchronize()
        assert pb.pa_get_device_status() == 0
        assert torch.equal(out_a, ref_a) and torch.equal(out_b, ref_b)
