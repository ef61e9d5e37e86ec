"""GPU parity of the CUDA decode path against the float64 oracle, through the C ABI.

Small shapes cover several tiles and ragged tails in every mode; the five
named workloads run at full size in the launch configuration the benchmark
times, every output element compared with the oracle.  Gather exactness
(permuted pool, sequence alone vs in a batch, repeat runs) must be
bit-identical, also on the one-wave plan of one long sequence.  Device-side error paths are exercised without faulting: bad
block ids and lengths are caught by the kernel's own checks, and the forced
timeout makes the bounded waits give up.
"""
import math
import os

import numpy as np
import pytest
import torch

from paged_kv_cache_308_gb300 import binding as pb
from paged_kv_cache_308_gb300 import workloads as W
from parity_helpers import assert_parity, compare, oracle_ref, oracle_ref_subset

pytestmark = pytest.mark.gpu
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def run(w, **opt):
    out = pb.decode_workload(w, **opt)
    torch.cuda.synchronize()
    st = pb.pa_get_device_status()
    assert st == 0, f"device status {st}"
    return out


SMALL_LENS = [[1], [15], [16], [17], [511], [512], [513], [1, 16, 17, 511, 512, 513, 1029], [2048, 3, 700]]
MODES = [dict(), dict(mode="single"), dict(mode="split", partition_size=16), dict(mode="split", partition_size=64),
         dict(mode="split", partition_size=512), dict(mode="split", partition_size=1024),
         dict(mode="fused", partition_size=16), dict(mode="fused", partition_size=512),
         dict(mode="persistent"), dict(mode="persistent", partition_size=64), dict(mode="flat")]


@pytest.mark.parametrize("lens", SMALL_LENS, ids=lambda x: "L" + "-".join(map(str, x)))
@pytest.mark.parametrize("opt", MODES, ids=lambda o: "-".join(f"{v}" for v in o.values()) or "default")
def test_small_gqa6_d256(dev, lens, opt):
    w = W.make_workload("small", lens, num_blocks=sum((L + 15) // 16 for L in lens) + 7, seed=len(lens) + lens[0],
                        device=dev, tail_fill=float("nan"))
    out = run(w, **opt)
    assert_parity(out, oracle_ref(w), f"lens={lens} {opt}")


@pytest.mark.parametrize("H,Hkv,D", [(4, 4, 64), (8, 4, 128), (16, 2, 256), (12, 4, 64), (12, 2, 128),
                                     (16, 4, 256), (5, 5, 128), (7, 1, 256)])
@pytest.mark.parametrize("mode", ["single", "split", "fused", "persistent", "flat"])
def test_group_sizes_and_head_dims(dev, H, Hkv, D, mode):
    lens = [1, 37, 700, 1500, 16 * 33]
    w = W.make_workload("shape", lens, num_heads=H, num_kv_heads=Hkv, head_dim=D, num_blocks=300, seed=H * D,
                        device=dev, scale=1 / math.sqrt(D), tail_fill=float("inf"))
    out = run(w, mode=mode, partition_size=0 if mode in ("single", "flat") else 256)
    assert_parity(out, oracle_ref(w), f"H={H} Hkv={Hkv} D={D} {mode}")


@pytest.mark.parametrize("name,opt", [
    ("b1_l2048", dict()),
    ("b1_l2048", dict(mode="single")),
    ("b8_u8192", dict(mode="single")),
    ("b8_u8192", dict(mode="split")),
    ("b8_u8192", dict()),
    ("b8_u8192", dict(mode="fused")),
    ("b1_l2048", dict(mode="fused", partition_size=128)),
    ("b4_l32768_peaked", dict()),
    ("b1_l102400", dict()),
    ("b1_l102400", dict(mode="fused")),
    ("b8_u8192", dict(mode="persistent")),
    ("b4_l32768_peaked", dict(mode="persistent")),
    ("b1_l102400", dict(mode="persistent")),
    ("b1_l2048", dict(mode="flat")),
    ("b8_u8192", dict(mode="flat")),
    ("b4_l32768_peaked", dict(mode="flat")),
    ("b1_l102400", dict(mode="flat")),
])
def test_named_workload_full(dev, name, opt):
    w = W.make_config(name, device=dev)
    out = run(w, **opt) if opt else pb.decode_workload(w)  # the benchmark's call: library workspace, AUTO
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    r = assert_parity(out, oracle_ref(w, THREADS), f"{name} {opt}")
    print(name, opt, r)


@pytest.mark.parametrize("opt", [dict(), dict(mode="persistent"), dict(mode="split", partition_size=512),
                                 dict(mode="flat")],
                         ids=["default", "persistent", "split512", "flat"])
def test_mixed_batch_full(dev, opt):
    # all 64 sequences, element by element; the oracle reads only the blocks
    # the batch uses (gathered into a compact pool), not the whole 1.5M-token pool
    w = W.make_config("b64_loguniform", device=dev)
    out = pb.decode_workload(w, **opt)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    ref = oracle_ref_subset(w, range(w.num_seqs), THREADS)
    r = assert_parity(out, ref, f"b64_loguniform {opt}")
    print("b64_loguniform", opt, r)


def test_peaked_keys_both_modes(dev):
    w = W.make_workload("peaked", [4096, 777], num_blocks=400, seed=3, device=dev, peaked_fraction=0.01)
    ref = oracle_ref(w)
    for opt in (dict(mode="single"), dict(mode="split", partition_size=512), dict(mode="split", partition_size=32)):
        assert_parity(run(w, **opt), ref, f"peaked {opt}")


def _permuted_pool(w, seed):
    g = torch.Generator(device=w.k_cache.device).manual_seed(seed)
    perm = torch.randperm(w.num_blocks, generator=g, device=w.k_cache.device)
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt = w.block_tables.long()
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).to(torch.int32)
    return W.Workload(w.name, w.q, k2, v2, bt2, w.seq_lens, w.seq_lens_host, w.num_heads, w.num_kv_heads,
                      w.head_dim, w.block_size, w.scale, w.partition_size)


@pytest.mark.parametrize("opt", [dict(mode="single"), dict(mode="split", partition_size=512),
                                 dict(mode="split", partition_size=48), dict(mode="persistent"),
                                 dict(mode="fused", partition_size=512), dict(mode="flat")])
def test_permuted_block_table_is_bit_identical(dev, opt):
    w = W.make_workload("perm", [3000, 517, 8000, 1], num_blocks=900, seed=5, device=dev)
    a = run(w, **opt)
    b = run(_permuted_pool(w, 11), **opt)
    assert torch.equal(a, b)
    # the identity table over a freshly laid out pool gives the same bits too
    assert torch.equal(a, run(_permuted_pool(w, 12), **opt))


@pytest.mark.parametrize("opt", [dict(flags=pb.PA_FLAG_DETERMINISTIC),
                                 dict(mode="fused", flags=pb.PA_FLAG_DETERMINISTIC)],
                         ids=["one_wave_deterministic", "fused"])
def test_permuted_block_table_is_bit_identical_on_one_long_sequence(dev, opt):
    # the plan the benchmark times for one long sequence (one wave of one
    # 4-warp CTA per SM), with fixed partitions; and the fused combine
    w = W.make_workload("permlong", [96000], num_blocks=96000 // 16 + 37, seed=24, device=dev)
    if "flags" in opt:
        plan = pb.pa_decode_plan(torch.empty_like(w.q), w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                                 w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                                 max_seq_len=w.max_seq_len, **opt)
        assert plan["partition_size"] > 2048 and plan["threads"] == 128 and plan["pooled"] == 0
    a = run(w, **opt)
    assert torch.equal(a, run(_permuted_pool(w, 25), **opt))
    assert torch.equal(a, run(_permuted_pool(w, 26), **opt))
    assert_parity(a, oracle_ref(w, THREADS), f"permuted long {opt}")


def test_sequence_alone_and_in_batch_are_bit_identical(dev):
    w = W.make_workload("batch", [5000, 123, 2048, 999], num_blocks=700, seed=6, device=dev)
    full = run(w, mode="split", partition_size=512)
    for b in range(w.num_seqs):
        one = W.Workload(w.name, w.q[b:b + 1].contiguous(), w.k_cache, w.v_cache,
                         w.block_tables[b:b + 1].contiguous(), w.seq_lens[b:b + 1].contiguous(),
                         [w.seq_lens_host[b]], w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale)
        assert torch.equal(full[b:b + 1], run(one, mode="split", partition_size=512))


def test_repeat_runs_are_bit_identical(dev):
    w = W.make_config("b8_u8192", device=dev)
    a = run(w)
    for _ in range(3):
        assert torch.equal(a, run(w))


def test_single_key_returns_v_exactly(dev):
    w = W.make_workload("one", [1, 1, 1], num_blocks=9, seed=7, device=dev, tail_fill=float("nan"))
    for opt in (dict(mode="single"), dict(mode="split", partition_size=16)):
        out = run(w, **opt)
        for b in range(3):
            phys = int(w.block_tables[b, 0])
            for h in range(w.num_heads):
                assert torch.equal(out[b, h], w.v_cache[phys, h // 6, 0])


def test_empty_sequences_give_zero(dev):
    w = W.make_workload("empty", [0, 600, 0, 17], num_blocks=50, seed=8, device=dev)
    for opt in (dict(mode="single"), dict(mode="split", partition_size=128)):
        out = run(w, **opt)
        assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[2]) == 0
        assert_parity(out, oracle_ref(w), f"empty {opt}")
    allempty = W.make_workload("allempty", [0, 0], num_blocks=4, seed=9, device=dev)
    assert torch.count_nonzero(run(allempty)) == 0


def test_library_and_caller_workspace_calls_agree(dev):
    w = W.make_config("b1_l2048", device=dev)
    a = pb.decode_workload(w)
    b = run(w, mode="auto")
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_graph_capture_of_caller_workspace_call(dev):
    w = W.make_workload("graph", [4000, 100, 2500], num_blocks=500, seed=10, device=dev)
    out = torch.empty_like(w.q)
    kw = dict(max_seq_len=w.max_seq_len, mode="split", partition_size=512)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, **kw)
    ws = pb.alloc_workspace(plan, dev)
    args = (out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads, w.head_dim,
            w.block_size, w.scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pb.pa_decode_ex(*args, s, workspace=ws, **kw)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pb.pa_decode_ex(*args, torch.cuda.current_stream(), workspace=ws, **kw)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


def test_bad_block_id_sets_device_status(dev):
    w = W.make_workload("badid", [100, 40], num_blocks=20, seed=11, device=dev)
    pb.pa_get_device_status()  # clear
    w.block_tables[0, 2] = w.num_blocks + 3
    w.block_tables[1, 0] = -5
    pb.decode_workload(w, mode="split", partition_size=32)
    assert pb.pa_get_device_status() & pb.PA_DEV_BAD_BLOCK_ID
    assert pb.pa_get_device_status() == 0  # reading clears it


def test_bad_seq_len_sets_device_status(dev):
    w = W.make_workload("badlen", [100, 40], num_blocks=20, seed=12, device=dev, extra_table_cols=4)
    pb.pa_get_device_status()
    out = torch.empty_like(w.q)
    w.seq_lens[1] = 101  # above the max_seq_len hint of 100
    pb.pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                 w.head_dim, w.block_size, w.scale, max_seq_len=100)
    assert pb.pa_get_device_status() & pb.PA_DEV_BAD_SEQ_LEN


def test_forced_timeout_returns_status_and_context_survives(dev):
    w = W.make_workload("timeout", [3000, 64], num_blocks=200, seed=13, device=dev)
    pb.pa_get_device_status()
    for mode in ("single", "split", "fused", "persistent", "flat"):
        pb.decode_workload(w, mode=mode, partition_size=0 if mode in ("single", "flat") else 512,
                           flags=pb.PA_FLAG_FORCE_TIMEOUT)
        assert pb.pa_get_device_status() & pb.PA_DEV_TIMEOUT
    # the context is still healthy: a normal call afterwards is correct
    assert_parity(run(w), oracle_ref(w), "after forced timeout")


def test_caller_workspace_too_small_is_rejected(dev):
    w = W.make_workload("ws", [2000], num_blocks=200, seed=14, device=dev)
    out = torch.empty_like(w.q)
    small = torch.empty(64, dtype=torch.uint8, device=dev)
    with pytest.raises(pb.PaDecodeError) as e:
        pb.pa_decode_ex(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                        w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len, mode="split",
                        workspace=small)
    assert e.value.code == pb.PA_ERR_WORKSPACE


@pytest.mark.parametrize("warps,stages", [(2, 2), (1, 2), (1, 3), (4, 2)])
@pytest.mark.parametrize("mode", ["single", "split"])
def test_every_cta_shape(dev, warps, stages, mode):
    w = W.make_workload("shape", [1, 17, 513, 3000, 100], num_blocks=300, seed=warps * 10 + stages, device=dev,
                        tail_fill=float("nan"))
    out = run(w, mode=mode, partition_size=256 if mode == "split" else 0, warps=warps, stages=stages)
    assert_parity(out, oracle_ref(w), f"{warps}x{stages} {mode}")
    # the result does not depend on the CTA shape beyond rounding order
    ref = run(w, mode=mode, partition_size=256 if mode == "split" else 0, warps=2, stages=2)
    assert (out.float() - ref.float()).abs().max().item() < 2e-3


def _fused_call(w, out, ws, stream=None, **extra):
    pb.pa_decode_ex(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                    w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len, mode="fused",
                    partition_size=128, workspace=ws, **extra)


def _tickets(w, ws, plan_split_bytes):
    # after the partials and a slot the size of the pooled claim counters: two
    # 4-byte words per (sequence, kv head)
    off = plan_split_bytes + (8 * len(w.seq_lens_host) * w.num_kv_heads + 255) // 256 * 256
    return ws[off:off + 8 * len(w.seq_lens_host) * w.num_kv_heads]


def test_fused_combine_is_deterministic_and_leaves_tickets_zero(dev):
    w = W.make_workload("fused", [3000, 17, 1029, 513, 128, 1], num_blocks=400, seed=15, device=dev,
                        tail_fill=float("nan"))
    out = torch.empty_like(w.q)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len,
                             mode="fused", partition_size=128)
    split = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                              w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len,
                              mode="split", partition_size=128)
    assert plan["launch_reduce"] == 0 and plan["workspace_bytes"] > split["workspace_bytes"]
    ws = pb.alloc_workspace(plan, dev)
    outs = []
    for _ in range(4):
        _fused_call(w, out, ws)
        torch.cuda.synchronize()
        assert pb.pa_get_device_status() == 0
        assert torch.count_nonzero(_tickets(w, ws, split["workspace_bytes"])) == 0
        outs.append(out.clone())
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    assert_parity(outs[0], oracle_ref(w), "fused")
    # the same merge order as the separate reduce up to rounding
    ref = run(w, mode="split", partition_size=128)
    assert (outs[0].float() - ref.float()).abs().max().item() < 2e-3


def test_pooled_then_fused_on_one_caller_workspace(dev):
    # A pooled call arms its claim counters right after the partials; a fused
    # call of the same shape on the same workspace keeps its tickets in a slot
    # of its own, so neither disturbs the other, in either order.
    w = W.make_workload("poolfuse", [20000, 77, 9000], num_blocks=2000, seed=27, device=dev)
    kw = dict(mode="split", partition_size=512)
    pooled = _pooled_plan(w, **kw)
    fused = pb.pa_decode_plan(torch.empty_like(w.q), w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                              w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                              max_seq_len=w.max_seq_len, mode="fused", partition_size=512)
    assert pooled["pooled"] == 1 and fused["workspace_bytes"] > pooled["workspace_bytes"]
    ws = pb.alloc_workspace(fused, dev)
    ref = oracle_ref(w)
    for k in range(2):
        assert_parity(run(w, workspace=ws, flags=pb.PA_FLAG_POOLED, **kw), ref, f"pooled {k}")
        assert (_claims(ws[:pooled["workspace_bytes"]], pooled, w) == CLAIM_ARMED).all()
        out = run(w, workspace=ws, mode="fused", partition_size=512)
        assert_parity(out, ref, f"fused after pooled {k}")
        tickets = ws[fused["workspace_bytes"] - (len(w.seq_lens_host) * w.num_kv_heads * 8 + 255) // 256 * 256:]
        assert torch.count_nonzero(tickets) == 0


def test_fused_combine_after_forced_timeout_and_in_a_graph(dev):
    w = W.make_workload("fusedg", [4000, 100, 2500], num_blocks=500, seed=16, device=dev)
    out = torch.empty_like(w.q)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len,
                             mode="fused", partition_size=128)
    ws = pb.alloc_workspace(plan, dev)
    pb.pa_get_device_status()
    _fused_call(w, out, ws, flags=pb.PA_FLAG_FORCE_TIMEOUT)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() & pb.PA_DEV_TIMEOUT
    # the tickets stayed consistent: the next call on the same workspace is right
    _fused_call(w, out, ws)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    eager = out.clone()
    assert_parity(eager, oracle_ref(w), "fused after timeout")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _fused_call(w, out, ws, stream=torch.cuda.current_stream())
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert torch.equal(out, eager)


def test_persistent_schedule_empty_bad_and_graph(dev):
    # empty sequences are zero, single-partition ones are written directly, the rest merged
    w = W.make_workload("pers", [0, 700, 16, 5000, 0, 513, 1], num_blocks=500, seed=17, device=dev,
                        tail_fill=float("nan"))
    out = run(w, mode="persistent")
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[4]) == 0
    assert_parity(out, oracle_ref(w), "persistent ragged")
    assert torch.equal(out, run(w, mode="persistent"))  # repeat: bit-identical
    # a length beyond the host bound is reported, as in the grid schedule
    bad = W.make_workload("persbad", [100, 40], num_blocks=20, seed=18, device=dev, extra_table_cols=4)
    pb.pa_get_device_status()
    o2 = torch.empty_like(bad.q)
    bad.seq_lens[1] = 101
    pb.pa_decode_ex(o2, bad.q, bad.k_cache, bad.v_cache, bad.block_tables, bad.seq_lens, bad.num_heads,
                    bad.num_kv_heads, bad.head_dim, bad.block_size, bad.scale, max_seq_len=100, mode="persistent",
                    workspace=pb.alloc_workspace(pb.pa_decode_plan(
                        o2, bad.q, bad.k_cache, bad.v_cache, bad.block_tables, bad.seq_lens, bad.num_heads,
                        bad.num_kv_heads, bad.head_dim, bad.block_size, bad.scale, max_seq_len=100,
                        mode="persistent"), dev))
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() & pb.PA_DEV_BAD_SEQ_LEN
    # captured once, replayed with new lengths: the work list is rebuilt on the device
    kw = dict(max_seq_len=w.max_seq_len, mode="persistent")
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, **kw)
    ws = pb.alloc_workspace(plan, dev)
    args = (out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads, w.head_dim,
            w.block_size, w.scale)
    pb.pa_decode_ex(*args, workspace=ws, **kw)
    torch.cuda.synchronize()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pb.pa_decode_ex(*args, torch.cuda.current_stream(), workspace=ws, **kw)
    new_lens = [0, 690, 16, 4000, 0, 500, 1]  # within each sequence's blocks
    w.seq_lens.copy_(torch.tensor(new_lens, dtype=torch.int32, device=dev))
    w.seq_lens_host[:] = new_lens
    g.replay()
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), "persistent graph replay with new lengths")


@pytest.mark.parametrize("warps", [1, 2, 4])
@pytest.mark.parametrize("P", [16, 64, 512])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_persistent_many_items_per_cta(dev, warps, P, D):
    # small partitions give many more work items than resident CTAs, so each
    # CTA draws many items from the counter and its warps stream their blocks
    # across items and sequences through one ring each
    lens = [1, 17, 513, 3000, 100, 0, 2049, 16, 4000, 777] * 3
    w = W.make_workload("pmany", lens, num_blocks=2100, seed=40 + warps, device=dev, tail_fill=float("nan"),
                        head_dim=D, num_heads=24 if D == 256 else 16, num_kv_heads=4)
    out = run(w, mode="persistent", partition_size=P, warps=warps, stages=2)
    assert_parity(out, oracle_ref(w), f"persistent P={P} warps={warps} D={D}")
    assert torch.count_nonzero(out[5]) == 0
    # which CTA draws which item changes from call to call; the bits do not
    assert torch.equal(out, run(w, mode="persistent", partition_size=P, warps=warps, stages=2))


# ---- pooled split (PA_FLAG_POOLED): warps claim chunks of blocks from a counter ----

CLAIM_ARMED = 0x5A17C0DE << 32  # the value the reduce kernel leaves in every claim counter


def _claims(ws, plan, w):
    """The (sequence, kv head) claim counters at the end of the workspace."""
    n = w.block_tables.shape[0] * w.num_kv_heads
    tail = (n * 8 + 255) // 256 * 256
    return ws[plan["workspace_bytes"] - tail:].view(torch.int64)[:n]


def _pooled_plan(w, **opt):
    out = torch.empty_like(w.q)
    return pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len,
                             flags=pb.PA_FLAG_POOLED, **opt)


@pytest.mark.parametrize("lens,opt", [
    ([102400], dict()),                                              # the one-wave plan, 4 warps per CTA
    ([1, 15, 16, 17, 63, 64, 65, 1029, 4097], dict(mode="split", partition_size=256)),
    ([3000, 517, 8000, 1, 0], dict(mode="split", partition_size=512, warps=1, stages=3)),
    ([3000, 517, 8000, 1, 0], dict(mode="split", partition_size=512, warps=2, stages=2)),
    ([2048, 3, 700, 12000], dict(mode="split", partition_size=1024, warps=4, stages=2)),
    ([5000] * 6, dict(mode="split", partition_size=256, warps=1, stages=2)),
    ([1, 47, 48, 49, 700, 3001], dict(mode="split", partition_size=48, warps=1, stages=3)),
    ([129, 128, 127, 4000, 9999], dict(mode="split", partition_size=128, warps=4, stages=2)),
], ids=["b1_l102400", "ragged_P256", "P512_1x3", "P512_2x2", "P1024_4x2", "b6_P256_1x2", "P48_1x3", "P128_4x2"])
def test_pooled_split_parity(dev, lens, opt):
    w = W.make_workload("pooled", lens, num_blocks=sum((L + 15) // 16 for L in lens) + 11, seed=sum(lens) % 97,
                        device=dev, tail_fill=float("nan"), extra_table_cols=len(lens) % 3 * 5)
    plan = _pooled_plan(w, **opt)
    assert plan["pooled"] == 1
    ws = pb.alloc_workspace(plan, dev)  # zero: the first call deals the chunks round-robin
    ref = oracle_ref(w, THREADS)
    for k in range(3):
        out = run(w, workspace=ws, flags=pb.PA_FLAG_POOLED, **opt)
        assert_parity(out, ref, f"pooled call {k} lens={lens} {opt}")
        assert (_claims(ws, plan, w) == CLAIM_ARMED).all()
        assert torch.count_nonzero(out[[i for i, L in enumerate(lens) if L == 0]]) == 0


@pytest.mark.parametrize("name", ["b1_l102400", "b4_l32768_peaked", "b8_u8192"])
def test_pooled_named_workload_full(dev, name):
    w = W.make_config(name, device=dev)
    plan = _pooled_plan(w)
    ws = pb.alloc_workspace(plan, dev)
    ref = oracle_ref(w, THREADS)
    for k in range(2):
        out = run(w, workspace=ws, flags=pb.PA_FLAG_POOLED)
        print(name, "pooled" if k else "round-robin", assert_parity(out, ref, f"{name} pooled call {k}"))


def test_pooled_garbage_workspace_timeout_and_graph(dev):
    w = W.make_workload("poolg", [20000, 77, 9000], num_blocks=2000, seed=17, device=dev)
    opt = dict(mode="split", partition_size=512, flags=pb.PA_FLAG_POOLED)
    plan = _pooled_plan(w, mode="split", partition_size=512)
    ref = oracle_ref(w)
    # any bytes in a fresh workspace: the counters are not armed, the chunks go round-robin
    ws = torch.randint(0, 256, (plan["workspace_bytes"],), dtype=torch.uint8, device=dev)
    assert_parity(run(w, workspace=ws, **opt), ref, "pooled on a random workspace")
    assert (_claims(ws, plan, w) == CLAIM_ARMED).all()
    # a forced timeout is reported and leaves the counters armed for the next call
    pb.pa_get_device_status()
    pb.decode_workload(w, workspace=ws, mode="split", partition_size=512,
                       flags=pb.PA_FLAG_POOLED | pb.PA_FLAG_FORCE_TIMEOUT)
    assert pb.pa_get_device_status() & pb.PA_DEV_TIMEOUT
    assert (_claims(ws, plan, w) == CLAIM_ARMED).all()
    assert_parity(run(w, workspace=ws, **opt), ref, "pooled after a timeout")
    # captured once, replayed: each replay claims from the counter its predecessor re-armed
    out = torch.empty_like(w.q)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pb.decode_workload(w, out=out, stream=torch.cuda.current_stream(), workspace=ws, **opt)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert pb.pa_get_device_status() == 0
        assert_parity(out, ref, "pooled graph replay")


def test_one_wave_plan_pools_by_default_and_deterministic_flag_fixes_the_bits(dev):
    w = W.make_workload("onewave", [90000], num_blocks=90000 // 16 + 5, seed=23, device=dev)
    assert _pooled_plan(w)["pooled"] == 1
    ref = oracle_ref(w, THREADS)
    fixed = [run(w, flags=pb.PA_FLAG_DETERMINISTIC) for _ in range(3)]
    assert all(torch.equal(fixed[0], f) for f in fixed[1:])
    assert_parity(fixed[0], ref, "one wave, deterministic")
    ws = pb.alloc_workspace(_pooled_plan(w), dev)
    for k in range(3):  # round-robin first, then claimed chunks
        out = run(w, workspace=ws, mode="auto")
        assert_parity(out, ref, f"one wave, pooled call {k}")
        assert (out.float() - fixed[0].float()).abs().max().item() < 2e-3


def test_pooled_bad_block_id_and_bad_length(dev):
    # the kernel's own checks in the pooled form: an illegal block id is
    # reported and skipped, an illegal length reported, and the claim
    # counters stay armed for the next call
    w = W.make_workload("poolbad", [5000, 3000], num_blocks=600, seed=19, device=dev)
    opt = dict(mode="split", partition_size=512, flags=pb.PA_FLAG_POOLED)
    plan = _pooled_plan(w, mode="split", partition_size=512)
    ws = pb.alloc_workspace(plan, dev)
    ref = oracle_ref(w)
    assert_parity(run(w, workspace=ws, **opt), ref, "pooled before")
    good = w.block_tables.clone()
    pb.pa_get_device_status()
    w.block_tables[0, 37] = w.num_blocks + 3
    w.block_tables[1, 5] = -5
    pb.decode_workload(w, workspace=ws, **opt)
    assert pb.pa_get_device_status() & pb.PA_DEV_BAD_BLOCK_ID
    assert (_claims(ws, plan, w) == CLAIM_ARMED).all()
    w.block_tables.copy_(good)
    w.seq_lens[1] = 5001  # above the max_seq_len hint
    pb.decode_workload(w, workspace=ws, **opt)
    assert pb.pa_get_device_status() & pb.PA_DEV_BAD_SEQ_LEN
    w.seq_lens[1] = 3000
    assert_parity(run(w, workspace=ws, **opt), ref, "pooled after the errors")


# ---- flat one-wave split (PA_MODE_FLAT): every CTA streams an equal share of the batch's blocks ----

@pytest.mark.parametrize("warps,stages", [(1, 2), (2, 2), (4, 2)])
def test_flat_split_shapes_ragged_empty_and_bad(dev, warps, stages):
    lens = [0, 1, 15, 16, 17, 511, 512, 513, 0, 3000, 7000, 2, 100]
    w = W.make_workload("flat", lens, num_blocks=900, seed=50 + warps, device=dev, tail_fill=float("nan"))
    out = run(w, mode="flat", warps=warps, stages=stages)
    assert torch.count_nonzero(out[0]) == 0 and torch.count_nonzero(out[8]) == 0
    assert_parity(out, oracle_ref(w), f"flat {warps}x{stages}")
    assert torch.equal(out, run(w, mode="flat", warps=warps, stages=stages))  # fixed shares: same bits
    # a length beyond the host bound is reported and the rest is still right
    bad = W.make_workload("flatbad", [100, 40, 700], num_blocks=60, seed=51, device=dev, extra_table_cols=4)
    pb.pa_get_device_status()
    o2 = torch.empty_like(bad.q)
    bad.seq_lens[1] = 101
    kw = dict(max_seq_len=100, mode="flat", warps=warps, stages=stages)
    args = (o2, bad.q, bad.k_cache, bad.v_cache, bad.block_tables, bad.seq_lens, bad.num_heads, bad.num_kv_heads,
            bad.head_dim, bad.block_size, bad.scale)
    pb.pa_decode_ex(*args, workspace=pb.alloc_workspace(pb.pa_decode_plan(*args, **kw), dev), **kw)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() & pb.PA_DEV_BAD_SEQ_LEN


def test_flat_split_many_short_sequences_and_graph_replay(dev):
    # more sequences than CTAs of a kv head, most shorter than a CTA's share;
    # then one capture replayed with new lengths (the host never reads them)
    lens = [1 + (37 * i) % 900 for i in range(200)]
    w = W.make_workload("flatmany", lens, num_blocks=sum((L + 15) // 16 for L in lens) + 3, seed=52, device=dev,
                        tail_fill=float("nan"))
    out = run(w, mode="flat")
    assert_parity(out, oracle_ref(w), "flat, 200 sequences")
    kw = dict(max_seq_len=w.max_seq_len, mode="flat")
    args = (out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads, w.head_dim,
            w.block_size, w.scale)
    ws = pb.alloc_workspace(pb.pa_decode_plan(*args, **kw), dev)
    pb.pa_decode_ex(*args, workspace=ws, **kw)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pb.pa_decode_ex(*args, torch.cuda.current_stream(), workspace=ws, **kw)
    new = [max(0, L - (i % 7) * 3) for i, L in enumerate(lens)]  # within each sequence's blocks, some empty
    w.seq_lens.copy_(torch.tensor(new, dtype=torch.int32, device=dev))
    w.seq_lens_host[:] = new
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), "flat graph replay with new lengths")



# ---- fused combine on a co-resident grid: a group barrier, then every CTA merges its slice ----

@pytest.mark.parametrize("lens,opt,pooled", [
    ([102400], dict(), True),                                        # the one-wave plan, pooled
    ([102400], dict(flags=pb.PA_FLAG_DETERMINISTIC), False),
    ([2048], dict(partition_size=256), False),
    ([3000, 17, 1029, 513, 128, 1, 0], dict(partition_size=128, warps=1, stages=2), False),
    ([5000, 700, 64], dict(partition_size=512, warps=2, stages=2), False),
    ([7000, 4000], dict(partition_size=1024, warps=4, stages=2), False),
], ids=["one_wave_pooled", "one_wave_fixed", "b1_l2048_P256", "ragged_P128", "P512_2x2", "P1024_4x2"])
def test_fused_parallel_merge(dev, lens, opt, pooled):
    w = W.make_workload("coop", lens, num_blocks=sum((L + 15) // 16 for L in lens) + 9, seed=60 + len(lens),
                        device=dev, tail_fill=float("nan"))
    out = torch.empty_like(w.q)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len,
                             mode="fused", **opt)
    assert plan["coop"] == 1 and plan["launch_reduce"] == 0 and plan["pooled"] == int(pooled)
    ws = pb.alloc_workspace(plan, dev)
    ref = oracle_ref(w, THREADS)
    outs = []
    for k in range(3):  # the group words are left zero, the pooled counters re-armed
        outs.append(run(w, workspace=ws, mode="fused", **opt))
        assert_parity(outs[-1], ref, f"fused parallel merge, call {k}")
        assert torch.count_nonzero(_tickets(w, ws, _split_bytes(w, plan))) == 0
        if pooled:
            assert (_claims_at(ws, _split_bytes(w, plan), w) == CLAIM_ARMED).all()
    if not pooled:
        assert all(torch.equal(outs[0], o) for o in outs[1:])
    # the same merge as the reduce kernel up to rounding
    split = run(w, mode="split", **{k: v for k, v in opt.items() if k != "flags"})
    assert (outs[0].float() - split.float()).abs().max().item() < 2e-3
    # captured and replayed
    g = torch.cuda.CUDAGraph()
    res = torch.empty_like(w.q)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        pb.decode_workload(w, out=res, stream=torch.cuda.current_stream(), workspace=ws, mode="fused", **opt)
    for _ in range(3):
        res.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert pb.pa_get_device_status() == 0
        assert_parity(res, ref, "fused parallel merge, graph replay")


def test_fused_parallel_merge_after_forced_timeout(dev):
    w = W.make_workload("coopto", [20000, 3000], num_blocks=1500, seed=61, device=dev)
    kw = dict(mode="fused", partition_size=512)
    out = torch.empty_like(w.q)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len, **kw)
    assert plan["coop"] == 1
    ws = pb.alloc_workspace(plan, dev)
    pb.pa_get_device_status()
    pb.decode_workload(w, workspace=ws, flags=pb.PA_FLAG_FORCE_TIMEOUT, **kw)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() & pb.PA_DEV_TIMEOUT
    assert torch.count_nonzero(_tickets(w, ws, _split_bytes(w, plan))) == 0  # every group left them zero
    assert_parity(run(w, workspace=ws, **kw), oracle_ref(w), "fused after a forced timeout")


def _split_bytes(w, plan):
    """Bytes of the partials in a fused plan's workspace (before the claim and ticket slots)."""
    n = len(w.seq_lens_host) * w.num_kv_heads
    return plan["workspace_bytes"] - (n * 8 + 255) // 256 * 256 - (n * 8 + 255) // 256 * 256


def _claims_at(ws, split_bytes, w):
    n = len(w.seq_lens_host) * w.num_kv_heads
    return ws[split_bytes:split_bytes + 8 * n].view(torch.int64)


@pytest.mark.parametrize("lens", [[4000] * 4, [4000, 100, 3000, 0], [1, 17, 4000], [2048] * 8])
def test_uniform_lengths_flag(dev, lens):
    # the batch's one-wave plan (PA_FLAG_UNIFORM_LENGTHS) on uniform batches and,
    # where the statement is wrong, on ragged ones: correct either way
    w = W.make_workload("uniform", lens, num_blocks=sum((L + 15) // 16 for L in lens) + 5, seed=len(lens) + lens[0],
                        device=dev, tail_fill=float("nan"))
    flags = pb.PA_FLAG_UNIFORM_LENGTHS
    plan = pb.pa_decode_plan(torch.empty_like(w.q), w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                             w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                             max_seq_len=w.max_seq_len, flags=flags)
    assert plan["threads"] == 128 and plan["grid_x"] * plan["grid_y"] * plan["grid_z"] <= 152
    out = pb.decode_workload(w, flags=flags)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), f"uniform-lengths plan {lens}")
    assert all(torch.count_nonzero(out[b]) == 0 for b, L in enumerate(lens) if L == 0)
    # fixed partitions: repeats give the same bits
    again = pb.decode_workload(w, flags=flags)
    torch.cuda.synchronize()
    assert torch.equal(out, again)


def test_uniform_lengths_flag_on_the_peaked_workload(dev):
    w = W.make_config("b4_l32768_peaked", device=dev)
    out = pb.decode_workload(w, flags=pb.PA_FLAG_UNIFORM_LENGTHS)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), "b4_l32768_peaked, uniform-lengths plan")


@pytest.mark.parametrize("H,Hkv,D,L,pooled", [(32, 8, 128, 102400, 1), (32, 4, 64, 131072, 0), (64, 8, 128, 50000, 0)])
def test_one_wave_at_smaller_head_dims(dev, H, Hkv, D, L, pooled):
    # the one-wave plan runs 256 / head_dim CTAs per SM (2 at 128, 4 at 64);
    # at 32/8 heads and 102400 tokens its 2704-token partitions are pooled
    w = W.make_workload("hd", [L], num_heads=H, num_kv_heads=Hkv, head_dim=D, num_blocks=(L + 15) // 16 + 4,
                        seed=H + D, device=dev, scale=D ** -0.5, tail_fill=float("nan"))
    plan = pb.pa_decode_plan(torch.empty_like(w.q), w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                             w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                             max_seq_len=w.max_seq_len)
    assert plan["grid_x"] * plan["grid_y"] == 152 * (256 // D) and plan["pooled"] == pooled
    out = pb.decode_workload(w)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), f"one wave, H={H} Hkv={Hkv} D={D} L={L}")


@pytest.mark.parametrize("lens,flags", [([2048, 700, 1500], 0), ([4000] * 4, pb.PA_FLAG_UNIFORM_LENGTHS),
                                        ([3000], 0), ([90000], 0)])
def test_one_wave_plans_replay_from_a_graph_with_new_lengths(dev, lens, flags):
    # the host never reads the lengths: a captured one-wave call (short batch,
    # uniform-lengths batch, short and long single sequences) replays with
    # other lengths under the same bound and matches the oracle
    w = W.make_workload("owgraph", lens, num_blocks=sum((L + 15) // 16 for L in lens) + 5, seed=len(lens) + lens[0],
                        device=dev, tail_fill=float("nan"))
    out = torch.full_like(w.q, float("nan"))
    kw = dict(max_seq_len=w.max_seq_len, flags=flags)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, **kw)
    assert plan["threads"] == 128 and plan["launch_reduce"] == 1
    ws = pb.alloc_workspace(plan, dev)
    args = (out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads, w.head_dim,
            w.block_size, w.scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pb.pa_decode_ex(*args, s, workspace=ws, **kw)  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pb.pa_decode_ex(*args, torch.cuda.current_stream(), workspace=ws, **kw)
    for new in ([L // 3 for L in lens], [max(0, L - 17) for L in lens], lens):
        w.seq_lens.copy_(torch.tensor(new, dtype=torch.int32, device=dev))
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pb.pa_get_device_status() == 0
        assert_parity(out, oracle_ref(w), f"graph replay, lengths {new}")
