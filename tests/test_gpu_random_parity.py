"""Seeded random sweep of decode shapes on the GPU against the float64 oracle.

Each case draws a batch size, ragged lengths (including 0 and 1 and
lengths that end inside a block), a GQA ratio, a head_dim and a call mode,
runs the CUDA path through the C ABI and compares every output element with
the oracle.  The draws come from a fixed seed, so a failure names a case that
reproduces.
"""
import random

import pytest
import torch

from paged_kv_cache_308_gb300 import binding as pb
from paged_kv_cache_308_gb300 import split_kv
from paged_kv_cache_308_gb300 import workloads as W
from parity_helpers import assert_parity, oracle_ref

pytestmark = pytest.mark.gpu

MODES = [dict(), dict(mode="single"), dict(mode="split"), dict(mode="fused"), dict(mode="persistent"),
         dict(mode="split", partition_size=32), dict(mode="fused", partition_size=64),
         dict(mode="persistent", partition_size=48), dict(mode="persistent", warps=2, stages=2),
         dict(mode="flat"), dict(mode="flat", warps=1, stages=2), dict(mode="flat", warps=2, stages=2)]


def draw_case(i):
    r = random.Random(1000 + i)
    hkv = r.choice([1, 2, 4, 8])
    g = r.choice([1, 2, 3, 4, 6, 8])
    d = r.choice([64, 128, 256])
    b = r.choice([1, 2, 3, 5, 8, 13])
    longest = r.choice([16, 100, 700, 3000])
    lens = [r.choice([0, 1, 15, 16, 17, r.randint(1, longest), longest]) for _ in range(b)]
    return dict(lens=lens, num_heads=hkv * g, num_kv_heads=hkv, head_dim=d, opt=MODES[i % len(MODES)], seed=i)


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


@pytest.mark.parametrize("i", range(48))
def test_random_case(dev, i):
    c = draw_case(i)
    blocks = sum((L + 15) // 16 for L in c["lens"]) + 3
    w = W.make_workload(f"rand{i}", c["lens"], num_heads=c["num_heads"], num_kv_heads=c["num_kv_heads"],
                        head_dim=c["head_dim"], num_blocks=blocks, seed=c["seed"], device=dev,
                        tail_fill=float("nan"))
    out = pb.decode_workload(w, **c["opt"])
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), f"case {i}: {c}")
    for b, L in enumerate(c["lens"]):
        if L == 0:
            assert torch.count_nonzero(out[b]) == 0, f"case {i}: empty sequence {b} not zero"


POOL_SHAPES = [(1, 2), (1, 3), (2, 2), (4, 2)]


@pytest.mark.parametrize("i", range(12))
def test_random_pooled_case(dev, i):
    # the pooled split on random shapes: the first call on a fresh workspace
    # deals the chunks round-robin, the later ones claim them from the counter
    c = draw_case(100 + i)
    warps, stages = POOL_SHAPES[i % len(POOL_SHAPES)]
    part = warps * 16 * max(2, stages) * random.Random(i).choice([1, 2, 3])
    opt = dict(mode="split", partition_size=part, warps=warps, stages=stages, flags=pb.PA_FLAG_POOLED)
    blocks = sum((L + 15) // 16 for L in c["lens"]) + 3
    w = W.make_workload(f"randpool{i}", c["lens"], num_heads=c["num_heads"], num_kv_heads=c["num_kv_heads"],
                        head_dim=c["head_dim"], num_blocks=blocks, seed=c["seed"], device=dev,
                        tail_fill=float("nan"))
    out = torch.empty_like(w.q)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len, **opt)
    ws = pb.alloc_workspace(plan, dev)
    ref = oracle_ref(w)
    for k in range(2):
        out = pb.decode_workload(w, workspace=ws, **opt)
        torch.cuda.synchronize()
        assert pb.pa_get_device_status() == 0
        assert_parity(out, ref, f"pooled case {i} call {k}: {c} {opt} pooled={plan['pooled']}")
        for b, L in enumerate(c["lens"]):
            if L == 0:
                assert torch.count_nonzero(out[b]) == 0, f"pooled case {i}: empty sequence {b} not zero"


@pytest.mark.parametrize("i", range(12))
def test_random_split_kv_case(dev, i):
    # the partitions spread over R sources (one pa_decode_partials call each,
    # into its slot of the gathered buffer), then pa_merge_partials
    c = draw_case(200 + i)
    r = random.Random(300 + i)
    P = 16 * r.choice([1, 2, 5, 16, 32, 64])
    R = r.choice([1, 2, 3, 4])
    blocks = sum((L + 15) // 16 for L in c["lens"]) + 3
    w = W.make_workload(f"randskv{i}", c["lens"], num_heads=c["num_heads"], num_kv_heads=c["num_kv_heads"],
                        head_dim=c["head_dim"], num_blocks=blocks, seed=c["seed"], device=dev,
                        tail_fill=float("nan"))
    ranges = [split_kv.partition_range(k, R, w.max_seq_len, P) for k in range(R)]
    count = ranges[0][1]
    gm, gl, gacc = split_kv.alloc_partials(w.num_seqs, w.num_heads, w.head_dim, count, dev, sources=R)
    for k, (begin, n) in enumerate(ranges):
        pb.pa_decode_partials(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                              w.head_dim, w.block_size, w.scale, P, begin, n, gm[k], gl[k], gacc[k],
                              max_seq_len=w.max_seq_len)
    out = torch.full_like(w.q, float("nan"))
    pb.pa_merge_partials(out, gm, gl, gacc, w.seq_lens, w.num_heads, w.head_dim, P, R, count,
                         max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), f"split-KV case {i}: {c} P={P} R={R}")


def draw_short_case(i):
    # AUTO's short one-wave plans: longest sequence 513..4864 tokens, small
    # batches (partitions of at most 128 tokens, one copy round per CTA);
    # every other case states uniform lengths, right or wrong
    r = random.Random(5000 + i)
    hkv = r.choice([1, 2, 4, 8])
    g = r.choice([1, 2, 4, 6, 8])
    d = r.choice([64, 128, 256])
    b = r.choice([1, 1, 2, 3, 4])
    longest = r.randint(513, 4864)
    lens = [longest] + [r.choice([0, 1, 17, r.randint(1, longest), longest]) for _ in range(b - 1)]
    r.shuffle(lens)
    opt = dict(flags=pb.PA_FLAG_UNIFORM_LENGTHS) if i % 2 else dict()
    return dict(lens=lens, num_heads=hkv * g, num_kv_heads=hkv, head_dim=d, opt=opt, seed=500 + i)


@pytest.mark.parametrize("i", range(16))
def test_random_short_auto_case(dev, i):
    c = draw_short_case(i)
    blocks = sum((L + 15) // 16 for L in c["lens"]) + 3
    w = W.make_workload(f"short{i}", c["lens"], num_heads=c["num_heads"], num_kv_heads=c["num_kv_heads"],
                        head_dim=c["head_dim"], num_blocks=blocks, seed=c["seed"], device=dev,
                        tail_fill=float("nan"))
    out = pb.decode_workload(w, **c["opt"])
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), f"short case {i}: {c}")
    assert all(torch.count_nonzero(out[b]) == 0 for b, L in enumerate(c["lens"]) if L == 0)


def draw_large_case(i):
    # AUTO at realistic sizes: one-wave plans at 1, 2 or 4 CTAs per SM
    # (head_dim 256, 128, 64), pooled and fixed, and the grid for batches
    r = random.Random(9000 + i)
    hkv = r.choice([1, 2, 4, 8])
    g = r.choice([1, 4, 6, 8])
    d = r.choice([64, 128, 256])
    b = r.choice([1, 1, 2, 4, 16, 48])
    cap = max(16, (400_000_000 // (4 * hkv * d)) // b)  # about 400 MB of K/V at most
    lens = [min(cap, int(round(2 ** r.uniform(10, 17)))) for _ in range(b)]
    return dict(lens=lens, num_heads=hkv * g, num_kv_heads=hkv, head_dim=d, seed=900 + i)


@pytest.mark.parametrize("i", range(10))
def test_random_large_auto_case(dev, i):
    c = draw_large_case(i)
    blocks = sum((L + 15) // 16 for L in c["lens"]) + 3
    w = W.make_workload(f"large{i}", c["lens"], num_heads=c["num_heads"], num_kv_heads=c["num_kv_heads"],
                        head_dim=c["head_dim"], num_blocks=blocks, seed=c["seed"], device=dev,
                        scale=c["head_dim"] ** -0.5, tail_fill=float("nan"))
    out = pb.decode_workload(w)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), f"large case {i}: B={len(c['lens'])} max={max(c['lens'])} "
                                      f"H={c['num_heads']}/{c['num_kv_heads']} D={c['head_dim']}")


@pytest.mark.parametrize("B,L,H,Hkv,D", [(64, 4096, 24, 4, 256), (16, 16384, 32, 8, 128)])
def test_many_short_pairs_run_2x2_ctas(dev, B, L, H, Hkv, D):
    # at least 64 (sequence, kv head) pairs of at most 16K tokens: AUTO picks
    # 2x2 CTAs over 512-token partitions; ragged lengths, NaN past each end
    g = torch.Generator().manual_seed(B * L + D)
    lens = torch.randint(1, L + 1, (B,), generator=g).tolist()
    w = W.make_workload(f"pairs_{B}x{L}", lens, num_heads=H, num_kv_heads=Hkv, head_dim=D,
                        num_blocks=sum((x + 15) // 16 for x in lens) + 3, seed=B + D, device=dev,
                        scale=D ** -0.5, tail_fill=float("nan"))
    out = torch.empty_like(w.q)
    plan = pb.pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                             w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len)
    assert (plan["mode"], plan["partition_size"], plan["threads"] // 32, plan["stages"]) == (pb.PA_MODE_SPLIT, 512, 2, 2)
    out = pb.decode_workload(w)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert_parity(out, oracle_ref(w), f"{B} x U[1, {L}] H={H}/{Hkv} D={D}")
