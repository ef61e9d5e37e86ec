"""Numerically adversarial decode inputs on the GPU, every mode, against the
float64 oracle (and closed forms where one exists).

- scale 0: every score is 0, so the output is the mean of the sequence's V
  rows (a closed form, independent of the oracle);
- a negative scale, and a large one that makes the softmax nearly one-hot;
- fp16 inputs of large magnitude (q and K ~ N(0, 12^2)), whose scaled scores
  spread over hundreds (e^s would overflow fp32 without the running max);
  the magnitudes stay where fp32 accumulation of the dot products is exact
  enough for the tolerance (a few 1e-4 of score error);
- tied keys: every key of a sequence equal, so the weights are uniform;
- a batch of 1024 short sequences (more sequences than any grid dimension of
  one wave).
"""
import numpy as np
import pytest
import torch

from paged_kv_cache_308_gb300 import binding as pb
from paged_kv_cache_308_gb300 import workloads as W
from parity_helpers import ATOL, RTOL, assert_parity, compare, oracle_ref

pytestmark = pytest.mark.gpu

MODES = [dict(), dict(mode="single"), dict(mode="split", partition_size=64), dict(mode="fused", partition_size=128),
         dict(mode="persistent"), dict(mode="flat")]
IDS = ["auto", "single", "split64", "fused128", "persistent", "flat"]
LENS = [1, 17, 300, 1029, 4000, 0]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _run(w, **opt):
    out = pb.decode_workload(w, **opt)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    return out


def _with_scale(w, scale):
    return W.Workload(w.name, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.seq_lens_host, w.num_heads,
                      w.num_kv_heads, w.head_dim, w.block_size, scale, w.partition_size)


@pytest.mark.parametrize("opt", MODES, ids=IDS)
def test_zero_scale_gives_the_mean_of_v(dev, opt):
    w = _with_scale(W.make_workload("zero", LENS, num_blocks=420, seed=70, device=dev, tail_fill=float("nan")), 0.0)
    out = _run(w, **opt)
    G = w.num_heads // w.num_kv_heads
    for b, L in enumerate(LENS):
        if L == 0:
            assert torch.count_nonzero(out[b]) == 0
            continue
        nblk = (L + 15) // 16
        rows = w.v_cache[w.block_tables[b, :nblk].long()].float()        # [nblk, Hkv, 16, D]
        rows = rows.permute(1, 0, 2, 3).reshape(w.num_kv_heads, nblk * 16, w.head_dim)[:, :L]
        mean = rows.double().mean(dim=1).repeat_interleave(G, dim=0)    # [H, D]
        err = (out[b].double() - mean).abs()
        assert bool((err <= ATOL + RTOL * mean.abs()).all()), f"{opt} seq {b}: {err.max().item()}"


@pytest.mark.parametrize("scale", [-1 / 16, 0.75, 4.0])
@pytest.mark.parametrize("opt", MODES, ids=IDS)
def test_negative_and_large_scales(dev, scale, opt):
    w = _with_scale(W.make_workload("scale", LENS, num_blocks=420, seed=71, device=dev, tail_fill=float("nan")),
                    scale)
    assert_parity(_run(w, **opt), oracle_ref(w), f"scale {scale} {opt}")


@pytest.mark.parametrize("opt", MODES, ids=IDS)
def test_large_magnitude_inputs(dev, opt):
    # q, K ~ N(0, 12^2): scaled scores with a standard deviation near 144
    w = W.make_workload("big", LENS, num_blocks=420, seed=72, device=dev, tail_fill=float("inf"))
    g = torch.Generator(device=dev).manual_seed(73)
    w.q.copy_((torch.randn(w.q.shape, generator=g, device=dev) * 12).half())
    k = torch.randn(w.k_cache.shape, generator=g, device=dev) * 12
    keep_tail = ~torch.isfinite(w.k_cache)
    w.k_cache.copy_(torch.where(keep_tail, w.k_cache.float(), k).half())
    out = _run(w, **opt)
    assert torch.isfinite(out).all()
    ref = oracle_ref(w)
    r = compare(out, ref)
    # near one-hot softmax: the output is close to single V rows, and the
    # element-wise bound applies as everywhere
    assert r["ok"], f"{opt}: {r}"


@pytest.mark.parametrize("opt", MODES, ids=IDS)
def test_tied_keys_give_uniform_weights(dev, opt):
    w = W.make_workload("tied", LENS, num_blocks=420, seed=74, device=dev, tail_fill=float("nan"))
    finite = torch.isfinite(w.k_cache)
    row = torch.linspace(-1, 1, w.head_dim, device=dev).half()
    w.k_cache.copy_(torch.where(finite, row.expand_as(w.k_cache), w.k_cache))
    out = _run(w, **opt)
    assert_parity(out, oracle_ref(w), f"tied {opt}")
    # with every key equal the weights are uniform: the output is the mean of V
    zero = _run(_with_scale(w, 0.0), **opt)
    assert (out.float() - zero.float()).abs().max().item() < 2e-3


@pytest.mark.parametrize("opt", [dict(), dict(mode="split", partition_size=32), dict(mode="persistent")],
                         ids=["auto", "split32", "persistent"])
def test_a_thousand_short_sequences(dev, opt):
    rng = np.random.default_rng(75)
    lens = rng.integers(0, 65, 1024).tolist()
    w = W.make_workload("many", lens, num_blocks=sum((L + 15) // 16 for L in lens) + 5, seed=75, device=dev,
                        tail_fill=float("nan"))
    out = _run(w, **opt)
    assert_parity(out, oracle_ref(w), f"1024 sequences {opt}")
    assert all(torch.count_nonzero(out[b]) == 0 for b, L in enumerate(lens) if L == 0)
