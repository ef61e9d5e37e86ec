"""Split-KV across devices, kernel side, on one GPU through the C ABI.

pa_decode_partials computes the partials of a range of partitions;
pa_merge_partials merges partials gathered from several sources.  Here the
"devices" are separate calls on one GPU writing the slots of one gathered
buffer, as an all-gather would lay them out.  Checked against the float64
oracle: the per-partition partials against its partition pass, the merged
output against its definition; and bit for bit against the single-device split
call, which computes the same partials and folds them in the same order.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_308_gb300 import binding as pb
from paged_kv_cache_308_gb300 import split_kv
from paged_kv_cache_308_gb300 import workloads as W
from parity_helpers import ATOL, RTOL, assert_parity, host_bits, oracle_ref

pytestmark = pytest.mark.gpu
LN2 = math.log(2.0)


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda:0")


def _partials_into(w, P, begin, count, m, l, acc, **opt):
    pb.pa_decode_partials(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                          w.head_dim, w.block_size, w.scale, P, begin, count, m, l, acc,
                          max_seq_len=w.max_seq_len, **opt)


def _gathered(w, P, R, **opt):
    """Every source's partials in one [R, ...] buffer, one call per source."""
    ranges = [split_kv.partition_range(r, R, w.max_seq_len, P) for r in range(R)]
    count = ranges[0][1]
    gm, gl, gacc = split_kv.alloc_partials(w.num_seqs, w.num_heads, w.head_dim, count, w.q.device, sources=R)
    for r, (begin, c) in enumerate(ranges):
        _partials_into(w, P, begin, c, gm[r], gl[r], gacc[r], **opt)
    return gm, gl, gacc, count


def _merge(w, gm, gl, gacc, P, R, count):
    out = torch.full_like(w.q, float("nan"))
    pb.pa_merge_partials(out, gm, gl, gacc, w.seq_lens, w.num_heads, w.head_dim, P, R, count,
                         max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    return out


@pytest.mark.parametrize("begin,count", [(0, 12), (2, 3), (5, 9)])
def test_partials_match_the_oracle_partition_pass(dev, begin, count):
    lens = [1, 17, 700, 1500, 0, 2900]
    w = W.make_workload("partials", lens, num_blocks=400, seed=31, device=dev, tail_fill=float("nan"))
    P = 256
    m, l, acc = split_kv.alloc_partials(w.num_seqs, w.num_heads, w.head_dim, count, dev)
    _partials_into(w, P, begin, count, m, l, acc)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    m, l, acc = m.cpu().numpy(), l.cpu().numpy(), acc.cpu().numpy()
    args = (host_bits(w.q), host_bits(w.k_cache), host_bits(w.v_cache), host_bits(w.block_tables),
            host_bits(w.seq_lens), w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale)
    for b, L in enumerate(lens):
        for h in range(w.num_heads):
            om, ol, oacc = oracle.partition_partials(*args, b, h, P, 16)
            for j in range(count):
                p = begin + j
                if p < len(om):
                    # base-2 max on the GPU, natural on the oracle
                    assert abs(m[b, h, j] * LN2 - om[p]) <= 1e-3 + 1e-5 * abs(om[p]), (b, h, p)
                    assert abs(l[b, h, j] - ol[p]) <= 2e-3 * ol[p], (b, h, p)
                    err = np.abs(acc[b, h, j] - oacc[p])
                    assert np.all(err <= ATOL + RTOL * np.abs(oacc[p])), (b, h, p, err.max())
                else:  # past the sequence's end: the empty partial
                    assert m[b, h, j] == -np.inf and l[b, h, j] == 0 and not acc[b, h, j].any(), (b, h, p)


def test_two_ranges_of_the_100k_sequence_merge_to_the_oracle(dev):
    w = W.make_config("b1_l102400", device=dev)
    P, R = 512, 2
    shape = dict(warps=1, stages=2)
    gm, gl, gacc, count = _gathered(w, P, R, **shape)
    assert count == 100
    out = _merge(w, gm, gl, gacc, P, R, count)
    r = assert_parity(out, oracle_ref(w, 0), "two ranges merged")
    print("b1_l102400 split over 2 sources:", r)
    # the same partials and the same fold order as the one-device split call
    one = pb.decode_workload(w, mode="split", partition_size=P, flags=pb.PA_FLAG_DETERMINISTIC, **shape)
    torch.cuda.synchronize()
    assert torch.equal(out, one)


def test_a_range_never_reads_the_block_table_outside_it(dev):
    # a device holds only its own range of blocks: entries of other ranges
    # are never followed (no bad-block report, same partials)
    w = W.make_workload("range", [4000, 2500], num_blocks=500, seed=32, device=dev)
    P, begin, count = 512, 2, 3
    m0, l0, a0 = split_kv.alloc_partials(w.num_seqs, w.num_heads, w.head_dim, count, dev)
    _partials_into(w, P, begin, count, m0, l0, a0)
    torch.cuda.synchronize()
    pb.pa_get_device_status()
    lo, hi = begin * P // 16, (begin + count) * P // 16
    w.block_tables[:, :lo] = -7
    w.block_tables[:, hi:] = w.num_blocks + 9
    m1, l1, a1 = split_kv.alloc_partials(w.num_seqs, w.num_heads, w.head_dim, count, dev)
    _partials_into(w, P, begin, count, m1, l1, a1)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert torch.equal(m0, m1) and torch.equal(l0, l1) and torch.equal(a0, a1)


@pytest.mark.parametrize("R", [1, 3, 4])
@pytest.mark.parametrize("shape", [dict(), dict(warps=2, stages=2), dict(warps=4, stages=2)])
def test_ragged_batch_over_several_sources(dev, R, shape):
    lens = [0, 1, 16, 17, 511, 513, 3000, 8000]
    w = W.make_workload("ragged", lens, num_blocks=1000, seed=33 + R, device=dev, tail_fill=float("nan"))
    P = 512
    gm, gl, gacc, count = _gathered(w, P, R, **shape)
    out = _merge(w, gm, gl, gacc, P, R, count)
    assert torch.count_nonzero(out[0]) == 0
    assert_parity(out, oracle_ref(w), f"ragged batch over {R} sources")
    if shape:  # same CTA shape: bit-identical to the one-device split where it merges
        one = pb.decode_workload(w, mode="split", partition_size=P, **shape)
        torch.cuda.synchronize()
        multi = [b for b, L in enumerate(lens) if L > P]
        assert torch.equal(out[multi], one[multi])


def test_merge_of_the_mixed_batch(dev):
    w = W.make_config("b64_loguniform", device=dev)
    P, R = 1024, 2
    gm, gl, gacc, count = _gathered(w, P, R)
    out = _merge(w, gm, gl, gacc, P, R, count)
    one = pb.decode_workload(w)
    torch.cuda.synchronize()
    assert (out.float() - one.float()).abs().max().item() < 2e-3


def test_argument_errors(dev):
    w = W.make_workload("args", [3000], num_blocks=200, seed=34, device=dev)
    m, l, acc = split_kv.alloc_partials(1, w.num_heads, w.head_dim, 4, dev)
    for P, begin, count in ((500, 0, 4), (512, -1, 4), (512, 0, 0)):
        with pytest.raises(pb.PaDecodeError) as e:
            _partials_into(w, P, begin, count, m, l, acc)
        assert e.value.code == pb.PA_ERR_INVALID_ARG
    with pytest.raises(pb.PaDecodeError) as e:
        _partials_into(w, 512, 0, 4, m, l, acc, mode="fused")
    assert e.value.code == pb.PA_ERR_INVALID_ARG
    gm, gl, gacc = split_kv.alloc_partials(1, w.num_heads, w.head_dim, 2, dev, sources=2)
    out = torch.empty_like(w.q)
    # 2 sources x 2 partitions of 512 tokens do not cover 3000 tokens
    with pytest.raises(pb.PaDecodeError) as e:
        pb.pa_merge_partials(out, gm, gl, gacc, w.seq_lens, w.num_heads, w.head_dim, 512, 2, 2, max_seq_len=3000)
    assert e.value.code == pb.PA_ERR_INVALID_ARG
    # a length above the host bound is reported by the merge too
    gm, gl, gacc, count = _gathered(w, 512, 2)
    pb.pa_get_device_status()
    w.seq_lens[0] = 3001
    pb.pa_merge_partials(out, gm, gl, gacc, w.seq_lens, w.num_heads, w.head_dim, 512, 2, count, max_seq_len=3000)
    assert pb.pa_get_device_status() & pb.PA_DEV_BAD_SEQ_LEN


def _free_port():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_split_kv_decode_through_nccl(dev):
    # the whole host path -- ranges, partials, an NCCL all-gather of the local
    # buffers, the merge -- in a process group of one rank on this GPU
    import os
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=dev)
    try:
        w = W.make_workload("nccl", [5000, 0, 17, 12000], num_blocks=1200, seed=35, device=dev,
                            tail_fill=float("nan"))
        out = torch.full_like(w.q, float("nan"))
        split_kv.split_kv_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                                 w.num_kv_heads, w.head_dim, w.block_size, w.scale, 512, max_seq_len=w.max_seq_len)
        torch.cuda.synchronize()
        assert pb.pa_get_device_status() == 0
        assert_parity(out, oracle_ref(w), "split_kv_decode over NCCL")
    finally:
        dist.destroy_process_group()
