"""Pins of the float64 oracle to things other than itself (CPU only).

Each test ties the oracle to a fact the pages or the mathematics fix: the
binary16 format (via numpy), hand-derived worked examples (tests/golden),
a library implementation of dense attention on a layout built the other way
round (dense first, then scattered into a paged pool), closed forms
(single key, zero query, constant V per kv head), an invariant of the method
(partition + alpha/beta combine == unsplit, both second-pass forms agree),
and the exclusion of slots past the sequence end.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")


def _scale(v):
    return {"ln3": math.log(3.0), "ln2": math.log(2.0), "2ln2": 2 * math.log(2.0)}.get(v, v)


def _fp16(a):
    return np.asarray(a, dtype=np.float16)


def test_half_decode_matches_numpy_on_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("case", ["two_token_ln3", "gqa_two_groups"])
def test_golden_outputs(case):
    c = json.load(open(GOLDEN))[case]
    out = oracle.paged_decode(_fp16(c["q"]), _fp16(c["k_cache"]), _fp16(c["v_cache"]),
                              np.array(c["block_tables"]), np.array(c["seq_lens"]), c["num_heads"],
                              c["num_kv_heads"], c["head_dim"], c["block_size"], _scale(c["scale"]))
    np.testing.assert_allclose(out, np.array(c["out"]), rtol=0, atol=1e-14)


def test_golden_partials_and_combine():
    c = json.load(open(GOLDEN))["three_token_two_partitions"]
    args = (_fp16(c["q"]), _fp16(c["k_cache"]), _fp16(c["v_cache"]), np.array(c["block_tables"]),
            np.array(c["seq_lens"]), c["num_heads"], c["num_kv_heads"], c["head_dim"], c["block_size"],
            _scale(c["scale"]))
    for tile in (1, 2):
        m, l, acc = oracle.partition_partials(*args, 0, 0, c["partition_size"], tile)
        np.testing.assert_allclose(m, [_scale(x) for x in c["partials_m"]], rtol=1e-15, atol=0)
        np.testing.assert_allclose(l, c["partials_l"], rtol=1e-15, atol=0)
        np.testing.assert_allclose(acc, c["partials_acc"], rtol=1e-15, atol=0)
        for comb in (oracle.combine_lse, oracle.combine_fold):
            np.testing.assert_allclose(comb(m, l, acc), np.array(c["out"])[0, 0], rtol=1e-14)
    np.testing.assert_allclose(oracle.paged_decode(*args), np.array(c["out"]), rtol=1e-14)


def _dense_then_paged(seq_lens, H, Hkv, D, bs, extra_blocks, seed):
    """Dense per-sequence K/V first, then scattered into a shuffled paged pool."""
    rng = np.random.default_rng(seed)
    nblk = [(L + bs - 1) // bs for L in seq_lens]
    NB = sum(nblk) + extra_blocks
    perm = rng.permutation(NB)
    kc = _fp16(rng.standard_normal((NB, Hkv, bs, D)))
    vc = _fp16(rng.standard_normal((NB, Hkv, bs, D)))
    q = _fp16(rng.standard_normal((len(seq_lens), H, D)))
    mbps = max(nblk) + 1
    bt = np.full((len(seq_lens), mbps), -1, dtype=np.int32)
    dense_k, dense_v = [], []
    off = 0
    for b, L in enumerate(seq_lens):
        kd = _fp16(rng.standard_normal((Hkv, L, D)))
        vd = _fp16(rng.standard_normal((Hkv, L, D)))
        for i in range(nblk[b]):
            phys = perm[off + i]
            bt[b, i] = phys
            n = min(bs, L - i * bs)
            kc[phys, :, :n, :] = kd[:, i * bs:i * bs + n, :]
            vc[phys, :, :n, :] = vd[:, i * bs:i * bs + n, :]
        off += nblk[b]
        dense_k.append(kd)
        dense_v.append(vd)
    return q, kc, vc, bt, np.array(seq_lens, dtype=np.int32), dense_k, dense_v


@pytest.mark.parametrize("H,Hkv,D,bs,lens", [
    (6, 1, 32, 4, [1, 3, 4, 5, 17]),
    (12, 2, 16, 8, [9, 16, 33]),
    (4, 4, 8, 2, [7, 2]),
    (24, 4, 64, 16, [15, 16, 17, 40]),
])
def test_paged_equals_dense_library_attention(H, Hkv, D, bs, lens):
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged(lens, H, Hkv, D, bs, extra_blocks=3, seed=H + D)
    scale = 1.0 / math.sqrt(D)
    out = oracle.paged_decode(q, kc, vc, bt, sl, H, Hkv, D, bs, scale)
    G = H // Hkv
    for b, L in enumerate(lens):
        qq = torch.from_numpy(q[b].astype(np.float64)).view(1, H, 1, D)
        kk = torch.from_numpy(dk[b].astype(np.float64)).repeat_interleave(G, dim=0).view(1, H, L, D)
        vv = torch.from_numpy(dv[b].astype(np.float64)).repeat_interleave(G, dim=0).view(1, H, L, D)
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale)
        np.testing.assert_allclose(out[b], ref.view(H, D).numpy(), rtol=1e-12, atol=1e-13)


def test_single_key_returns_its_value_exactly():
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([1, 1], 6, 2, 32, 4, 2, seed=1)
    out = oracle.paged_decode(q, kc, vc, bt, sl, 6, 2, 32, 4, 0.125)
    for b in range(2):
        for h in range(6):
            assert np.array_equal(out[b, h], dv[b][h // 3, 0].astype(np.float64))


def test_zero_query_gives_mean_of_values():
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([37, 5], 4, 2, 16, 8, 0, seed=2)
    q[:] = 0
    out = oracle.paged_decode(q, kc, vc, bt, sl, 4, 2, 16, 8, 0.25)
    for b in range(2):
        for h in range(4):
            np.testing.assert_allclose(out[b, h], dv[b][h // 2].astype(np.float64).mean(axis=0),
                                       rtol=1e-13, atol=1e-15)


def test_identical_keys_give_mean_of_values():
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([23], 2, 1, 8, 4, 0, seed=3)
    kc[:] = _fp16(np.linspace(-2, 2, 8))
    out = oracle.paged_decode(q, kc, vc, bt, sl, 2, 1, 8, 4, 0.5)
    np.testing.assert_allclose(out[0, 0], dv[0][0].astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-15)


def test_dominant_key_without_overflow():
    # scores of order 1e5: a plain exp(s) would overflow; subtracting the max must not.
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([20], 1, 1, 4, 4, 0, seed=4)
    q[:] = _fp16([256, 0, 0, 0])
    kc[:] = 0
    winner = 13
    kc[bt[0, winner // 4], 0, winner % 4, 0] = 400.0   # s = 256*400 = 102400 vs 0 elsewhere
    out = oracle.paged_decode(q, kc, vc, bt, sl, 1, 1, 4, 4, 1.0)
    assert np.all(np.isfinite(out))
    assert np.array_equal(out[0, 0], dv[0][0, winner].astype(np.float64))


def test_slots_past_the_end_are_excluded():
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([6, 13], 4, 2, 8, 4, 1, seed=5)
    clean = oracle.paged_decode(q, kc, vc, bt, sl, 4, 2, 8, 4, 0.3)
    for b, L in enumerate([6, 13]):
        phys = bt[b, L // 4]
        kc[phys, :, L % 4:, :] = np.nan
        vc[phys, :, L % 4:, :] = np.inf
    poisoned = oracle.paged_decode(q, kc, vc, bt, sl, 4, 2, 8, 4, 0.3)
    assert np.array_equal(clean, poisoned)


def test_block_table_permutation_is_exact():
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([33, 12], 6, 3, 16, 4, 5, seed=6)
    base = oracle.paged_decode(q, kc, vc, bt, sl, 6, 3, 16, 4, 0.25)
    rng = np.random.default_rng(7)
    perm = rng.permutation(kc.shape[0])          # new position of every block
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    bt2 = np.where(bt >= 0, perm[np.maximum(bt, 0)], -1).astype(np.int32)
    assert np.array_equal(base, oracle.paged_decode(q, kc2, vc2, bt2, sl, 6, 3, 16, 4, 0.25))


def test_empty_sequence_gives_zero():
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([5, 1], 2, 1, 8, 4, 0, seed=8)
    sl = np.array([0, 1], dtype=np.int32)
    out = oracle.paged_decode(q, kc, vc, bt, sl, 2, 1, 8, 4, 0.5)
    assert np.array_equal(out[0], np.zeros((2, 8)))
    m, l, acc = oracle.partition_partials(q, kc, vc, bt, sl, 2, 1, 8, 4, 0.5, 0, 0, 4, 4)
    assert len(m) == 0


def test_out_of_range_block_id_is_an_error():
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([8], 1, 1, 4, 4, 0, seed=9)
    bt[0, 1] = kc.shape[0]
    with pytest.raises(oracle.OracleError):
        oracle.paged_decode(q, kc, vc, bt, sl, 1, 1, 4, 4, 1.0)


@pytest.mark.parametrize("P,T", [(4, 4), (16, 4), (16, 16), (12, 4), (48, 16), (512, 16), (7, 3), (1000, 1000)])
@pytest.mark.parametrize("form", ["lse", "fold"])
def test_partition_and_combine_equals_unsplit(P, T, form):
    lens = [1, 15, 16, 17, 64, 100, 511 % 200 + 3]
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged(lens, 6, 2, 16, 4, 0, seed=10)
    kc = (kc.astype(np.float32) * 3).astype(np.float16)   # wider score range
    ref = oracle.paged_decode(q, kc, vc, bt, sl, 6, 2, 16, 4, 0.25)
    got = oracle.split_decode(q, kc, vc, bt, sl, 6, 2, 16, 4, 0.25, P, T, form)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("where", ["first", "last", "middle"])
def test_tile_holding_the_max_in_any_position(where):
    # Regression for the reference-max mistake: the partition max may sit in
    # the first tile, the last tile or between; every placement must match.
    L, bs = 64, 4
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([L], 1, 1, 8, bs, 0, seed=11)
    q[:] = _fp16([1] * 8)
    kc[:] = _fp16(np.random.default_rng(12).uniform(-0.5, 0.5, kc.shape))
    t = {"first": 1, "last": L - 2, "middle": 30}[where]
    kc[bt[0, t // bs], 0, t % bs, :] = 3.0
    ref = oracle.paged_decode(q, kc, vc, bt, sl, 1, 1, 8, bs, 1.0)
    for T in (4, 16):
        got = oracle.split_decode(q, kc, vc, bt, sl, 1, 1, 8, bs, 1.0, L, T, "lse")
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_lse_and_fold_agree_on_random_partials():
    rng = np.random.default_rng(13)
    for n in (1, 2, 5, 64):
        m = rng.normal(0, 20, n)
        l = rng.uniform(0.5, 100, n)
        acc = rng.normal(0, 1, (n, 32))
        np.testing.assert_allclose(oracle.combine_lse(m, l, acc), oracle.combine_fold(m, l, acc),
                                   rtol=1e-12, atol=1e-14)
    z = oracle.combine_lse(np.zeros(0), np.zeros(0), np.zeros((0, 4)))
    assert np.array_equal(z, np.zeros(4))


@pytest.mark.parametrize("H,Hkv,D,bs,lens", [
    (6, 2, 16, 4, [1, 9, 23]),      # more heads than sequences
    (4, 4, 8, 2, [7, 2, 5, 11, 3]),  # more sequences than heads
    (24, 4, 64, 16, [15, 40]),
])
def test_decode_one_row_by_row_against_dense_library_attention(H, Hkv, D, bs, lens):
    # The single-(sequence, head) entry point, pinned independently of the
    # batch routine: each (b, h) row against torch's dense attention on the
    # dense K/V the paged pool was scattered from, and against the batch.
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged(lens, H, Hkv, D, bs, extra_blocks=2, seed=100 + H + D)
    scale = 1.0 / math.sqrt(D)
    G = H // Hkv
    full = oracle.paged_decode(q, kc, vc, bt, sl, H, Hkv, D, bs, scale)
    for b, L in enumerate(lens):
        for h in range(H):
            row = oracle.paged_decode_one(q, kc, vc, bt, sl, H, Hkv, D, bs, scale, b, h)
            qq = torch.from_numpy(q[b, h].astype(np.float64)).view(1, 1, 1, D)
            kk = torch.from_numpy(dk[b][h // G].astype(np.float64)).view(1, 1, L, D)
            vv = torch.from_numpy(dv[b][h // G].astype(np.float64)).view(1, 1, L, D)
            ref = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, scale=scale).view(D).numpy()
            np.testing.assert_allclose(row, ref, rtol=1e-12, atol=1e-13)
            assert np.array_equal(row, full[b, h])


def test_decode_one_closed_forms_and_bounds():
    q, kc, vc, bt, sl, dk, dv = _dense_then_paged([1, 30], 4, 2, 8, 4, 1, seed=101)
    # one key: its value exactly; zero query: the mean of the values
    for h in range(4):
        assert np.array_equal(oracle.paged_decode_one(q, kc, vc, bt, sl, 4, 2, 8, 4, 0.5, 0, h),
                              dv[0][h // 2, 0].astype(np.float64))
    q0 = q.copy()
    q0[1] = 0
    for h in range(4):
        np.testing.assert_allclose(oracle.paged_decode_one(q0, kc, vc, bt, sl, 4, 2, 8, 4, 0.5, 1, h),
                                   dv[1][h // 2].astype(np.float64).mean(axis=0), rtol=1e-13, atol=1e-15)
    for b, h in ((2, 0), (-1, 0), (0, 4), (0, -1)):
        with pytest.raises(oracle.OracleError):
            oracle.paged_decode_one(q, kc, vc, bt, sl, 4, 2, 8, 4, 0.5, b, h)
