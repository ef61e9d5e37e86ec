"""Pins of the chunked-prefill oracle (CPU only).

The oracle's prefix attention is tied to: torch's dense scaled-dot-product
attention (a library routine) with a causal mask when there is no context and
an explicit context-plus-causal mask otherwise, on K/V built dense first and
then scattered into a shuffled paged pool; the decode oracle on a cache that
holds the single new token; the closed form for the first token of an empty
sequence; and exclusion of future chunk tokens and of cache slots past the
context.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _f16(a):
    return np.asarray(a, dtype=np.float16)


def _build(ctx_lens, q_lens, H, Hkv, D, bs, seed, extra_blocks=2):
    """Dense context K/V per sequence scattered into a shuffled paged pool, plus packed chunk tensors."""
    rng = np.random.default_rng(seed)
    nblk = [(C + bs - 1) // bs for C in ctx_lens]
    NB = max(sum(nblk) + extra_blocks, 1)
    perm = rng.permutation(NB)
    kc = _f16(rng.standard_normal((NB, Hkv, bs, D)))
    vc = _f16(rng.standard_normal((NB, Hkv, bs, D)))
    bt = np.full((len(ctx_lens), max(max(nblk, default=0), 1)), -1, dtype=np.int32)
    dk, dv = [], []
    off = 0
    for b, C in enumerate(ctx_lens):
        kd = _f16(rng.standard_normal((Hkv, C, D)))
        vd = _f16(rng.standard_normal((Hkv, C, D)))
        for i in range(nblk[b]):
            phys = perm[off + i]
            bt[b, i] = phys
            n = min(bs, C - i * bs)
            kc[phys, :, :n] = kd[:, i * bs:i * bs + n]
            vc[phys, :, :n] = vd[:, i * bs:i * bs + n]
        off += nblk[b]
        dk.append(kd)
        dv.append(vd)
    T = sum(q_lens)
    qs = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    q = _f16(rng.standard_normal((T, H, D)))
    kn = _f16(rng.standard_normal((T, Hkv, D)))
    vn = _f16(rng.standard_normal((T, Hkv, D)))
    return q, kn, vn, kc, vc, bt, np.array(ctx_lens, dtype=np.int32), qs, dk, dv


def _sdpa_reference(q, kn, vn, dk, dv, ctx_lens, qs, H, Hkv, D, scale):
    G = H // Hkv
    outs = []
    for b, C in enumerate(ctx_lens):
        a, e = qs[b], qs[b + 1]
        L = e - a
        keys = np.concatenate([dk[b], kn[a:e].transpose(1, 0, 2)], axis=1).astype(np.float64)   # [Hkv, C+L, D]
        vals = np.concatenate([dv[b], vn[a:e].transpose(1, 0, 2)], axis=1).astype(np.float64)
        kk = torch.from_numpy(keys).repeat_interleave(G, 0)[None]
        vv = torch.from_numpy(vals).repeat_interleave(G, 0)[None]
        qq = torch.from_numpy(q[a:e].astype(np.float64).transpose(1, 0, 2))[None]              # [1, H, L, D]
        if C == 0:
            o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True, scale=scale)
        else:
            mask = torch.ones((L, C + L), dtype=torch.bool)
            mask[:, C:] = torch.tril(torch.ones((L, L), dtype=torch.bool))
            o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=scale)
        outs.append(o[0].numpy().transpose(1, 0, 2))                                               # [L, H, D]
    return np.concatenate(outs, axis=0)


@pytest.mark.parametrize("ctx,ql,H,Hkv,D,bs", [
    ([0, 0, 0], [1, 5, 17], 4, 2, 16, 4),            # no context: causal self-attention over the chunk
    ([13, 0, 40], [3, 8, 1], 6, 1, 32, 8),
    ([16, 33], [16, 7], 24, 4, 64, 16),
    ([5], [30], 8, 8, 8, 4),
])
def test_prefix_equals_dense_masked_library_attention(ctx, ql, H, Hkv, D, bs):
    q, kn, vn, kc, vc, bt, cl, qs, dk, dv = _build(ctx, ql, H, Hkv, D, bs, seed=sum(ctx) + D)
    scale = 1 / math.sqrt(D)
    got = oracle.prefix_attention(q, kn, vn, kc, vc, bt, cl, qs, H, Hkv, D, bs, scale)
    ref = _sdpa_reference(q, kn, vn, dk, dv, ctx, qs, H, Hkv, D, scale)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_single_new_token_equals_decode_over_the_extended_cache():
    ctx, H, Hkv, D, bs = [7, 16, 30], 6, 2, 16, 8
    q, kn, vn, kc, vc, bt, cl, qs, dk, dv = _build(ctx, [1, 1, 1], H, Hkv, D, bs, seed=3, extra_blocks=6)
    pre = oracle.prefix_attention(q, kn, vn, kc, vc, bt, cl, qs, H, Hkv, D, bs, 0.3)
    # append each sequence's new token to its paged context, then decode
    kc2, vc2, bt2 = kc.copy(), vc.copy(), np.concatenate([bt, np.full((3, 1), -1, np.int32)], axis=1)
    used = set(bt[bt >= 0].tolist())
    free = [i for i in range(kc.shape[0]) if i not in used]
    for b, C in enumerate(ctx):
        blk = C // bs
        if bt2[b, blk] < 0:
            bt2[b, blk] = free.pop()
        kc2[bt2[b, blk], :, C % bs] = kn[b]
        vc2[bt2[b, blk], :, C % bs] = vn[b]
    dec = oracle.paged_decode(q, kc2, vc2, bt2, np.array(ctx) + 1, H, Hkv, D, bs, 0.3)
    np.testing.assert_allclose(pre, dec, rtol=1e-13, atol=1e-15)


def test_first_token_without_context_returns_its_own_value():
    q, kn, vn, kc, vc, bt, cl, qs, dk, dv = _build([0, 0], [4, 2], 4, 2, 8, 4, seed=4)
    out = oracle.prefix_attention(q, kn, vn, kc, vc, bt, cl, qs, 4, 2, 8, 4, 0.5)
    for tok in (0, 4):
        for h in range(4):
            assert np.array_equal(out[tok, h], vn[tok, h // 2].astype(np.float64))


def test_future_chunk_tokens_and_slots_past_the_context_are_excluded():
    ctx, ql = [10, 3], [6, 5]
    q, kn, vn, kc, vc, bt, cl, qs, dk, dv = _build(ctx, ql, 4, 1, 8, 4, seed=5)
    clean = oracle.prefix_attention(q, kn, vn, kc, vc, bt, cl, qs, 4, 1, 8, 4, 0.4)
    kn2, vn2, kc2, vc2 = kn.copy(), vn.copy(), kc.copy(), vc.copy()
    for b in range(2):
        last = qs[b + 1] - 1
        kn2[last], vn2[last] = np.nan, np.inf            # the chunk's last token
        phys = bt[b, ctx[b] // 4]
        kc2[phys, :, ctx[b] % 4:], vc2[phys, :, ctx[b] % 4:] = np.nan, np.nan
    poisoned = oracle.prefix_attention(q, kn2, vn2, kc2, vc2, bt, cl, qs, 4, 1, 8, 4, 0.4)
    keep = np.ones(qs[-1], bool)
    keep[qs[1:] - 1] = False                              # rows that attend to the poisoned token
    assert np.array_equal(clean[keep], poisoned[keep])


def test_one_row_matches_the_batch():
    q, kn, vn, kc, vc, bt, cl, qs, dk, dv = _build([9, 20], [5, 3], 6, 2, 16, 4, seed=6)
    full = oracle.prefix_attention(q, kn, vn, kc, vc, bt, cl, qs, 6, 2, 16, 4, 0.25)
    for tok in range(qs[-1]):
        for h in (0, 5):
            assert np.array_equal(full[tok, h], oracle.prefix_attention_one(q, kn, vn, kc, vc, bt, cl, qs, 6, 2,
                                                                            16, 4, 0.25, tok, h))
