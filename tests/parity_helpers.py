"""Helpers shared by the GPU parity tests: host copies for the oracle and the
pass criterion.

Pass criterion (fp16 output, fp32 accumulation): every element must satisfy
    |gpu - ref| <= ATOL + RTOL * |ref|,   ATOL = 2e-3, RTOL = 1e-2,
the max-abs 2e-3 / max-rel 1e-2 bound read element-wise so that it stays
meaningful where the reference is near zero.  The report also gives the
max-abs error, the max relative error over |ref| >= 0.05, and the error
normalised by the output's rms (expected near fp16 output rounding).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL = 2e-3
RTOL = 1e-2


def host_bits(t: torch.Tensor) -> np.ndarray:
    a = t.detach().cpu().contiguous().numpy()
    return a.view(np.uint16) if a.dtype == np.float16 else a


def oracle_ref(w, threads: int = 0) -> np.ndarray:
    return oracle.paged_decode(host_bits(w.q), host_bits(w.k_cache), host_bits(w.v_cache), host_bits(w.block_tables),
                               host_bits(w.seq_lens), w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                               threads=threads)


def oracle_ref_subset(w, seqs, threads: int = 0) -> np.ndarray:
    """Oracle outputs of selected sequences only: their blocks are gathered
    (torch indexing on the device, not the library) into a compact pool."""
    seqs = list(seqs)
    bt = w.block_tables[seqs].long()
    lens = [w.seq_lens_host[s] for s in seqs]
    nblk = [(L + w.block_size - 1) // w.block_size for L in lens]
    ids = torch.cat([bt[i, :n] for i, n in enumerate(nblk)]) if sum(nblk) else torch.zeros(0, dtype=torch.long,
                                                                                           device=bt.device)
    k = host_bits(w.k_cache[ids]) if len(ids) else np.zeros((1,) + tuple(w.k_cache.shape[1:]), np.uint16)
    v = host_bits(w.v_cache[ids]) if len(ids) else np.zeros((1,) + tuple(w.v_cache.shape[1:]), np.uint16)
    new_bt = np.full((len(seqs), max(max(nblk, default=0), 1)), -1, dtype=np.int32)
    off = 0
    for i, n in enumerate(nblk):
        new_bt[i, :n] = np.arange(off, off + n)
        off += n
    q = host_bits(w.q[seqs])
    return oracle.paged_decode(q, k, v, new_bt, np.array(lens, dtype=np.int32), w.num_heads, w.num_kv_heads,
                               w.head_dim, w.block_size, w.scale, threads=threads)


def compare(gpu: torch.Tensor, ref: np.ndarray) -> dict:
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    big = np.abs(ref) >= 0.05
    rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    return {
        "ok": bool(np.all(err <= bound)) and bool(np.all(np.isfinite(g))),
        "max_abs": float(err.max()) if err.size else 0.0,
        "max_rel_big": float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0,
        "err_over_rms": float(np.sqrt(np.mean(err ** 2)) / rms) if rms > 0 else 0.0,
        "worst_excess": float((err - bound).max()) if err.size else 0.0,
    }


def assert_parity(gpu: torch.Tensor, ref: np.ndarray, what: str = "") -> dict:
    r = compare(gpu, ref)
    assert r["ok"], f"{what} parity failed: {r}"
    # fp16 output rounding alone gives ~3e-4 of the rms; a much larger value
    # points at a real error that the loose absolute bound would hide
    assert r["err_over_rms"] < 5e-3, f"{what} error too large relative to the output scale: {r}"
    return r
