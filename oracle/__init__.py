"""Float64 CPU oracle for paged-attention decode (ctypes wrapper of pa_oracle.c).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library and its Python binding
never import this package, and this package imports nothing from them.

Functions (all float64, inputs as numpy arrays; fp16 tensors are passed as
their uint16 bit patterns):

* ``paged_decode``       -- the definition  softmax(scale q K^T) V  per (seq, head),
                            gathered through the block table.
* ``paged_decode_one``   -- the same for a single (seq, head).
* ``partition_partials`` -- the method's first pass: partitions of P tokens,
                            tiles folded with the alpha/beta online-softmax rule
                            of the "paged_attention_v2_triton.py" commit page.
* ``combine_lse`` / ``combine_fold`` -- the second pass over the partials
                            ("docs" commit page, Phase 2 reduce).
* ``prefix_attention``   -- chunked-prefill attention: each new token attends to
                            its sequence's paged context and causally to the chunk
                            ("qwen3_6_scripts/paged_attn.py" commit page, prefix path).
* ``half_to_double``     -- exact binary16 decode, written from the format.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)


def build(force: bool = False) -> str:
    """Compile pa_oracle.c into liboracle.so with gcc (OpenMP when available)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_half_to_double.restype = ctypes.c_double
            lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
            common = [_u16p, _u16p, _u16p, _i32p, _i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_longlong, ctypes.c_double]
            lib.oracle_paged_decode.restype = ctypes.c_int
            lib.oracle_paged_decode.argtypes = [_dp] + common + [ctypes.c_int]
            lib.oracle_paged_decode_one.restype = ctypes.c_int
            lib.oracle_paged_decode_one.argtypes = [_dp] + common + [ctypes.c_int, ctypes.c_int]
            lib.oracle_partition_partials.restype = ctypes.c_int
            lib.oracle_partition_partials.argtypes = [_dp, _dp, _dp] + common + [ctypes.c_int] * 4
            pre = [_u16p, _u16p, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_longlong,
                   ctypes.c_double]
            lib.oracle_prefix_attention.restype = ctypes.c_int
            lib.oracle_prefix_attention.argtypes = [_dp] + pre + [ctypes.c_int]
            lib.oracle_prefix_attention_one.restype = ctypes.c_int
            lib.oracle_prefix_attention_one.argtypes = [_dp] + pre + [ctypes.c_int, ctypes.c_int]
            for name in ("oracle_combine_lse", "oracle_combine_fold"):
                fn = getattr(lib, name)
                fn.restype = ctypes.c_int
                fn.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int, ctypes.c_int]
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _bits(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("fp16 data must be float16 or its uint16 bit pattern")
    return np.ascontiguousarray(a)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a, t):
    return a.ctypes.data_as(t)


def _common(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
            block_size, scale):
    q, k, v = _bits(q), _bits(k_cache), _bits(v_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    num_seqs = int(sl.shape[0])
    mbps = int(bt.shape[1]) if bt.ndim == 2 else 0
    row = num_kv_heads * block_size * head_dim
    num_blocks = k.size // row if row else 0
    if q.size != num_seqs * num_heads * head_dim or k.size != v.size or k.size != num_blocks * row:
        raise OracleError("shape mismatch")
    keep = (q, k, v, bt, sl)
    args = [_ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), _ptr(bt, _i32p), _ptr(sl, _i32p),
            num_seqs, mbps, num_heads, num_kv_heads, head_dim, block_size, num_blocks, float(scale)]
    return keep, args, num_seqs


def _check(rc: int):
    if rc < 0:
        raise OracleError({-1: "bad argument", -2: "block id out of range",
                           -3: "seq_len out of range"}.get(rc, f"error {rc}"))


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits) & 0xFFFF)


def paged_decode(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                 block_size, scale, threads: int = 0) -> np.ndarray:
    """float64 [num_seqs, num_heads, head_dim]; cache layout [blocks, kv_heads, block_size, head_dim]."""
    keep, args, num_seqs = _common(q, k_cache, v_cache, block_tables, seq_lens, num_heads,
                                   num_kv_heads, head_dim, block_size, scale)
    out = np.zeros((num_seqs, num_heads, head_dim), dtype=np.float64)
    _check(_load().oracle_paged_decode(_ptr(out, _dp), *args, int(threads)))
    del keep
    return out


def paged_decode_one(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                     block_size, scale, b: int, h: int) -> np.ndarray:
    keep, args, _ = _common(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads,
                            head_dim, block_size, scale)
    out = np.zeros((head_dim,), dtype=np.float64)
    _check(_load().oracle_paged_decode_one(_ptr(out, _dp), *args, int(b), int(h)))
    del keep
    return out


def partition_partials(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                       block_size, scale, b: int, h: int, partition_size: int, tile_size: int):
    """Returns (m [n], l [n], acc [n, head_dim]) for one (seq, head)."""
    keep, args, _ = _common(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads,
                            head_dim, block_size, scale)
    L = int(np.asarray(seq_lens)[b])
    n = (L + partition_size - 1) // partition_size
    m = np.zeros(max(n, 1)); l = np.zeros(max(n, 1)); acc = np.zeros((max(n, 1), head_dim))
    rc = _load().oracle_partition_partials(_ptr(m, _dp), _ptr(l, _dp), _ptr(acc, _dp), *args,
                                           int(b), int(h), int(partition_size), int(tile_size))
    _check(rc)
    del keep
    return m[:rc], l[:rc], acc[:rc]


def _combine(name, m, l, acc):
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    n, d = (acc.shape[0], acc.shape[1]) if acc.ndim == 2 else (0, 1)
    out = np.zeros((d,), dtype=np.float64)
    _check(getattr(_load(), name)(_ptr(out, _dp), _ptr(m, _dp), _ptr(l, _dp), _ptr(acc, _dp), n, d))
    return out


def combine_lse(m, l, acc) -> np.ndarray:
    return _combine("oracle_combine_lse", m, l, acc)


def combine_fold(m, l, acc) -> np.ndarray:
    return _combine("oracle_combine_fold", m, l, acc)


def split_decode(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                 block_size, scale, partition_size: int, tile_size: int, form: str = "lse") -> np.ndarray:
    """Both passes of the method for every (seq, head)."""
    sl = np.asarray(seq_lens)
    out = np.zeros((sl.shape[0], num_heads, head_dim))
    comb = combine_lse if form == "lse" else combine_fold
    for b in range(sl.shape[0]):
        for h in range(num_heads):
            m, l, acc = partition_partials(q, k_cache, v_cache, block_tables, seq_lens, num_heads,
                                           num_kv_heads, head_dim, block_size, scale, b, h,
                                           partition_size, tile_size)
            out[b, h] = comb(m, l, acc.reshape(len(m), head_dim)) if len(m) else 0.0
    return out


def _prefix_args(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_heads,
                 num_kv_heads, head_dim, block_size, scale):
    q, kn, vn, k, v = _bits(q), _bits(k_new), _bits(v_new), _bits(k_cache), _bits(v_cache)
    bt, cl, qs = _i32(block_tables), _i32(context_lens), _i32(query_start_loc)
    num_seqs = int(cl.shape[0])
    num_tokens = int(qs[-1]) if qs.size else 0
    mbps = int(bt.shape[1]) if bt.ndim == 2 else 0
    row = num_kv_heads * block_size * head_dim
    num_blocks = k.size // row if row else 0
    if (q.size != num_tokens * num_heads * head_dim or kn.size != num_tokens * num_kv_heads * head_dim
            or vn.size != kn.size or qs.size != num_seqs + 1 or k.size != v.size):
        raise OracleError("shape mismatch")
    keep = (q, kn, vn, k, v, bt, cl, qs)
    args = [_ptr(q, _u16p), _ptr(kn, _u16p), _ptr(vn, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), _ptr(bt, _i32p),
            _ptr(cl, _i32p), _ptr(qs, _i32p), num_seqs, num_tokens, mbps, num_heads, num_kv_heads, head_dim,
            block_size, num_blocks, float(scale)]
    return keep, args, num_tokens


def prefix_attention(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_heads,
                     num_kv_heads, head_dim, block_size, scale, threads: int = 0) -> np.ndarray:
    """float64 [num_tokens, num_heads, head_dim] of chunked-prefill attention."""
    keep, args, n = _prefix_args(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                                 num_heads, num_kv_heads, head_dim, block_size, scale)
    out = np.zeros((n, num_heads, head_dim), dtype=np.float64)
    _check(_load().oracle_prefix_attention(_ptr(out, _dp), *args, int(threads)))
    del keep
    return out


def prefix_attention_one(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_heads,
                         num_kv_heads, head_dim, block_size, scale, tok: int, h: int) -> np.ndarray:
    keep, args, _ = _prefix_args(q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                                 num_heads, num_kv_heads, head_dim, block_size, scale)
    out = np.zeros((head_dim,), dtype=np.float64)
    _check(_load().oracle_prefix_attention_one(_ptr(out, _dp), *args, int(tok), int(h)))
    del keep
    return out
