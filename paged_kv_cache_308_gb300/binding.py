"""ctypes binding of libpa_decode.so (include/pa_decode.h), same names as the C ABI.

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  Tensors are torch tensors on the GPU; their device pointers,
sizes and the current CUDA stream are handed to the C functions.  If the
shared library is missing the import of this module fails loudly -- there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa_decode.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "pa_decode.h")

PA_OK = 0
PA_ERR_INVALID_ARG = -1
PA_ERR_UNSUPPORTED = -2
PA_ERR_CUDA = -3
PA_ERR_OOM = -4
PA_ERR_WORKSPACE = -5

PA_DEV_BAD_BLOCK_ID = 1
PA_DEV_BAD_SEQ_LEN = 2
PA_DEV_TIMEOUT = 4

PA_MODE_AUTO = 0
PA_MODE_SINGLE = 1
PA_MODE_SPLIT = 2
PA_MODE_FUSED = 3
PA_MODE_PERSISTENT = 4
PA_MODE_FLAT = 5
MODES = {"auto": PA_MODE_AUTO, "single": PA_MODE_SINGLE, "split": PA_MODE_SPLIT, "fused": PA_MODE_FUSED, "flat": PA_MODE_FLAT,
         "persistent": PA_MODE_PERSISTENT}

PA_FLAG_FORCE_TIMEOUT = 1
PA_FLAG_PREFIX_WARP_MMA = 2
PA_FLAG_POOLED = 4
PA_FLAG_DETERMINISTIC = 8
PA_FLAG_UNIFORM_LENGTHS = 16
PA_FLAG_PREFIX_GRID = 32


class pa_decode_args(ctypes.Structure):
    _fields_ = [
        ("out", ctypes.c_void_p), ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p), ("block_tables", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("num_seqs", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int), ("max_seq_len", ctypes.c_int),
        ("num_blocks", ctypes.c_int64), ("num_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int), ("scale", ctypes.c_float),
    ]


class pa_decode_opts(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int), ("partition_size", ctypes.c_int), ("flags", ctypes.c_int),
        ("wait_limit", ctypes.c_uint), ("event_partition_begin", ctypes.c_void_p),
        ("event_partition_end", ctypes.c_void_p), ("warps", ctypes.c_int), ("stages", ctypes.c_int),
    ]


class pa_decode_plan_t(ctypes.Structure):
    _fields_ = [
        ("mode", ctypes.c_int), ("partition_size", ctypes.c_int), ("grid_x", ctypes.c_int),
        ("grid_y", ctypes.c_int), ("grid_z", ctypes.c_int), ("threads", ctypes.c_int),
        ("smem_bytes", ctypes.c_int), ("launch_reduce", ctypes.c_int), ("reduce_grid_x", ctypes.c_int),
        ("reduce_grid_y", ctypes.c_int), ("reduce_grid_z", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t),
        ("stages", ctypes.c_int), ("max_partitions", ctypes.c_int), ("pooled", ctypes.c_int),
        ("coop", ctypes.c_int),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class pa_prefix_args(ctypes.Structure):
    _fields_ = [
        ("out", ctypes.c_void_p), ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
        ("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("block_tables", ctypes.c_void_p),
        ("context_lens", ctypes.c_void_p), ("query_start_loc", ctypes.c_void_p), ("num_seqs", ctypes.c_int),
        ("num_tokens", ctypes.c_int), ("max_blocks_per_seq", ctypes.c_int), ("max_context_len", ctypes.c_int),
        ("max_query_len", ctypes.c_int), ("num_blocks", ctypes.c_int64), ("num_heads", ctypes.c_int),
        ("num_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("block_size", ctypes.c_int),
        ("scale", ctypes.c_float),
    ]


class pa_prefix_split_opts(ctypes.Structure):
    _fields_ = [("parts", ctypes.c_int), ("units", ctypes.c_int)]


class PaDecodeError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})" if what else f"{status_string(code)} ({code})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with `python -m paged_kv_cache_308_gb300.build` "
                          "(or __graft_entry__.build()); there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
    lib.pa_decode.restype = i32
    lib.pa_decode.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, i32, i32, i32, f32, vp]
    lib.pa_decode_ex.restype = i32
    lib.pa_decode_ex.argtypes = [ctypes.POINTER(pa_decode_args), ctypes.POINTER(pa_decode_opts), vp,
                                 ctypes.c_size_t, vp]
    lib.pa_decode_plan.restype = i32
    lib.pa_decode_plan.argtypes = [ctypes.POINTER(pa_decode_args), ctypes.POINTER(pa_decode_opts), i32,
                                   ctypes.POINTER(pa_decode_plan_t)]
    lib.pa_decode_workspace_size.restype = ctypes.c_size_t
    lib.pa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.pa_get_device_status.restype = i32
    lib.pa_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [i32]
    lib.pa_release_workspace.restype = None
    lib.pa_release_workspace.argtypes = []
    lib.pa_version.restype = i32
    lib.pa_version.argtypes = []
    lib.pa_prefix.restype = i32
    lib.pa_prefix.argtypes = [vp] * 9 + [i32] * 5 + [i64, i32, i32, i32, i32, f32, vp]
    lib.pa_prefix_ex.restype = i32
    lib.pa_prefix_ex.argtypes = [ctypes.POINTER(pa_prefix_args), ctypes.POINTER(pa_decode_opts), vp]
    lib.pa_prefix_split_workspace_size.restype = i32
    lib.pa_prefix_split_workspace_size.argtypes = [ctypes.POINTER(pa_prefix_args), ctypes.POINTER(pa_prefix_split_opts),
                                                   ctypes.POINTER(ctypes.c_size_t)]
    lib.pa_prefix_split.restype = i32
    lib.pa_prefix_split.argtypes = [ctypes.POINTER(pa_prefix_args), ctypes.POINTER(pa_decode_opts),
                                    ctypes.POINTER(pa_prefix_split_opts), vp, ctypes.c_size_t, vp]
    lib.pa_decode_partials.restype = i32
    lib.pa_decode_partials.argtypes = [ctypes.POINTER(pa_decode_args), ctypes.POINTER(pa_decode_opts), i32, i32, i32,
                                       vp, vp, vp, vp]
    lib.pa_merge_partials.restype = i32
    lib.pa_merge_partials.argtypes = [vp, vp, vp, vp, vp] + [i32] * 7 + [vp]
    lib.pa_decode_noalloc.restype = i32
    lib.pa_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i32, i32, i32, i64, i32, i32, i32, i32, f32, vp]
    return lib


lib = _load()


def header_functions() -> list:
    """Names of the functions include/pa_decode.h declares."""
    text = open(HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text)))


def status_string(code: int) -> str:
    return lib.pa_status_string(int(code)).decode()


def version() -> int:
    return lib.pa_version()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def make_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
              block_size, scale, max_seq_len) -> pa_decode_args:
    return pa_decode_args(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(seq_lens),
        int(seq_lens.shape[0]), int(block_tables.shape[1]) if block_tables.dim() == 2 else 0,
        int(max_seq_len), int(k_cache.shape[0]), int(num_heads), int(num_kv_heads), int(head_dim),
        int(block_size), float(scale))


def make_opts(mode="auto", partition_size: int = 0, flags: int = 0, wait_limit: int = 0,
              events=None, warps: int = 0, stages: int = 0) -> pa_decode_opts:
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    ev0 = ev1 = None
    if events is not None:
        ev0, ev1 = (e.cuda_event if hasattr(e, "cuda_event") else e for e in events)
    return pa_decode_opts(m, int(partition_size), int(flags), int(wait_limit), ev0, ev1, int(warps), int(stages))


def _check_tensors(out, q, k_cache, v_cache, block_tables, seq_lens):
    for name, t, dt in (("out", out, torch.float16), ("q", q, torch.float16), ("k_cache", k_cache, torch.float16),
                        ("v_cache", v_cache, torch.float16), ("block_tables", block_tables, torch.int32),
                        ("seq_lens", seq_lens, torch.int32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
              block_size, scale, stream=None, *, max_seq_len: int) -> None:
    """The library-owned-workspace call; raises PaDecodeError on a non-zero code."""
    _check_tensors(out, q, k_cache, v_cache, block_tables, seq_lens)
    rc = lib.pa_decode(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                       block_tables.data_ptr(), seq_lens.data_ptr(), int(seq_lens.shape[0]),
                       int(block_tables.shape[1]), int(max_seq_len), int(k_cache.shape[0]), int(num_heads),
                       int(num_kv_heads), int(head_dim), int(block_size), float(scale), _stream_handle(stream))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_decode")


def pa_decode_plan(out, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                   block_size, scale, *, max_seq_len: int, num_sms: int = 0, **opt) -> dict:
    args = make_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                     block_size, scale, max_seq_len)
    plan = pa_decode_plan_t()
    rc = lib.pa_decode_plan(ctypes.byref(args), ctypes.byref(make_opts(**opt)), int(num_sms), ctypes.byref(plan))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_decode_plan")
    return plan.as_dict()


def pa_decode_ex(out, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                 block_size, scale, stream=None, *, max_seq_len: int, workspace: Optional[torch.Tensor] = None,
                 **opt) -> None:
    """Caller-workspace call (graph-capturable).  `workspace` is a uint8 CUDA tensor or None."""
    _check_tensors(out, q, k_cache, v_cache, block_tables, seq_lens)
    args = make_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                     block_size, scale, max_seq_len)
    opts = make_opts(**opt)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib.pa_decode_ex(ctypes.byref(args), ctypes.byref(opts), ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_decode_ex")


def alloc_workspace(plan: dict, device) -> Optional[torch.Tensor]:
    """A zeroed device buffer of plan['workspace_bytes'] (256-byte aligned by the
    caching allocator); zero because the fused combine's tickets start at zero."""
    n = int(plan["workspace_bytes"])
    return torch.zeros(n, dtype=torch.uint8, device=device) if n else None


def pa_decode_workspace_size(num_seqs, max_seq_len, num_heads, head_dim, partition_size=0) -> int:
    return lib.pa_decode_workspace_size(int(num_seqs), int(max_seq_len), int(num_heads), int(head_dim),
                                        int(partition_size))


def pa_get_device_status(stream=None) -> int:
    st = ctypes.c_int(0)
    rc = lib.pa_get_device_status(_stream_handle(stream), ctypes.byref(st))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_get_device_status")
    return st.value


def pa_status_string(code: int) -> str:
    return status_string(code)


def pa_release_workspace() -> None:
    lib.pa_release_workspace()


def pa_version() -> int:
    return lib.pa_version()


def decode_workload(w, out: Optional[torch.Tensor] = None, stream=None, workspace: Optional[torch.Tensor] = None,
                    **opt) -> torch.Tensor:
    """Run one decode call on a workloads.Workload (tensors already on the GPU).
    With options, `workspace` (kept across calls, e.g. for the pooled split's
    claim counters) replaces a fresh zeroed buffer."""
    if out is None:
        out = torch.empty_like(w.q)
    if opt:
        plan = pa_decode_plan(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads,
                              w.num_kv_heads, w.head_dim, w.block_size, w.scale, max_seq_len=w.max_seq_len, **opt)
        ws = workspace if workspace is not None else alloc_workspace(plan, w.q.device)
        if ws is not None and stream is not None:
            ws.record_stream(stream)  # keep the buffer alive until that stream's work is done
        pa_decode_ex(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                     w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len, workspace=ws, **opt)
    else:
        pa_decode(out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads,
                  w.head_dim, w.block_size, w.scale, stream, max_seq_len=w.max_seq_len)
    return out


def pa_decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                      block_size, scale, stream=None, *, max_seq_len: int) -> None:
    """The no-allocation call: the partials live in the library's fixed device
    scratch (PA_NOALLOC_SCRATCH_BYTES); raises PaDecodeError on a non-zero code."""
    _check_tensors(out, q, k_cache, v_cache, block_tables, seq_lens)
    rc = lib.pa_decode_noalloc(out.data_ptr(), q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            seq_lens.data_ptr(), int(seq_lens.shape[0]), int(block_tables.shape[1]), int(max_seq_len),
            int(k_cache.shape[0]), int(num_heads), int(num_kv_heads), int(head_dim), int(block_size), float(scale),
            _stream_handle(stream))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_decode_noalloc")


def _prefix_args(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_heads,
                 num_kv_heads, head_dim, block_size, scale, max_context_len, max_query_len) -> pa_prefix_args:
    for name, t, dt in (("out", out, torch.float16), ("q", q, torch.float16), ("k_new", k_new, torch.float16),
                        ("v_new", v_new, torch.float16), ("k_cache", k_cache, torch.float16),
                        ("v_cache", v_cache, torch.float16), ("block_tables", block_tables, torch.int32),
                        ("context_lens", context_lens, torch.int32),
                        ("query_start_loc", query_start_loc, torch.int32)):
        if t.dtype != dt or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    return pa_prefix_args(out.data_ptr(), q.data_ptr(), k_new.data_ptr(), v_new.data_ptr(), k_cache.data_ptr(),
                          v_cache.data_ptr(), block_tables.data_ptr(), context_lens.data_ptr(),
                          query_start_loc.data_ptr(), int(context_lens.shape[0]), int(q.shape[0]),
                          int(block_tables.shape[1]), int(max_context_len), int(max_query_len),
                          int(k_cache.shape[0]), int(num_heads), int(num_kv_heads), int(head_dim), int(block_size),
                          float(scale))


def pa_prefix(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_heads,
              num_kv_heads, head_dim, block_size, scale, stream=None, *, max_context_len: int, max_query_len: int,
              **opt) -> None:
    """Chunked-prefill attention (see include/pa_decode.h); options as for pa_decode_ex."""
    args = _prefix_args(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                        num_heads, num_kv_heads, head_dim, block_size, scale, max_context_len, max_query_len)
    if opt:
        rc = lib.pa_prefix_ex(ctypes.byref(args), ctypes.byref(make_opts(**opt)), _stream_handle(stream))
    else:
        rc = lib.pa_prefix(args.out, args.q, args.k_new, args.v_new, args.k_cache, args.v_cache, args.block_tables,
                           args.context_lens, args.query_start_loc, args.num_seqs, args.num_tokens,
                           args.max_blocks_per_seq, args.max_context_len, args.max_query_len, args.num_blocks,
                           args.num_heads, args.num_kv_heads, args.head_dim, args.block_size, args.scale,
                           _stream_handle(stream))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_prefix")


def pa_prefix_split(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc, num_heads,
                    num_kv_heads, head_dim, block_size, scale, stream=None, *, max_context_len: int,
                    max_query_len: int, workspace: Optional[torch.Tensor] = None, parts: int = 0, units: int = 0,
                    **opt) -> None:
    """Chunked prefill with the last wave's query tiles split by key range
    (see include/pa_decode.h).  `workspace`: a CUDA uint8 tensor of at least
    prefix_split_workspace_size(...) bytes; None allocates one here (the
    call itself allocates nothing).  parts/units force a split (0: the
    library's plan)."""
    args = _prefix_args(out, q, k_new, v_new, k_cache, v_cache, block_tables, context_lens, query_start_loc,
                        num_heads, num_kv_heads, head_dim, block_size, scale, max_context_len, max_query_len)
    split = pa_prefix_split_opts(int(parts), int(units))
    if workspace is None:
        nbytes = ctypes.c_size_t(0)
        rc = lib.pa_prefix_split_workspace_size(ctypes.byref(args), ctypes.byref(split), ctypes.byref(nbytes))
        if rc != PA_OK:
            raise PaDecodeError(rc, "pa_prefix_split_workspace_size")
        workspace = torch.empty(max(int(nbytes.value), 1), dtype=torch.uint8, device=out.device)
    rc = lib.pa_prefix_split(ctypes.byref(args), ctypes.byref(make_opts(**opt)), ctypes.byref(split),
                             workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_prefix_split")


def prefix_split_workspace_size(w, parts: int = 0, units: int = 0) -> int:
    """Bytes of workspace pa_prefix_split needs for a workloads.PrefixWorkload."""
    out = torch.empty_like(w.q)
    args = _prefix_args(out, w.q, w.k_new, w.v_new, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                        w.query_start_loc, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale,
                        w.max_context_len, w.max_query_len)
    nbytes = ctypes.c_size_t(0)
    rc = lib.pa_prefix_split_workspace_size(ctypes.byref(args), ctypes.byref(pa_prefix_split_opts(parts, units)),
                                            ctypes.byref(nbytes))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_prefix_split_workspace_size")
    return int(nbytes.value)


def prefix_split_workload(w, out: Optional[torch.Tensor] = None, stream=None, **kw) -> torch.Tensor:
    """pa_prefix_split on a workloads.PrefixWorkload (tensors on the GPU)."""
    if out is None:
        out = torch.empty_like(w.q)
    pa_prefix_split(out, w.q, w.k_new, w.v_new, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                    w.query_start_loc, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale, stream,
                    max_context_len=w.max_context_len, max_query_len=w.max_query_len, **kw)
    return out


def prefix_workload(w, out: Optional[torch.Tensor] = None, stream=None, **opt) -> torch.Tensor:
    """Run chunked-prefill attention on a workloads.PrefixWorkload (tensors on the GPU)."""
    if out is None:
        out = torch.empty_like(w.q)
    pa_prefix(out, w.q, w.k_new, w.v_new, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
              w.query_start_loc, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.scale, stream,
              max_context_len=w.max_context_len, max_query_len=w.max_query_len, **opt)
    return out



def _check_partials(max_logits, exp_sums, tmp_out):
    for name, t in (("max_logits", max_logits), ("exp_sums", exp_sums), ("tmp_out", tmp_out)):
        if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA float32 tensor")


def pa_decode_partials(q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim, block_size,
                       scale, partition_size: int, partition_begin: int, partition_count: int, max_logits,
                       exp_sums, tmp_out, stream=None, *, max_seq_len: int, **opt) -> None:
    """Partials of partitions [partition_begin, partition_begin + partition_count)
    of every sequence (split-KV across devices, step 1): max_logits / exp_sums
    float32 [B, H, count] (max in base 2), tmp_out float32 [B, H, count, D]."""
    dummy = q  # `out` is not used by this call
    _check_tensors(dummy, q, k_cache, v_cache, block_tables, seq_lens)
    _check_partials(max_logits, exp_sums, tmp_out)
    args = make_args(None, q, k_cache, v_cache, block_tables, seq_lens, num_heads, num_kv_heads, head_dim,
                     block_size, scale, max_seq_len)
    rc = lib.pa_decode_partials(ctypes.byref(args), ctypes.byref(make_opts(**opt)), int(partition_size),
                                int(partition_begin), int(partition_count), max_logits.data_ptr(),
                                exp_sums.data_ptr(), tmp_out.data_ptr(), _stream_handle(stream))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_decode_partials")


def pa_merge_partials(out, max_logits, exp_sums, tmp_out, seq_lens, num_heads, head_dim, partition_size: int,
                      num_sources: int, partitions_per_source: int, stream=None, *, max_seq_len: int) -> None:
    """Log-sum-exp merge of partials gathered from `num_sources` sources
    (split-KV across devices, step 2): max_logits / exp_sums float32
    [R, B, H, pps], tmp_out float32 [R, B, H, pps, D]; out fp16 [B, H, D]."""
    _check_partials(max_logits, exp_sums, tmp_out)
    for name, t, dt in (("out", out, torch.float16), ("seq_lens", seq_lens, torch.int32)):
        if t.dtype != dt or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA {dt} tensor")
    rc = lib.pa_merge_partials(out.data_ptr(), max_logits.data_ptr(), exp_sums.data_ptr(), tmp_out.data_ptr(),
                               seq_lens.data_ptr(), int(seq_lens.shape[0]), int(num_heads), int(head_dim),
                               int(max_seq_len), int(partition_size), int(num_sources), int(partitions_per_source),
                               _stream_handle(stream))
    if rc != PA_OK:
        raise PaDecodeError(rc, "pa_merge_partials")
