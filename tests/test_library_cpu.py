"""The C-ABI library without a GPU: it loads, exports every declared function,
and its host logic (validation, dispatch plan, workspace sizing, status text)
answers without touching a device."""
import ctypes
import math

import pytest

from paged_kv_cache_308_gb300 import binding as pb

SMS = 152
FAKE = 0x10000  # a 16-byte aligned non-null address; the plan never dereferences it


def args(num_seqs=1, max_seq_len=102400, H=24, Hkv=4, D=256, bs=16, num_blocks=6400, mbps=None, scale=1 / 16,
         **ptrs):
    mbps = mbps if mbps is not None else (max_seq_len + bs - 1) // bs
    p = dict(out=FAKE, q=FAKE, k_cache=FAKE, v_cache=FAKE, block_tables=FAKE, seq_lens=FAKE)
    p.update(ptrs)
    return pb.pa_decode_args(p["out"], p["q"], p["k_cache"], p["v_cache"], p["block_tables"], p["seq_lens"],
                             num_seqs, mbps, max_seq_len, num_blocks, H, Hkv, D, bs, scale)


def plan(a, mode=0, partition_size=0):
    o = pb.pa_decode_opts(mode, partition_size, 0, 0, None, None)
    pl = pb.pa_decode_plan_t()
    rc = pb.lib.pa_decode_plan(ctypes.byref(a), ctypes.byref(o), SMS, ctypes.byref(pl))
    return rc, pl.as_dict()


def test_library_exports_every_declared_function():
    names = pb.header_functions()
    assert {"pa_decode", "pa_decode_ex", "pa_decode_plan", "pa_decode_workspace_size", "pa_get_device_status",
            "pa_status_string", "pa_release_workspace", "pa_version"} <= set(names)
    for n in names:
        assert hasattr(pb.lib, n), n


def test_status_strings():
    for code in (pb.PA_OK, pb.PA_ERR_INVALID_ARG, pb.PA_ERR_UNSUPPORTED, pb.PA_ERR_CUDA, pb.PA_ERR_OOM,
                 pb.PA_ERR_WORKSPACE):
        s = pb.status_string(code)
        assert s and s != "unknown status"
    assert pb.status_string(-99) == "unknown status"
    assert pb.version() >= 100


def ws_bytes(B, H, parts, D):
    a = lambda x: (x + 255) // 256 * 256
    return 2 * a(B * H * parts * 4) + a(B * H * parts * D * 4)


def test_plan_long_context_runs_one_wave_of_one_cta_per_sm():
    # one 102400-token sequence: 152 SMs / 4 kv heads = 38 partitions of
    # ceil(102400 / 38) = 2695 -> 2704 tokens, one 4-warp CTA per SM
    rc, pl = plan(args())
    assert rc == pb.PA_OK
    assert pl["mode"] == pb.PA_MODE_SPLIT and pl["partition_size"] == 2704
    assert (pl["grid_x"], pl["grid_y"], pl["grid_z"]) == (38, 4, 1)
    assert pl["threads"] == 128 and pl["stages"] == 2
    assert pl["grid_x"] * pl["grid_y"] <= SMS
    assert pl["launch_reduce"] == 1
    assert pl["pooled"] == 1  # + one 8-byte claim counter per kv head, in its own 256-byte slot
    assert pl["workspace_bytes"] == ws_bytes(1, 24, 38, 256) + 256
    assert pl["workspace_bytes"] <= pb.pa_decode_workspace_size(1, 102400, 24, 256, 0)
    # below 2048 tokens per partition the one wave has fixed partitions
    rc, short = plan(args(max_seq_len=65536, num_blocks=4096))
    assert rc == 0 and short["partition_size"] == 1728 and short["grid_x"] == 38 and short["pooled"] == 0
    # batches keep the 512-token default
    rc, batch = plan(args(num_seqs=2, num_blocks=12800))
    assert rc == 0 and batch["partition_size"] == 512 and batch["grid_x"] == 200
    # an explicit partition size or mode keeps the old plan
    rc, fixed = plan(args(), partition_size=512)
    assert rc == 0 and (fixed["grid_x"], fixed["grid_y"]) == (200, 4)
    assert (fixed["reduce_grid_x"], fixed["reduce_grid_y"], fixed["reduce_grid_z"]) == (24, 1, 8)
    assert fixed["workspace_bytes"] == ws_bytes(1, 24, 200, 256)
    assert fixed["workspace_bytes"] == pb.pa_decode_workspace_size(1, 102400, 24, 256, 512)
    # FUSED takes the same one-wave decomposition (its CTAs merge after a group barrier)
    rc, fused = plan(args(), mode=pb.PA_MODE_FUSED)
    assert rc == 0 and fused["partition_size"] == 2704 and fused["coop"] == 1


def test_plan_modes():
    rc, pl = plan(args(max_seq_len=2048, num_blocks=128), mode=pb.PA_MODE_SINGLE)
    assert rc == 0 and pl["mode"] == pb.PA_MODE_SINGLE and pl["grid_x"] == 1 and pl["partition_size"] == 2048
    assert pl["launch_reduce"] == 0 and pl["workspace_bytes"] == 0
    rc, pl = plan(args(max_seq_len=1000, num_blocks=128), mode=pb.PA_MODE_SINGLE)
    assert pl["partition_size"] == 1008                                   # rounded up to whole blocks
    rc, pl = plan(args(max_seq_len=128, num_blocks=128))
    assert rc == 0 and pl["mode"] == pb.PA_MODE_SINGLE                    # one copy round: no reduce
    rc, pl = plan(args(max_seq_len=512, num_blocks=128))
    assert rc == 0 and pl["mode"] == pb.PA_MODE_SPLIT and pl["partition_size"] == 16   # the one wave
    rc, pl = plan(args(max_seq_len=513, num_blocks=128), mode=pb.PA_MODE_SPLIT, partition_size=64)
    assert rc == 0 and pl["grid_x"] == math.ceil(513 / 64) and pl["launch_reduce"] == 1
    rc, pl = plan(args(num_seqs=0))
    assert rc == 0


def test_plan_halves_the_partition_when_the_grid_is_smaller_than_the_gpu():
    o = pb.pa_decode_opts(0, 0, 0, 0, None, None)
    pl = pb.pa_decode_plan_t()
    # two 8192-token sequences: 16 partitions x 4 kv heads x 2 = 128 CTAs < 152 SMs
    assert pb.lib.pa_decode_plan(ctypes.byref(args(num_seqs=2, max_seq_len=8192, num_blocks=1024)), ctypes.byref(o),
                                 152, ctypes.byref(pl)) == 0
    assert pl.partition_size == 256 and pl.grid_x == 32
    # 64 of them give 1024 CTAs at the default size, which stays
    a = args(num_seqs=64, max_seq_len=2048, num_blocks=64 * 128)
    assert pb.lib.pa_decode_plan(ctypes.byref(a), ctypes.byref(o), 152, ctypes.byref(pl)) == 0
    assert pl.partition_size == 512
    # an explicit partition size is kept
    o2 = pb.pa_decode_opts(0, 1024, 0, 0, None, None)
    assert pb.lib.pa_decode_plan(ctypes.byref(args(max_seq_len=2048, num_blocks=128)), ctypes.byref(o2), 152,
                                 ctypes.byref(pl)) == 0
    assert pl.partition_size == 1024


def test_plan_persistent_mode_has_a_fixed_grid_and_a_work_list():
    a = args(num_seqs=64, max_seq_len=65536, num_blocks=64 * 4096)
    rc, pl = plan(a, mode=pb.PA_MODE_PERSISTENT)
    _, split = plan(a, mode=pb.PA_MODE_SPLIT)
    assert rc == 0 and pl["mode"] == pb.PA_MODE_PERSISTENT
    # apportioned partitions: 4-warp CTAs, one per SM; at most SMs / kv heads partitions per sequence
    assert pl["threads"] == 128 and pl["stages"] == 2 and pl["grid_y"] == pl["grid_z"] == 1
    assert pl["grid_x"] == SMS and pl["partition_size"] == 0
    assert pl["max_partitions"] == SMS // 4 == 38 and pl["launch_reduce"] == 1
    # + the work list with the item counter (66 ints), the order and the partition sizes (64 ints each)
    assert pl["workspace_bytes"] == ws_bytes(64, 24, 38, 256) + 512 + 256 + 256
    # a caller's partition size: that size per sequence, balanced, on one-warp CTAs (6 per SM)
    rc, fixed = plan(a, mode=pb.PA_MODE_PERSISTENT, partition_size=512)
    assert rc == 0 and fixed["threads"] == 32 and fixed["grid_x"] == SMS * 6 and fixed["partition_size"] == 512
    assert fixed["max_partitions"] == split["grid_x"] == 128
    assert fixed["workspace_bytes"] == split["workspace_bytes"] + 512 + 256 + 256
    for w, s, per_sm in ((1, 2, 6), (2, 2, 2)):
        o = pb.make_opts(mode="persistent", warps=w, stages=s)
        p2 = pb.pa_decode_plan_t()
        assert pb.lib.pa_decode_plan(ctypes.byref(a), ctypes.byref(o), SMS, ctypes.byref(p2)) == 0
        assert (p2.threads, p2.stages, p2.grid_x) == (32 * w, s, SMS * per_sm)
    for w, s in ((3, 2), (4, 3)):
        o = pb.make_opts(mode="persistent", warps=w, stages=s)
        assert pb.lib.pa_decode_plan(ctypes.byref(a), ctypes.byref(o), SMS,
                                     ctypes.byref(pb.pa_decode_plan_t())) == pb.PA_ERR_UNSUPPORTED


def test_plan_fused_mode_keeps_partials_and_tickets_and_launches_once():
    a = args(max_seq_len=102400)
    rc, fused = plan(a, mode=pb.PA_MODE_FUSED, partition_size=512)
    _, split = plan(a, mode=pb.PA_MODE_SPLIT, partition_size=512)
    assert rc == 0 and fused["mode"] == pb.PA_MODE_FUSED and fused["launch_reduce"] == 0
    assert fused["grid_x"] == split["grid_x"] == 200 and fused["partition_size"] == 512
    # the split partials, a slot the size of the pooled claim counters (8 bytes per
    # (sequence, kv head)), then two 4-byte group words per (sequence, kv head), each 256-byte aligned
    assert fused["workspace_bytes"] == split["workspace_bytes"] + 256 + 256
    rc, one = plan(args(max_seq_len=128, num_blocks=128), mode=pb.PA_MODE_FUSED)
    assert rc == 0 and one["grid_x"] == 1 and one["workspace_bytes"] == 0   # one partition: written directly


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), pb.PA_ERR_INVALID_ARG),
    (dict(out=FAKE + 2), pb.PA_ERR_INVALID_ARG),
    (dict(k_cache=FAKE + 8), pb.PA_ERR_INVALID_ARG),
    (dict(block_tables=FAKE + 2), pb.PA_ERR_INVALID_ARG),
    (dict(H=24, Hkv=5), pb.PA_ERR_INVALID_ARG),
    (dict(D=100), pb.PA_ERR_UNSUPPORTED),
    (dict(D=96), pb.PA_ERR_UNSUPPORTED),
    (dict(bs=32), pb.PA_ERR_UNSUPPORTED),
    (dict(H=48, Hkv=4), pb.PA_ERR_UNSUPPORTED),     # GQA ratio 12 > 8
    (dict(scale=float("nan")), pb.PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), pb.PA_ERR_INVALID_ARG),
    (dict(mbps=10), pb.PA_ERR_INVALID_ARG),         # max_seq_len beyond the block table
    (dict(num_seqs=-1), pb.PA_ERR_INVALID_ARG),
    (dict(num_seqs=70000), pb.PA_ERR_INVALID_ARG),
    (dict(num_blocks=0), pb.PA_ERR_INVALID_ARG),
    (dict(num_blocks=1 << 26), pb.PA_ERR_UNSUPPORTED),  # rows past 32-bit TMA coordinates
])
def test_plan_rejects_bad_arguments(kw, code):
    rc, _ = plan(args(**kw))
    assert rc == code


def test_plan_rejects_bad_options():
    assert plan(args(), mode=7)[0] == pb.PA_ERR_INVALID_ARG
    assert plan(args(), partition_size=100)[0] == pb.PA_ERR_INVALID_ARG   # not a multiple of 16
    assert plan(args(), partition_size=-16)[0] == pb.PA_ERR_INVALID_ARG


@pytest.mark.parametrize("G", [1, 2, 3, 6, 8])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_plan_accepts_supported_shapes(G, D):
    rc, pl = plan(args(H=4 * G, Hkv=4, D=D))
    assert rc == 0 and pl["threads"] % 32 == 0 and 0 < pl["smem_bytes"] <= 227 * 1024


def test_decode_ex_checks_workspace_before_any_cuda_call():
    a = args()
    o = pb.pa_decode_opts(0, 0, 0, 0, None, None)
    rc = pb.lib.pa_decode_ex(ctypes.byref(a), ctypes.byref(o), None, 0, None)
    assert rc == pb.PA_ERR_WORKSPACE
    rc = pb.lib.pa_decode_ex(ctypes.byref(a), ctypes.byref(o), FAKE + 64, 1 << 30, None)  # misaligned
    assert rc == pb.PA_ERR_WORKSPACE


def test_calls_fail_cleanly_without_a_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    a = args(max_seq_len=256, num_blocks=16)
    o = pb.pa_decode_opts(pb.PA_MODE_SINGLE, 0, 0, 0, None, None)
    assert pb.lib.pa_decode_ex(ctypes.byref(a), ctypes.byref(o), None, 0, None) == pb.PA_ERR_CUDA
    st = ctypes.c_int(0)
    assert pb.lib.pa_get_device_status(None, ctypes.byref(st)) == pb.PA_ERR_CUDA
    pb.pa_release_workspace()  # nothing allocated: a no-op


@pytest.mark.parametrize("B,L,z", [(1, 102400, 8), (4, 32768, 4), (8, 8192, 2), (64, 65536, 1), (16, 4096, 1),
                                   (2, 65536, 8)])
def test_reduce_slice_follows_the_batch(B, L, z):
    # the widest head_dim slice that still gives >= 2 reduce CTAs per SM
    rc, pl = plan(args(num_seqs=B, max_seq_len=L, num_blocks=B * L // 16))
    assert rc == 0 and pl["launch_reduce"] == 1
    assert pl["reduce_grid_z"] == z and (pl["reduce_grid_x"], pl["reduce_grid_y"]) == (24, B)


def test_cta_shape_option():
    a = args()
    for w, s in ((2, 2), (1, 2), (1, 3), (4, 2)):
        o = pb.make_opts(warps=w, stages=s)
        pl = pb.pa_decode_plan_t()
        assert pb.lib.pa_decode_plan(ctypes.byref(a), ctypes.byref(o), SMS, ctypes.byref(pl)) == pb.PA_OK
        assert (pl.threads, pl.stages) == (32 * w, s)
        # one stage holds the K and V of a 16-token block: 2 x 16 x 256 x 2 B
        assert pl.smem_bytes >= w * s * 16384
    for w, s in ((3, 2), (2, 5), (0, 2)):
        o = pb.make_opts(warps=w, stages=s)
        pl = pb.pa_decode_plan_t()
        assert pb.lib.pa_decode_plan(ctypes.byref(a), ctypes.byref(o), SMS, ctypes.byref(pl)) == pb.PA_ERR_UNSUPPORTED


@pytest.mark.parametrize("B,L,shape", [
    (1, 2048, (4, 2)),       # 16 CTAs: the most bytes in flight per CTA
    (8, 8192, (2, 2)),       # ~256 CTAs: one wave of 2-warp CTAs
    (4, 32768, (1, 3)),      # ~512-1024 CTAs: two waves of 4 CTAs/SM
    (1, 102400, (1, 2)),     # 800 CTAs: one wave at 6 CTAs/SM
    (64, 65536, (1, 2)),     # many waves: the finest slots
])
def test_cta_shape_follows_the_wave_model(B, L, shape):
    # at the 512-token partitions the model was fitted for
    rc, pl = plan(args(num_seqs=B, max_seq_len=L, num_blocks=B * L // 16), partition_size=512 if L > 2048 else 0)
    assert rc == 0 and (pl["threads"] // 32, pl["stages"]) == shape


def _plan_opts(num_seqs, max_seq_len, mode=0, partition_size=0, flags=0, warps=0, stages=0):
    o = pb.pa_decode_opts(mode, partition_size, flags, 0, None, None, warps, stages)
    pl = pb.pa_decode_plan_t()
    rc = pb.lib.pa_decode_plan(ctypes.byref(args(num_seqs=num_seqs, max_seq_len=max_seq_len,
                                                 num_blocks=num_seqs * ((max_seq_len + 15) // 16))),
                               ctypes.byref(o), SMS, ctypes.byref(pl))
    assert rc == 0
    return pl.as_dict()


def test_pooled_plan_flags_and_workspace():
    base = _plan_opts(1, 102400, flags=pb.PA_FLAG_DETERMINISTIC)
    pooled = _plan_opts(1, 102400, flags=pb.PA_FLAG_POOLED)
    assert base["pooled"] == 0 and pooled["pooled"] == 1
    # the one-wave plan of one long sequence is pooled by default; DETERMINISTIC wins over POOLED
    assert _plan_opts(1, 102400) == pooled
    assert _plan_opts(1, 102400, flags=pb.PA_FLAG_POOLED | pb.PA_FLAG_DETERMINISTIC) == base
    assert _plan_opts(4, 32768)["pooled"] == 0  # several waves: fixed
    # same grid and partials as the fixed split, plus one 8-byte counter per (sequence, kv head)
    for k in ("mode", "partition_size", "grid_x", "grid_y", "grid_z", "threads", "max_partitions"):
        assert pooled[k] == base[k]
    assert pooled["workspace_bytes"] == base["workspace_bytes"] + 256
    # pooled only for SPLIT plans with at least one chunk (max(2, stages) blocks) per warp of every partition
    assert _plan_opts(4, 4096, mode=2, partition_size=112, flags=pb.PA_FLAG_POOLED, warps=4, stages=2)["pooled"] == 0
    assert _plan_opts(4, 4096, mode=2, partition_size=128, flags=pb.PA_FLAG_POOLED, warps=4, stages=2)["pooled"] == 1
    assert _plan_opts(4, 4096, mode=2, partition_size=32, flags=pb.PA_FLAG_POOLED, warps=1, stages=3)["pooled"] == 0
    assert _plan_opts(4, 4096, mode=2, partition_size=48, flags=pb.PA_FLAG_POOLED, warps=1, stages=3)["pooled"] == 1
    assert _plan_opts(4, 500, flags=pb.PA_FLAG_POOLED)["pooled"] == 0  # one partition: no reduce
    for mode in (1, 3, 4):
        assert _plan_opts(4, 4096, mode=mode, flags=pb.PA_FLAG_POOLED)["pooled"] == 0


@pytest.mark.parametrize("B,L", [(1, 2048), (1, 30000), (1, 77824), (1, 102400), (1, 1 << 20), (8, 8192), (64, 65536)])
def test_workspace_size_bounds_every_automatic_plan(B, L):
    # pa_decode_workspace_size(..., 0) is documented as an upper bound for the
    # automatic partition size, pooled counters included
    pl = _plan_opts(B, L)
    assert pb.pa_decode_workspace_size(B, L, 24, 256, 0) >= pl["workspace_bytes"]


def _plan_heads(num_kv_heads, max_seq_len, flags=0, num_heads=None):
    H = num_heads or 6 * num_kv_heads
    o = pb.pa_decode_opts(0, 0, flags, 0, None, None, 0, 0)
    pl = pb.pa_decode_plan_t()
    a = args(num_seqs=1, max_seq_len=max_seq_len, H=H, Hkv=num_kv_heads,
             num_blocks=(max_seq_len + 15) // 16)
    assert pb.lib.pa_decode_plan(ctypes.byref(a), ctypes.byref(o), SMS, ctypes.byref(pl)) == 0
    return pl.as_dict()


@pytest.mark.parametrize("hkv", [1, 2, 4, 8])
@pytest.mark.parametrize("L", [102400, 262144, 1 << 20])
def test_one_wave_pooled_plan_for_every_kv_head_count(hkv, L):
    pl = _plan_heads(hkv, L)
    per_head = SMS // hkv
    # one 4-warp CTA per SM at most, partitions of whole blocks covering the sequence,
    # pooled from 2048-token partitions on
    assert pl["threads"] == 128 and pl["stages"] == 2
    assert pl["grid_x"] * pl["grid_y"] <= SMS and pl["grid_y"] == hkv
    assert pl["partition_size"] % 16 == 0 and pl["partition_size"] * pl["grid_x"] >= L
    if -(-L // per_head) < 2048:
        assert pl["pooled"] == 0
        return
    assert pl["pooled"] == 1
    fixed = _plan_heads(hkv, L, flags=pb.PA_FLAG_DETERMINISTIC)
    assert fixed["pooled"] == 0 and fixed["grid_x"] == pl["grid_x"] and fixed["partition_size"] == pl["partition_size"]
    assert fixed["workspace_bytes"] + 256 == pl["workspace_bytes"]


def _partials(a, P, begin, count, m=FAKE, l=FAKE, acc=FAKE, mode=0):
    o = pb.pa_decode_opts(mode, 0, 0, 0, None, None)
    return pb.lib.pa_decode_partials(ctypes.byref(a), ctypes.byref(o), P, begin, count, m, l, acc, None)


def test_partials_and_merge_check_their_arguments_before_any_cuda_call():
    a = args(max_seq_len=102400, out=None)  # the output is not used by the partials call
    for P, begin, count in ((500, 0, 4), (0, 0, 4), (512, -1, 4), (512, 0, 0), (1 << 20, 4096, 4)):
        assert _partials(a, P, begin, count) == pb.PA_ERR_INVALID_ARG, (P, begin, count)
    assert _partials(a, 512, 0, 100, mode=pb.PA_MODE_FUSED) == pb.PA_ERR_INVALID_ARG
    assert _partials(a, 512, 0, 100, m=None) == pb.PA_ERR_INVALID_ARG
    assert _partials(a, 512, 0, 100, acc=FAKE + 4) == pb.PA_ERR_INVALID_ARG  # tmp_out not 16-byte aligned
    assert _partials(args(D=96, out=None), 512, 0, 100) == pb.PA_ERR_UNSUPPORTED

    def merge(num_seqs=1, H=24, D=256, max_seq_len=102400, P=512, R=2, pps=100, out=FAKE, acc=FAKE):
        return pb.lib.pa_merge_partials(out, FAKE, FAKE, acc, FAKE, num_seqs, H, D, max_seq_len, P, R, pps, None)

    assert merge(pps=99) == pb.PA_ERR_INVALID_ARG          # 2 x 99 partitions of 512 miss the last tokens
    assert merge(P=500) == pb.PA_ERR_INVALID_ARG
    assert merge(R=0) == pb.PA_ERR_INVALID_ARG
    assert merge(D=96) == pb.PA_ERR_UNSUPPORTED
    assert merge(out=None) == pb.PA_ERR_INVALID_ARG
    assert merge(acc=FAKE + 8) == pb.PA_ERR_INVALID_ARG
    assert merge(num_seqs=0, out=None) == pb.PA_OK              # nothing to do


def test_partials_and_merge_fail_cleanly_without_a_device():
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _partials(args(max_seq_len=102400, out=None), 512, 0, 100) == pb.PA_ERR_CUDA
    assert pb.lib.pa_merge_partials(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 24, 256, 102400, 512, 2, 100,
                                    None) == pb.PA_ERR_CUDA


def test_plan_flat_mode_one_cta_per_sm_and_its_workspace():
    a = args(num_seqs=8, max_seq_len=8192, num_blocks=8192)
    rc, fl = plan(a, mode=pb.PA_MODE_FLAT)
    assert rc == 0 and fl["mode"] == pb.PA_MODE_FLAT and fl["launch_reduce"] == 1
    assert (fl["grid_x"], fl["grid_y"], fl["grid_z"], fl["threads"]) == (152, 1, 1, 128)
    assert fl["max_partitions"] == 38 and fl["partition_size"] == 0
    rows = 8 * 24 * 38
    part = 2 * ((rows * 4 + 255) // 256 * 256) + (rows * 256 * 4 + 255) // 256 * 256
    assert fl["workspace_bytes"] == part + 256  # + one partial count per sequence
    rc, one = plan(args(num_seqs=3, max_seq_len=4096, Hkv=4, num_blocks=2000), mode=pb.PA_MODE_FLAT)
    assert rc == 0 and one["grid_x"] == 152
    # at most 256 sequences: the lengths and prefix sums live in each CTA's shared memory
    assert plan(args(num_seqs=256, max_seq_len=64, num_blocks=2000), mode=pb.PA_MODE_FLAT)[0] == 0
    assert plan(args(num_seqs=257, max_seq_len=64, num_blocks=2000), mode=pb.PA_MODE_FLAT)[0] == pb.PA_ERR_UNSUPPORTED
    # 8 kv heads: 19 CTAs each; one kv head: 152
    assert plan(args(num_seqs=2, H=32, Hkv=8), mode=pb.PA_MODE_FLAT)[1]["max_partitions"] == 19
    assert plan(args(num_seqs=2, H=8, Hkv=1), mode=pb.PA_MODE_FLAT)[1]["max_partitions"] == 152


def test_plan_fused_merges_in_parallel_on_a_grid_the_device_holds():
    # one long sequence: the one-wave plan (one 4-warp CTA per SM), pooled, cooperative
    rc, fw = plan(args(max_seq_len=102400), mode=pb.PA_MODE_FUSED)
    assert rc == 0 and fw["coop"] == 1 and fw["pooled"] == 1 and fw["launch_reduce"] == 0
    assert (fw["grid_x"], fw["grid_y"], fw["threads"]) == (38, 4, 128)
    o = pb.pa_decode_opts(pb.PA_MODE_FUSED, 0, pb.PA_FLAG_DETERMINISTIC, 0, None, None)
    pl = pb.pa_decode_plan_t()
    assert pb.lib.pa_decode_plan(ctypes.byref(args(max_seq_len=102400)), ctypes.byref(o), SMS, ctypes.byref(pl)) == 0
    assert pl.coop == 1 and pl.pooled == 0
    # 6400 partitions of 16 tokens x 4 kv heads: more CTAs than the SMs hold, so the last CTA merges
    rc, big = plan(args(max_seq_len=102400), mode=pb.PA_MODE_FUSED, partition_size=16)
    assert rc == 0 and big["coop"] == 0 and big["pooled"] == 0
    # the split and the other modes never take the cooperative form
    for mode in (pb.PA_MODE_SPLIT, pb.PA_MODE_SINGLE, pb.PA_MODE_PERSISTENT, pb.PA_MODE_FLAT, pb.PA_MODE_AUTO):
        assert plan(args(max_seq_len=102400), mode=mode)[1]["coop"] == 0


def prefix_args(B=4, ctx=8192, ql=512, H=24, Hkv=4, D=256):
    mbps = (ctx + 15) // 16
    return pb.pa_prefix_args(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, B * ql, mbps, ctx, ql,
                             B * mbps, H, Hkv, D, 16, 1 / 16)


def split_size(a, parts, units):
    n = ctypes.c_size_t(123)
    rc = pb.lib.pa_prefix_split_workspace_size(ctypes.byref(a), ctypes.byref(pb.pa_prefix_split_opts(parts, units)),
                                               ctypes.byref(n))
    return rc, n.value


def test_prefix_split_workspace_size_of_a_forced_split():
    # rows of 128 (the MMA M) per part: O in fp32, then (m, l), each 256-byte aligned
    a = prefix_args()
    r = lambda x: (x + 255) // 256 * 256
    for parts, units in ((3, 96), (1, 1), (64, 400), (2, 7)):
        rc, n = split_size(a, parts, units)
        assert rc == pb.PA_OK
        rows = parts * units * 128
        assert n == r(rows * 256 * 4) + r(rows * 2 * 4), (parts, units)
    assert split_size(a, 5, 0) == (pb.PA_OK, 0)  # nothing split


@pytest.mark.parametrize("parts,units", [(65, 1), (-1, 1), (2, 401), (2, -1)])
def test_prefix_split_rejects_a_split_out_of_range(parts, units):
    # 25 query tiles x 4 kv heads x 4 sequences = 400 units
    rc, n = split_size(prefix_args(), parts, units)
    assert rc == pb.PA_ERR_INVALID_ARG and n == 0


def test_prefix_split_fails_cleanly_without_a_device():
    a = prefix_args()
    # the library's own plan needs the SM count: no device, an error, no crash
    assert split_size(a, 0, 0)[0] == pb.PA_ERR_CUDA
    o = pb.make_opts()
    sp = pb.pa_prefix_split_opts(3, 96)
    # a forced split checks its workspace before any CUDA call
    rc = pb.lib.pa_prefix_split(ctypes.byref(a), ctypes.byref(o), ctypes.byref(sp), None, 0, None)
    assert rc == pb.PA_ERR_INVALID_ARG
    rc = pb.lib.pa_prefix_split(ctypes.byref(a), ctypes.byref(o), ctypes.byref(sp), FAKE + 16, 1 << 30, None)
    assert rc == pb.PA_ERR_INVALID_ARG  # misaligned


def plan_flags(a, flags, partition_size=0, warps=0, stages=0, mode=0):
    o = pb.pa_decode_opts(mode, partition_size, flags, 0, None, None, warps, stages)
    pl = pb.pa_decode_plan_t()
    rc = pb.lib.pa_decode_plan(ctypes.byref(a), ctypes.byref(o), SMS, ctypes.byref(pl))
    return rc, pl.as_dict()


@pytest.mark.parametrize("B,L,per_seq,P", [(4, 32768, 9, 3648), (4, 4096, 9, 464), (2, 65536, 19, 3456),
                                           (16, 16384, 2, 8192), (8, 8192, 4, 2048)])
def test_uniform_lengths_flag_gives_a_batch_the_one_wave_plan(B, L, per_seq, P):
    # floor(152 / (4 kv heads x B)) partitions per sequence of ceil(L / that)
    # tokens, rounded up to whole blocks; one 4-warp CTA per SM; fixed partitions
    a = args(num_seqs=B, max_seq_len=L, num_blocks=B * L // 16)
    rc, pl = plan_flags(a, pb.PA_FLAG_UNIFORM_LENGTHS)
    assert rc == pb.PA_OK
    assert pl["partition_size"] == P and (pl["grid_x"], pl["grid_y"], pl["grid_z"]) == (per_seq, 4, B)
    assert pl["threads"] == 128 and pl["stages"] == 2 and pl["pooled"] == 0 and pl["launch_reduce"] == 1
    assert pl["grid_x"] * pl["grid_y"] * pl["grid_z"] <= SMS
    # without the statement a batch keeps the 512-token grid
    rc, pl = plan_flags(a, 0)
    assert pl["partition_size"] in (256, 512)


def test_uniform_lengths_flag_leaves_other_plans_alone():
    # too many sequences for two partitions each (152 // (4 x 32) = 1): the grid
    rc, pl = plan_flags(args(num_seqs=32, max_seq_len=4096, num_blocks=8192), pb.PA_FLAG_UNIFORM_LENGTHS)
    assert rc == pb.PA_OK and pl["partition_size"] == 512 and pl["grid_x"] == 8
    # a caller's partition size or CTA shape wins over the flag
    a = args(num_seqs=4, max_seq_len=32768, num_blocks=8192)
    assert plan_flags(a, pb.PA_FLAG_UNIFORM_LENGTHS, partition_size=1024)[1]["partition_size"] == 1024
    rc, pl = plan_flags(a, pb.PA_FLAG_UNIFORM_LENGTHS, warps=2, stages=2)
    assert pl["partition_size"] == 512 and pl["threads"] == 64
    # one sequence: the flag changes nothing (the one-wave rule already holds, pooled)
    one = args()
    assert plan_flags(one, pb.PA_FLAG_UNIFORM_LENGTHS)[1] == plan_flags(one, 0)[1]
    # with PA_FLAG_POOLED the batch's one wave is pooled
    rc, pl = plan_flags(a, pb.PA_FLAG_UNIFORM_LENGTHS | pb.PA_FLAG_POOLED)
    assert pl["pooled"] == 1 and pl["partition_size"] == 3648


@pytest.mark.parametrize("B,L,P,parts", [(1, 2048, 64, 32), (1, 4096, 112, 37), (1, 513, 16, 33), (1, 3000, 80, 38),
                                          (1, 129, 16, 9), (1, 512, 16, 32), (4, 300, 48, 7), (8, 400, 112, 4),
                                          (1, 4864, 128, 38), (1, 8192, 224, 37), (1, 16384, 432, 38),
                                          (2, 2048, 112, 19), (4, 1024, 128, 8), (3, 1500, 128, 12)])
def test_short_sequence_runs_one_wave_of_one_block_deep_ctas(B, L, P, parts):
    # one sequence over 512 tokens, or a batch whose one-wave partitions hold
    # at most 128 tokens (one round of copies for a 4-warp CTA):
    # floor(152 / (4 B)) partitions of ceil(L / that) tokens rounded up to
    # whole blocks, one 4-warp CTA per SM, fixed partitions
    rc, pl = plan_flags(args(num_seqs=B, max_seq_len=L, num_blocks=B * ((L + 15) // 16)), 0)
    assert rc == pb.PA_OK
    assert pl["partition_size"] == P and (pl["grid_x"], pl["grid_y"], pl["grid_z"]) == (parts, 4, B)
    assert pl["threads"] == 128 and pl["stages"] == 2 and pl["pooled"] == 0 and pl["launch_reduce"] == 1
    assert pb.pa_decode_workspace_size(B, L, 24, 256, 0) >= pl["workspace_bytes"]
    # in a batch, longer partitions keep the grid (two 5000-token sequences)
    rc, pl = plan_flags(args(num_seqs=2, max_seq_len=5000, num_blocks=626), 0)
    assert pl["partition_size"] == 256
    # 128 tokens or fewer: one partition, no reduce
    rc, pl = plan_flags(args(max_seq_len=128, num_blocks=8), 0)
    assert pl["launch_reduce"] == 0 and pl["grid_x"] == 1


@pytest.mark.parametrize("B,L", [(16, 200), (8, 256), (12, 300), (16, 129), (64, 512)])
def test_larger_short_batches_keep_single_pass(B, L):
    # fewer than 4 one-wave partitions per sequence, or sequences of at most
    # 256 tokens: SINGLE (no reduce) measured faster than a one-wave split
    rc, pl = plan_flags(args(num_seqs=B, max_seq_len=L, num_blocks=B * ((L + 15) // 16)), 0)
    assert rc == pb.PA_OK and pl["mode"] == pb.PA_MODE_SINGLE and pl["launch_reduce"] == 0


@pytest.mark.parametrize("H,Hkv,D,L,per_seq,P,pooled", [(32, 8, 128, 102400, 38, 2704, 1), (32, 4, 64, 131072, 152, 864, 0),
                                                         (16, 2, 256, 102400, 76, 1360, 0), (8, 8, 128, 65536, 38, 1728, 0)])
def test_one_wave_keeps_copies_in_flight_at_every_head_dim(H, Hkv, D, L, per_seq, P, pooled):
    # 256 / head_dim 4-warp CTAs per SM (1 at 256, 2 at 128, 4 at 64): about
    # 128 KB of K/V copies in flight per SM whatever the head_dim
    a = args(max_seq_len=L, H=H, Hkv=Hkv, D=D, num_blocks=(L + 15) // 16)
    rc, pl = plan_flags(a, 0)
    assert rc == pb.PA_OK
    assert (pl["grid_x"], pl["grid_y"]) == (per_seq, Hkv) and pl["partition_size"] == P and pl["pooled"] == pooled
    assert pl["grid_x"] * pl["grid_y"] == SMS * (256 // D) or pl["grid_x"] * P >= L
    assert pb.pa_decode_workspace_size(1, L, H, D, 0) >= pl["workspace_bytes"]


def test_workspace_bound_covers_every_automatic_plan_property():
    # pa_decode_workspace_size(..., 0) is documented as an upper bound for any
    # automatic plan (one-wave plans, PA_FLAG_UNIFORM_LENGTHS and the pooled
    # counters included): random shapes, AUTO and SPLIT, with and without flags
    import random
    r = random.Random(11)
    for _ in range(3000):
        hkv = r.choice([1, 2, 4, 8])
        H = hkv * r.choice([1, 2, 3, 4, 6, 8])
        D = r.choice([64, 128, 256])
        B = r.choice([1, 1, 2, 3, 4, 8, 16, 64, 300])
        L = r.choice([1, 16, 100, 129, 257, 512, 513, 2048, 4864, 8192, 30000, 102400, 524288, r.randint(1, 200000)])
        flags = r.choice([0, pb.PA_FLAG_UNIFORM_LENGTHS, pb.PA_FLAG_POOLED, pb.PA_FLAG_DETERMINISTIC])
        mode = r.choice([0, pb.PA_MODE_SPLIT])
        a = args(num_seqs=B, max_seq_len=L, H=H, Hkv=hkv, D=D, num_blocks=max(1, min(B * ((L + 15) // 16), (1 << 31) // (hkv * 16) - 1)))
        rc, pl = plan_flags(a, flags, mode=mode)
        if rc != pb.PA_OK:
            continue
        assert pb.pa_decode_workspace_size(B, L, H, D, 0) >= pl["workspace_bytes"], (B, L, H, hkv, D, flags, mode, pl)


def test_many_short_pairs_take_2x2_ctas():
    # at least 64 (sequence, kv head) pairs of at most 16K tokens in 512-token
    # partitions, head_dim >= 128: 2x2 CTAs; the named batches keep their shapes
    def shape(B, L, Hkv=4, H=24, D=256, **kw):
        rc, pl = plan(args(num_seqs=B, max_seq_len=L, num_blocks=B * L // 16 + 10, Hkv=Hkv, H=H, D=D), **kw)
        assert rc == 0
        return pl["partition_size"], (pl["threads"] // 32, pl["stages"])
    assert shape(32, 4096) == (512, (2, 2))
    assert shape(16, 16384) == (512, (2, 2))
    assert shape(100, 1500) == (512, (2, 2))
    assert shape(8, 8192, Hkv=8, H=32, D=128) == (512, (2, 2))
    # below the pair count, above the length, or a caller's partition size: the wave model's choice
    assert shape(15, 8192) == (512, (1, 3))
    assert shape(16, 16385) == (512, (1, 3))
    assert shape(32, 4096, mode=pb.PA_MODE_SPLIT, partition_size=256) == (256, (1, 3))
    assert shape(4, 32768) == (512, (1, 3))      # b4_l32768_peaked
    assert shape(64, 32768) == (512, (1, 2))     # b64_loguniform
    assert shape(8, 8192) == (512, (2, 2))       # b8_u8192 (the wave model's pick)


def test_prefix_refuses_a_unit_count_past_32_bits():
    # 200 query tiles of 128 tokens x 256 kv heads x 65535 sequences: 3.4e9 units,
    # refused before any CUDA call
    a = pb.pa_prefix_args(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 65535, 65535 * 25600, 0, 0, 25600,
                          0, 256, 256, 128, 16, 1 / 16)
    assert pb.lib.pa_prefix_ex(ctypes.byref(a), None, None) == pb.PA_ERR_UNSUPPORTED
    n = ctypes.c_size_t(7)
    assert pb.lib.pa_prefix_split_workspace_size(ctypes.byref(a), None, ctypes.byref(n)) == pb.PA_ERR_UNSUPPORTED
    # one sequence fewer tiles: accepted up to the device (none here)
    b = prefix_args()
    assert pb.lib.pa_prefix_split_workspace_size(ctypes.byref(b), ctypes.byref(pb.pa_prefix_split_opts(3, 96)),
                                                 ctypes.byref(n)) == pb.PA_OK


def test_binding_constants_match_the_header():
    # every PA_MODE_*, PA_FLAG_*, PA_ERR_* and PA_DEV_* enumerator of the header
    # exists in the binding with the same value
    import re
    text = re.sub(r"/\*.*?\*/", "", open(pb.HEADER_PATH).read(), flags=re.S)
    consts = {k: int(v) for k, v in re.findall(r"\b(PA_(?:MODE|FLAG|ERR|DEV)_[A-Z0-9_]+)\s*=\s*(-?\d+)", text)}
    assert {"PA_FLAG_PREFIX_GRID", "PA_FLAG_UNIFORM_LENGTHS", "PA_MODE_FLAT", "PA_DEV_TIMEOUT"} <= set(consts)
    for k, v in consts.items():
        assert getattr(pb, k) == v, k
