"""pa_decode_noalloc: the decode call for callers that cannot allocate device
memory (a framework owning all memory through its own pool, a loop that cannot
pay an allocation's synchronisation).  It must give the same results as
pa_decode, and match the float64 oracle, call after call, while keeping its
partials in the library's fixed device scratch.  This file is named so that
pytest collects it last."""
import pytest
import torch

from paged_kv_cache_308_gb300 import binding as pb
from paged_kv_cache_308_gb300 import workloads as W
from parity_helpers import ATOL, RTOL, assert_parity, oracle_ref

pytestmark = pytest.mark.gpu


def _args(w, out):
    return (out, w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.num_heads, w.num_kv_heads, w.head_dim,
            w.block_size, w.scale)


def _noalloc(w):
    out = torch.full_like(w.q, float("nan"))
    pb.pa_decode_noalloc(*_args(w, out), max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    assert pb.pa_get_device_status() == 0
    assert torch.isfinite(out).all()
    return out


def _close(out, ref, what):
    diff = (out.float() - ref.float()).abs()
    bound = ATOL + RTOL * ref.float().abs()
    assert bool((diff <= bound).all()), f"{what}: max diff {diff.max().item()}"


@pytest.mark.parametrize("name", ["b1_l102400", "b8_u8192"])
def test_noalloc_matches_pa_decode_on_two_calls_in_a_row(name):
    assert torch.cuda.is_available()
    dev = torch.device("cuda:0")
    w = W.make_config(name, device=dev)
    plan = pb.pa_decode_plan(*_args(w, torch.empty_like(w.q)), max_seq_len=w.max_seq_len)
    assert plan["launch_reduce"] == 1 and 0 < plan["workspace_bytes"] <= 16 << 20  # the scratch is used

    ref = torch.empty_like(w.q)
    pb.pa_decode(*_args(w, ref), max_seq_len=w.max_seq_len)
    want = oracle_ref(w, 0)
    for call in range(2):
        out = _noalloc(w)
        _close(out, ref, f"call {call} against pa_decode")
        assert_parity(out, want, f"{name} no-alloc call {call}")


def test_noalloc_after_a_call_of_another_shape():
    # The one-long-sequence plan keeps its claim counters in the scratch, armed
    # by the previous call of that shape; a call of another shape in between
    # overwrites that slot with its own partials.  The next long call must
    # still be right (the counters are then read as not armed).
    dev = torch.device("cuda:0")
    long_w = W.make_config("b1_l102400", device=dev)
    batch_w = W.make_config("b8_u8192", device=dev)
    want_long, want_batch = oracle_ref(long_w, 0), oracle_ref(batch_w, 0)
    assert pb.pa_decode_plan(*_args(long_w, torch.empty_like(long_w.q)), max_seq_len=long_w.max_seq_len)["pooled"]
    assert_parity(_noalloc(long_w), want_long, "long, first")
    assert_parity(_noalloc(long_w), want_long, "long, counters armed")
    assert_parity(_noalloc(batch_w), want_batch, "batch in between")
    assert_parity(_noalloc(long_w), want_long, "long, after the batch")


def test_noalloc_rejects_calls_beyond_its_scratch():
    dev = torch.device("cuda:0")
    # 64 sequences of up to 65536 tokens: 64 x 24 x 128 partials of 1032 B = 203 MB > 16 MiB
    out = torch.empty((64, 24, 256), dtype=torch.float16, device=dev)
    q = torch.zeros_like(out)
    kc = torch.zeros((1, 4, 16, 256), dtype=torch.float16, device=dev)
    bt = torch.zeros((64, 4096), dtype=torch.int32, device=dev)
    sl = torch.zeros((64,), dtype=torch.int32, device=dev)
    with pytest.raises(pb.PaDecodeError) as e:
        pb.pa_decode_noalloc(out, q, kc, kc, bt, sl, 24, 4, 256, 16, 1 / 16, max_seq_len=65536)
    assert e.value.code == pb.PA_ERR_WORKSPACE
