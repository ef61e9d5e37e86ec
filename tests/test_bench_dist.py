"""Host-side multi-rank logic of bench.py on CPU (gloo, world size 2): the
timed region's max over ranks and the whole-job aggregate of replicas, and
the reference arm's rank handling."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 0.5 + rank          # rank 1 is the slow one
        m = bench.max_over_ranks(local, dist, torch.device("cpu"))
        dist.barrier()
        q.put((rank, m, bench.aggregate_gbs(4096, 10, world, m)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, m, gbs in got:
        assert m == 1.5                               # every rank sees the slowest rank's time
        assert gbs == pytest.approx(2 * 4096 * 10 / 1.5 / 1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = bench.argparse.Namespace(gpus=2, steps=1, warmup=0, workload="b1_l2048", seed=0)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
