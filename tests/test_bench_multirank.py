"""bench.py's multi-GPU bookkeeping on CPU: N independent replicas, the job's
time is the slowest rank's (max over ranks through torch.distributed), the
value is the aggregate over ranks, and only rank 0 prints.  Two gloo ranks on
127.0.0.1 stand in for two GPUs."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(dist, 1.0 + rank * 0.5, "cpu")  # rank 1 is slower
        out.put((rank, ms, bench.aggregate_gbs(world, 2e9, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, gbs in got:
        assert ms == pytest.approx(1.5)       # the slowest rank's time
        assert gbs == pytest.approx(2 * 2e9 / 1.5e-3 / 1e9)  # both ranks' bytes


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(None, 3.0, "cpu") == 3.0
    assert bench.aggregate_gbs(1, 1e9, 1.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None) == 0  # returns before reading any argument
    assert capsys.readouterr().out == ""
