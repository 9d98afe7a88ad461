"""Host side of bench.py's multi-GPU path (replicas only: the path shards by
request or channel with no exchange step, so N GPUs run N independent copies of
the step and the only collectives are a barrier and a max over ranks of the
timed region). Run as world_size-2 gloo process groups on the CPU."""
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


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_env()
        elapsed = [0.25, 0.5][rank]                   # rank 1 is the slow one
        dist.barrier()
        slowest = bench.reduce_max(elapsed, ws)
        value = bench.whole_job_value(ws, 1_000_000, 10, slowest)
        # replicas draw the same seeded inputs: their checksums agree
        from state_cached_causal_gb300 import synth
        case = synth.single_prefill(torch.device("cpu"))
        cs = torch.tensor([float(case.x.double().sum())], dtype=torch.float64)
        allcs = [torch.zeros(1, dtype=torch.float64) for _ in range(ws)]
        dist.all_gather(allcs, cs)
        q.put((rank, got_ws, got_rank, got_local, slowest, value,
               [float(t.item()) for t in allcs]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got_ws, got_rank, got_local, slowest, value, allcs in res:
        assert (got_ws, got_rank, got_local) == (2, rank, rank)
        assert slowest == 0.5                          # max over ranks
        assert value == pytest.approx(2 * 1_000_000 * 10 / 0.5 / 1e9)
        assert allcs[0] == allcs[1]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class A:
        gpus, steps, warmup = 2, 1, 0
    assert bench.arm_reference(A()) == 0
    assert capsys.readouterr().out == ""


def test_single_process_needs_no_collective():
    assert bench.reduce_max(0.125, 1) == 0.125
    assert bench.whole_job_value(1, 2_000_000_000, 5, 10.0) == pytest.approx(1.0)
