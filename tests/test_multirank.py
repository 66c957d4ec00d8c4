"""The benchmark's multi-rank path on the CPU: world-size-2 gloo process
groups stand in for the GPU ranks (the layer itself has no cross-rank step:
N GPUs run N replicas, so what needs checking is the host logic - the job
time is the slowest rank's, the throughput counts every rank's tokens, only
rank 0 reports, and the reference arm runs on rank 0 alone)."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup()
        ms = bench.slowest_rank_ms(10.0 + 5.0 * rank, w)  # rank 1 is the slow one
        dist.barrier()
        out[rank] = (w, r, local, ms, bench.job_tokens_per_s(w, 4096, 20, ms))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_token():
    world = 2
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        w, r, local, ms, value = res[rank]
        assert (w, r, local) == (world, rank, rank)
        assert ms == 15.0  # both ranks report the slower rank's time
        assert value == pytest.approx(2 * 4096 * 20 / 15e-3)


def test_single_rank_needs_no_process_group():
    assert bench.slowest_rank_ms(3.5, 1) == 3.5
    assert bench.job_tokens_per_s(1, 64, 10, 2.0) == pytest.approx(64 * 10 / 2e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun every rank but 0 exits at once, without work or output."""
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 1, 0

    assert bench.bench_reference(Args(), bench.I.TINY) == 0
    assert capsys.readouterr().out == ""
