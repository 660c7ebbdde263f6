"""The multi-GPU bench path on CPU: replicas, one process per rank, joined by a
world-size-2 gloo group (no GPU, no data-path collective; only the step time is
reduced, max over ranks)."""
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


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        ms = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = ms
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, [0.37, 0.41], out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1] == 0.41


def test_weak_scaling_throughput():
    # every rank verifies its own batch: the job's rows scale with the ranks, the
    # step lasts as long as the slowest rank
    assert bench.job_rows_per_sec(2560, 1, 0.4) == pytest.approx(6.4e6)
    assert bench.job_rows_per_sec(2560, 4, 0.5) == pytest.approx(4 * 2560 / 0.5e-3)
    assert bench.max_over_ranks(0.3, 1, "cpu") == 0.3


def test_reference_arm_prints_on_rank_0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    import argparse
    ns = argparse.Namespace(workload="w0_v1024_f32", steps=1, warmup=0, cpu_sample=1)
    assert bench.run_reference(ns) == 0
    assert capsys.readouterr().out == ""
