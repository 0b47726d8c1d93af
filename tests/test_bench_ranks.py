"""The bench's multi-GPU host logic, run as two gloo ranks on the CPU: each
rank draws its own batch, the job's time is the slowest rank's, the
throughput counts every rank's tokens, and only rank 0 runs the reference
arm."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from dropless_mixture_experts_gb300.synthetic import MoEConfig, make_inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.rank_info() == (world, rank, rank)
        # per-rank times: the job's is the maximum, value by value
        times = bench.max_over_ranks([1.0 + rank, 10.0 - rank], "cpu")
        # each rank's batch differs (seeded per rank)
        cfg = MoEConfig(64, 64, 64, 4, 2, 0, "f32", "ranks")
        x = make_inputs(cfg, seed_offset=bench.rank_seed_offset(rank))["x"]
        digest = torch.tensor([float(np.sum(x * np.arange(x.size).reshape(x.shape)))],
                              dtype=torch.float64)
        digests = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(digests, digest)
        out[rank] = (times, [float(d) for d in digests])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        times, digests = res[r]
        assert times == [2.0, 10.0]
        assert digests[0] != digests[1]
    # whole-job throughput: both ranks' tokens over the slowest rank's time
    assert bench.job_tokens_per_s(2, 32768, 0.5) == 2 * 32768 / 0.5


def test_max_over_ranks_without_a_group():
    assert bench.max_over_ranks([3.0, 4.5], "cpu") == [3.0, 4.5]


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        warmup, steps, gpus = 1, 1, 2

    bench.reference_arm(Args, MoEConfig(64, 64, 64, 4, 2, 0, "f32", "ranks"))
    assert capsys.readouterr().out == ""
