"""The N > 1 path of bench.py on the CPU: two ranks over gloo (replicas only: the codec
shards by token group with no exchange, so the only collectives are the timing's barrier
and its max over ranks).  The GPU ranks run the same functions over NCCL."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own time; the job's is the slowest
        local = 10.0 + 7.5 * rank
        job = bench.max_over_ranks(local, dist, "cpu")
        dist.barrier()
        # the replicas' inputs: different tensors of the same workload
        w = synth.WORKLOADS["c1"]
        x = synth.generate(w, index=bench.replica_tensor_index(rank, 2, 0))
        digest = torch.tensor([float(np.abs(x).sum())], dtype=torch.float64)
        all_d = [torch.zeros(1, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(all_d, digest)
        out[rank] = (job, [float(d.item()) for d in all_d])
    finally:
        dist.destroy_process_group()


def test_two_ranks_gloo_timing_and_replica_inputs():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        job, digests = out[r]
        assert job == 17.5                        # max over ranks, on every rank
        assert digests[0] != digests[1]           # each replica encodes its own tensor


def test_job_value_counts_every_rank():
    # 2 ranks x 1 GiB per step x 10 steps in 20 ms of job time
    assert bench.job_value(2, 1 << 30, 10, 20.0) == pytest.approx(2 * (1 << 30) * 10 / 0.02 / 1e9)
    assert bench.max_over_ranks(3.0, None, "cpu") == 3.0


def test_reference_arm_other_ranks_exit_without_output(capsys, monkeypatch):
    monkeypatch.setenv("RANK", "1")
    args = bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
