"""The multi-GPU path of the benchmark is replicas only: every rank runs its
own layer and the job's step time is the slowest rank's.  This checks that
host logic with two gloo ranks on the CPU (no GPU): the max-over-ranks
reduction, the whole-job throughput, and that the reference arm does its
work on rank 0 only."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, world)          # rank 1 is the slow replica
    e2e = bench.max_over_ranks(0.002 * (rank + 1), world)
    value = bench.job_throughput(16, world, ms / 1e3)
    dist.barrier()
    results[rank] = (ms, e2e, value)
    dist.destroy_process_group()


def test_two_rank_reduction_and_throughput():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), results), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        ms, e2e, value = results[r]
        assert ms == 15.0 and e2e == 0.004
        assert value == pytest.approx(world * 16 / 0.015)


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(16, 1, 0.5) == 32.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    """Under torchrun every rank starts the reference arm; ranks other than 0
    return at once, without work and without printing."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    from nvfp4_mixture_experts_top_gb300 import workloads as wl
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        ref_tokens, warmup, steps, mode = 1, 3, 1, "w4a4"
    assert bench.run_reference(Args, wl.CONFIGS["tiny"], "m", "tokens/s") is None
    assert capsys.readouterr().out == ""
