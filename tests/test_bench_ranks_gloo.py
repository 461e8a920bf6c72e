"""The benchmark's multi-rank host logic on CPU, with two gloo ranks.

Under torchrun every rank runs its own replica of the step (no collective on
the data path); the job's time is the slowest rank's, taken by an all-reduce
of the timings, and the job's throughput counts the work of all ranks over
that time.  The reference arm runs on rank 0 alone: any other rank returns 0
without work and prints nothing.
"""
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    assert bench.dist_env() == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (10 + r) ms for the device loop and (20 - r) ms end to end
        ms, ems = bench.max_over_ranks(torch, [10.0 + rank, 20.0 - rank], "cpu", world)
        value = bench.job_tflops(1e12, 5, world, ms)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"ms": ms, "ems": ems, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        d = json.load(open(tmp_path / f"r{r}.json"))
        assert d["ms"] == 11.0 and d["ems"] == 20.0
        # 5 steps of 1 TFLOP on each of 2 ranks in 11 ms
        assert abs(d["value"] - 10.0 / 0.011) < 1e-9 * d["value"]


def test_one_rank_needs_no_collective():
    import bench
    assert bench.max_over_ranks(torch, [3.0, 4.0], "cpu", 1) == [3.0, 4.0]
    assert bench.job_tflops(2e12, 10, 1, 1000.0) == 20.0


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    import argparse
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = argparse.Namespace(workload="bf16_llama8b", steps=1, warmup=0, ref_tokens=16, t=8, tokens=0,
                              optimizer="sgd", precision="bf16", sequence_parallel=False, attn_path="fused")
    assert bench.reference_arm(args) == 0
    assert capsys.readouterr().out == ""
