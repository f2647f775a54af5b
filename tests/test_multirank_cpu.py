"""The multi-rank host logic of bench.py, run as two gloo ranks on the CPU.

Each rank of a multi-GPU run is an independent replica (the path has no
data-path exchange); the only collective is the maximum of the timing
numbers, and rank 0 alone prints.  Launched here with torch.multiprocessing
(spawn) on 127.0.0.1.
"""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took (r + 1) * 10 ms for its steps and (r + 1) * 30 ms end to end
    got = bench.max_over_ranks([(rank + 1) * 10.0, (rank + 1) * 30.0], world, "cpu")
    rate = bench.job_rate(1.0e12, 5, got[0], world)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": got, "rate": rate}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_aggregation(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["max"] == [20.0, 60.0]  # the slowest rank's times, on every rank
        # 2 ranks x 5 steps x 1e12 units over the slowest 20 ms
        assert r["rate"] == pytest.approx(2 * 5 * 1.0e12 / 0.020)


def test_reference_arm_is_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        gpus, steps, warmup, seed = 2, 1, 0, 0
    bench.run_reference(Args, None, rank=1, world=2)  # other ranks exit without work
    assert capsys.readouterr().out == ""
