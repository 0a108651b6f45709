"""The bench's multi-process path on CPU: two gloo ranks.

`bench.py --gpus N` runs one replica per GPU (the layer shards by tokens with
no exchange); what crosses ranks is the timing: the job's time is the slowest
rank's, and the value counts the tokens of every rank.  The reference arm is
printed by rank 0 only.
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
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, value = bench.job_time_and_value(10.0 + 5.0 * rank, T=32, K=100, dist=dist, device="cpu")
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_tokens(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    for r in range(world):
        d = json.load(open(tmp_path / f"rank{r}.json"))
        assert d["ms"] == 15.0                              # max over ranks
        assert d["value"] == pytest.approx(32 * 100 * world / 15e-3)


def test_single_process_value():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.job_time_and_value(20.0, T=16, K=10, dist=None, device="cpu")
    assert ms == 20.0 and value == pytest.approx(16 * 10 / 20e-3)


def _reference_rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    from synth import CONFIGS

    class Args:
        gpus, steps, warmup = world, 1, 0

    path = os.path.join(out_dir, f"ref{rank}.txt")
    with open(path, "w") as f:
        old = sys.stdout
        sys.stdout = f
        try:
            bench.run_reference(Args, CONFIGS["tiny"])
        finally:
            sys.stdout = old


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    world = 2
    mp.start_processes(_reference_rank, args=(world, 0, str(tmp_path)), nprocs=world, start_method="spawn")
    line = json.loads(open(tmp_path / "ref0.txt").read().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["config"]["T"] == 16
    assert open(tmp_path / "ref1.txt").read().strip() == ""
