"""The multi-process path of bench.py on the CPU: `--gpus N` runs N independent
replicas (the attention of one process never exchanges data with another),
so the only cross-rank steps are the barriers around the timed region and
the max over ranks of the elapsed time.  Two gloo ranks check that every
rank gets the slowest rank's time and that the whole-job rate counts the
units of all ranks over that time.  CPU only."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 * (rank + 1) + 0.25          # rank 1 is the slow one
        dist.barrier()
        slowest = bench.max_over_ranks(mine, torch.device("cpu"), world)
        rate = bench.job_rate(world, 1000.0, 4, slowest)
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump([mine, slowest, rate], f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank(tmp_path):
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = {r: json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)}
    for rank, (mine, slowest, rate) in res.items():
        assert mine == 10.0 * (rank + 1) + 0.25
        assert slowest == 20.25                    # every rank sees the max
        # 2 ranks x 1000 units x 4 steps over 20.25 ms
        assert rate == pytest.approx(2 * 1000.0 * 4 / 20.25e-3)


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(3.5, torch.device("cpu"), 1) == 3.5
    assert bench.job_rate(1, 10.0, 2, 4.0) == pytest.approx(5000.0)
