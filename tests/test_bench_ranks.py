"""The bench's multi-process host logic on CPU: two ranks over gloo (no GPU).
One process per GPU runs an independent replica of the layer (the path has
no exchange step); the job's time is the max over ranks, its throughput the
tokens of all ranks over that time, and the ranks draw disjoint tokens."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own timed region (ms); the job's is the slowest
        local = [41.5, 57.25][rank]
        job_ms = bench.max_over_ranks(torch, local, world, torch.device("cpu"))
        out[rank] = (job_ms, bench.job_tokens_per_s(world, 200, 1, job_ms),
                     bench.rank_draw0(rank, 200))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_rank_and_all_tokens():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 57.25
    # 2 ranks x 200 steps x 1 token in 57.25 ms
    assert res[0][1] == pytest.approx(2 * 200 / 57.25e-3)
    # disjoint token draws: rank 1 starts where rank 0's 200 draws end
    assert res[1][2] - res[0][2] == 200


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(torch, 12.5, 1, torch.device("cpu")) == 12.5
    assert bench.job_tokens_per_s(1, 100, 4096, 1000.0) == pytest.approx(409600.0)
