"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

SPRINT shards by sequence: each rank decodes its own sequences and the job's
numbers are the sum of steps over ranks divided by the slowest rank's time.
These tests run that arithmetic over a real process group without a GPU.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.rank_info()
    bench.init_dist(w, "gloo")
    elapsed = [1.5, 2.5][r]
    steps = [8, 7][r]
    t_max = bench.max_over_ranks(elapsed, w)
    total = bench.sum_over_ranks(steps, w)
    bench.barrier(w)
    from workload import WORKLOADS
    S = WORKLOADS["batch-16x8k"].S
    seqs = [r * S + s for s in range(S)]
    out[r] = (r, w, local, t_max, total, seqs[0], seqs[-1])
    dist.destroy_process_group()


def test_rank_arithmetic_gloo_world_2():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True,
                           start_method="spawn")
        got = dict(out)
    assert got[0][:3] == (0, 2, 0) and got[1][:3] == (1, 2, 1)
    for r in (0, 1):
        assert got[r][3] == pytest.approx(2.5)      # slowest rank's time
        assert got[r][4] == pytest.approx(15.0)     # steps summed over ranks
    # disjoint, contiguous sequence sets per rank
    assert got[0][5:] == (0, 15) and got[1][5:] == (16, 31)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.sum_over_ranks(4, 1) == 4.0


def test_gpus_flag_matches_the_launch():
    """--gpus N never silently measures another number of GPUs: without a
    launcher N > 1 spawns N ranks, and a launcher's world size must be N."""
    import bench
    assert bench.launch_plan(1, {}) == "run"
    assert bench.launch_plan(4, {}) == "spawn"
    assert bench.launch_plan(2, {"WORLD_SIZE": "2"}) == "run"
    with pytest.raises(SystemExit):
        bench.launch_plan(8, {"WORLD_SIZE": "1"})
    with pytest.raises(SystemExit):
        bench.launch_plan(1, {"WORLD_SIZE": "2"})
    with pytest.raises(SystemExit):
        bench.launch_plan(0, {})
