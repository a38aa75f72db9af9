"""The N > 1 path of bench.py on CPU: two gloo ranks, no GPU.

Each rank runs its own independent batch (the mixer has no collective), so the
only cross-rank steps are the host-side barrier around the timed region and
the max-over-ranks of the timed duration; the reported value aggregates all
ranks' tokens over the slowest rank's time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.dist_init(ws, "gloo")
    bench.barrier(ws)
    # rank r "took" (r + 1) seconds: the job time is the slowest rank's
    slowest = bench.max_over_ranks(float(rank + 1), ws, torch.device("cpu"))
    value = bench.aggregate_tokens_per_s(32768, 10, ws, slowest)
    bench.barrier(ws)
    out[rank] = (slowest, value)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_aggregate_over_slowest_rank():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    for rank in range(world):
        slowest, value = out[rank]
        assert slowest == 2.0
        assert value == pytest.approx(32768 * 10 * 2 / 2.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert bench.aggregate_tokens_per_s(100, 4, 1, 2.0) == 200.0
