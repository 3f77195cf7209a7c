"""Multi-rank host logic of the benchmark, on CPU with gloo (world size 2).

Each rank runs an independent replica of the chunk step (the path has no
exchange between GPUs); the job time is the slowest rank's and the
throughput counts every rank's tokens.  Nothing here touches a GPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [10.0 + 5.0 * rank, 20.0 - 3.0 * rank]      # ms: step, end-to-end
    times, tokens, value = bench.aggregate_ranks(local, 4096, world, "cpu")
    out[rank] = (times, tokens, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregate_is_max_time_and_total_tokens():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        times, tokens, value = out[rank]
        assert times == [15.0, 20.0]          # max over ranks, per timer
        assert tokens == 2 * 4096
        assert value == pytest.approx(2 * 4096 / 0.015)


def test_single_rank_needs_no_process_group():
    import bench
    times, tokens, value = bench.aggregate_ranks([8.0, 9.0], 4096, 1, "cpu")
    assert times == [8.0, 9.0] and tokens == 4096
    assert value == pytest.approx(4096 / 0.008)
