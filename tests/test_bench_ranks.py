"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
times its own replica; the reported time is the slowest rank's and the value
counts every rank's FLOPs. With --shard heads the ranks split the KV heads
into contiguous ranges that cover every head exactly once."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r, _ = bench.dist_setup()
    ms = 1.0 + r                      # rank 1 is the slower one
    slowest = bench.max_over_ranks(ms, w, torch.device("cpu"))
    out[rank] = (w, slowest, bench.whole_job_value(10e12, w, slowest))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    world, slowest, value = out[0]
    assert world == 2 and slowest == 2.0
    # 2 ranks x 10 TFLOP in 2 ms = 10,000 TFLOP/s
    assert value == pytest.approx(2 * 10e12 / 2e-3 / 1e12)


def _shard_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import argparse
    import bench
    from long_causal_gqa_gb300.inputs import WORKLOADS
    w, r, _ = bench.dist_setup()
    args = argparse.Namespace(shard="heads")
    mine = bench.shard_of(args, WORKLOADS["s10231"], w, r)
    got = [None] * w
    dist.all_gather_object(got, mine)       # host-side bookkeeping only
    out[rank] = got
    dist.destroy_process_group()


def test_two_ranks_split_the_heads():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_shard_worker, args=(2, port, out), nprocs=2, join=True,
                       start_method="spawn")
    assert out[0] == out[1]
    ranges = out[0]
    heads = [h for b, c in ranges for h in range(b, b + c)]
    assert heads == list(range(8))                  # every KV head once
    assert [c for _, c in ranges] == [4, 4]         # balanced
