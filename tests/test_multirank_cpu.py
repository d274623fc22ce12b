"""The N>1 path of bench.py on CPU: two gloo ranks. The path shards by anchor (each rank
runs its own batch of the same shape, no data-path collective); only the barrier and the
max-over-ranks of the timing cross ranks."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        got = bench.max_over_ranks(world, float(10 + 5 * rank), device="cpu")
        total = bench.sum_over_ranks(world, float(1 + rank), device="cpu")
        assert total == 3.0
        cfg = bench.rank_workload(workloads.ATTN_CONFIGS["tiny"], rank)
        lay = workloads.make_layout(cfg)
        t = workloads.make_attention_inputs(cfg, lay, "cpu")
        out[rank] = (got, cfg.seed, float(t["q_suf"].float().sum()), lay.total_suffix_tokens)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_timing_and_distinct_batches():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 15.0          # max over ranks
    assert out[0][1] != out[1][1]                  # rank-specific seeds
    assert out[0][2] != out[1][2]                  # so different data
    assert out[0][3] == out[1][3]                  # of the same shape (weak scaling)
