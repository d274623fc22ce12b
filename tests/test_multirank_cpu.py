"""The N>1 path on CPU with two gloo ranks. bench.py: the job's anchors are split over the
ranks by quail_shard_anchors / quail_shard_batch (N batches for weak scaling, one for
strong); only the barrier and the max-over-ranks of the timing cross ranks. One batch
split by anchor: the ranks' results reassemble the full batch's result; only results are
gathered."""
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
        cfg = workloads.ATTN_CONFIGS["ragged"]
        weak, plan = bench.rank_layout(cfg, world, rank)
        strong, _ = bench.rank_layout(cfg, world, rank, strong=True)
        tok = bench.sum_over_ranks(world, float(weak.total_suffix_tokens), device="cpu")
        out[rank] = (got, plan, weak.num_anchors, weak.total_suffix_tokens, tok,
                     strong.num_anchors, strong.total_suffix_tokens)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_timing_and_anchor_shards():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert out[0][0] == out[1][0] == 15.0          # max over ranks
    assert out[0][1] == out[1][1]                  # every rank derives the same plan
    cfg = workloads.ATTN_CONFIGS["ragged"]
    one = workloads.make_layout(cfg)
    # weak scaling: the job is two batches of the workload's shape, split by anchor
    assert out[0][2] + out[1][2] == 2 * cfg.num_anchors
    assert out[0][4] == bench.global_layout(cfg, 2).total_suffix_tokens
    assert abs(out[0][3] - out[1][3]) < 0.02 * out[0][3]   # balanced ranks
    # strong scaling: one batch split in two
    assert out[0][5] + out[1][5] == cfg.num_anchors
    assert out[0][6] + out[1][6] == one.total_suffix_tokens
    loads = out[0][1]["rank_pairs"]
    assert max(loads) <= 1.01 * sum(loads) / 2


def _shard_worker(rank, world, port, out):
    """One rank of a sharded join: the same seeded batch on every rank, the anchors split
    by quail_shard_anchors, this rank's sub-batch computed (float64 oracle on CPU, standing
    in for the GPU call), results gathered on rank 0 - the only cross-rank traffic is the
    gather of results, as the path has no exchange step."""
    import oracle
    import prefill_only_cascade_gb300 as q
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lay = workloads.layout_from_lengths([40, 0, 130, 64, 7], [3, 2, 4, 1, 2],
                                            [5, 1, 12, 3, 8, 9, 2, 20, 4, 6, 1, 11])
        rng = np.random.default_rng(29)
        T_S, T_A, hq, hkv, d = lay.total_suffix_tokens, lay.total_anchor_tokens, 4, 2, 16
        qs = rng.standard_normal((T_S, hq, d))
        ka, va = rng.standard_normal((T_A, hkv, d)), rng.standard_normal((T_A, hkv, d))
        ks, vs = rng.standard_normal((T_S, hkv, d)), rng.standard_normal((T_S, hkv, d))
        rank_of, pairs = q.shard_anchors(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                         lay.suffix_offsets, world)
        sb = q.shard_batch(lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets,
                           rank_of, rank)
        ar, sr = sb["anchor_rows"], sb["suffix_rows"]
        o, l_ = oracle.cascade_attention(qs[sr], ka[ar], va[ar], ks[sr], vs[sr],
                                         sb["anchor_offsets"], sb["anchor_suffix_ptr"],
                                         sb["suffix_offsets"])
        parts = [None] * world
        dist.all_gather_object(parts, (rank, sr, o, l_, rank_of.tolist()))
        if rank == 0:
            full_o = np.full((T_S, hq, d), np.nan)
            full_l = np.full((T_S, hq), np.nan)
            for _, rows, po, pl, _ in parts:
                full_o[rows], full_l[rows] = po, pl
            ref_o, ref_l = oracle.cascade_attention(qs, ka, va, ks, vs, lay.anchor_offsets,
                                                    lay.anchor_suffix_ptr, lay.suffix_offsets)
            out["max_err"] = float(max(np.abs(full_o - ref_o).max(), np.abs(full_l - ref_l).max()))
            out["same_plan"] = all(p[4] == parts[0][4] for p in parts)
            out["pairs"] = pairs.tolist()
            out["rows"] = sorted(int(x) for p in parts for x in p[1]) == list(range(T_S))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_one_batch_by_anchor():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_shard_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert out["same_plan"]                     # every rank derives the same plan
    assert out["rows"]                          # every suffix row computed exactly once
    assert out["max_err"] < 1e-12               # the union is the full batch's result
    from oracle import shard
    lay = workloads.layout_from_lengths([40, 0, 130, 64, 7], [3, 2, 4, 1, 2],
                                        [5, 1, 12, 3, 8, 9, 2, 20, 4, 6, 1, 11])
    costs = shard.anchor_pairs(lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets)
    assert out["pairs"] == shard.lpt(costs, world)[1]   # the plan's loads are LPT's
