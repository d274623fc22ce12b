"""quail_shard_anchors (host C++) against the sharding oracle, bit for bit, and the
sub-batch built for one rank: the oracle's cascade attention over each rank's sub-batch
gives exactly the full batch's rows. CPU only."""
import numpy as np
import pytest

import oracle
import prefill_only_cascade_gb300 as q
import workloads
from oracle import shard


def _random_layout(rng, max_anchors=12):
    A = int(rng.integers(1, max_anchors + 1))
    anchors = rng.integers(0, 300, size=A)
    counts = rng.integers(0, 6, size=A)
    lens = rng.integers(0, 40, size=int(counts.sum()))
    return workloads.layout_from_lengths(anchors, counts, lens)


def test_matches_the_oracle_bit_for_bit():
    rng = np.random.default_rng(17)
    for trial in range(40):
        lay = _random_layout(rng)
        ranks = int(rng.integers(1, 6))
        got_rank, got_pairs = q.shard_anchors(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                              lay.suffix_offsets, ranks)
        costs = shard.anchor_pairs(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                   lay.suffix_offsets)
        ref_rank, ref_loads = shard.lpt(costs, ranks)
        assert got_rank.tolist() == ref_rank, trial
        assert got_pairs.tolist() == ref_loads, trial


def test_full_size_join_is_balanced():
    cfg = workloads.ATTN_CONFIGS["ragged"]
    lay = workloads.make_layout(cfg)
    for ranks in (2, 4, 8):
        _, pairs = q.shard_anchors(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                   lay.suffix_offsets, ranks)
        total = int(pairs.sum())
        costs = shard.anchor_pairs(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                   lay.suffix_offsets)
        assert total == sum(costs)
        # 256 anchors of similar size over 8 ranks: within 1 % of a perfect split
        assert pairs.max() <= 1.01 * total / ranks


def test_rejects_bad_arguments():
    ao = np.array([0, 3, 5], np.int32)
    asp = np.array([0, 1, 2], np.int32)
    so = np.array([0, 2, 4], np.int32)
    with pytest.raises(RuntimeError):
        q.shard_anchors(ao, asp, so, 0)                                   # no rank
    with pytest.raises(RuntimeError):
        q.shard_anchors(np.array([0, 3, 2], np.int32), asp, so, 2)       # negative length
    with pytest.raises(RuntimeError):
        q.shard_anchors(ao, np.array([1, 1, 2], np.int32), so, 2)        # CSR not from 0
    with pytest.raises(RuntimeError):
        q.shard_anchors(ao, asp, np.array([0, 3, 1], np.int32), 2)       # suffix length < 0
    empty_rank, empty_pairs = q.shard_anchors(np.array([0], np.int32), np.array([0], np.int32),
                                              np.array([0], np.int32), 3)
    assert empty_rank.size == 0 and empty_pairs.tolist() == [0, 0, 0]


def test_sub_batches_reproduce_the_full_batch():
    rng = np.random.default_rng(23)
    lay = _random_layout(rng, max_anchors=7)
    hq, hkv, d = 4, 2, 16
    T_S, T_A = lay.total_suffix_tokens, lay.total_anchor_tokens
    qs = rng.standard_normal((T_S, hq, d))
    ka, va = rng.standard_normal((T_A, hkv, d)), rng.standard_normal((T_A, hkv, d))
    ks, vs = rng.standard_normal((T_S, hkv, d)), rng.standard_normal((T_S, hkv, d))
    ref_out, ref_lse = oracle.cascade_attention(qs, ka, va, ks, vs, lay.anchor_offsets,
                                                lay.anchor_suffix_ptr, lay.suffix_offsets)
    ranks = 3
    rank_of, _ = q.shard_anchors(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                 lay.suffix_offsets, ranks)
    out = np.full_like(ref_out, np.nan)
    lse = np.full_like(ref_lse, np.nan)
    seen = []
    for r in range(ranks):
        sb = q.shard_batch(lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets,
                           rank_of, r)
        ar, sr = sb["anchor_rows"], sb["suffix_rows"]
        o, l_ = oracle.cascade_attention(qs[sr], ka[ar], va[ar], ks[sr], vs[sr],
                                         sb["anchor_offsets"], sb["anchor_suffix_ptr"],
                                         sb["suffix_offsets"])
        out[sr], lse[sr] = o, l_
        seen.append(sr)
    rows = np.concatenate(seen)
    assert np.array_equal(np.sort(rows), np.arange(T_S))      # every row exactly once
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_sub_batch_matches_the_oracle_bit_for_bit():
    rng = np.random.default_rng(31)
    for trial in range(40):
        lay = _random_layout(rng)
        ranks = int(rng.integers(1, 5))
        rank_of, _ = q.shard_anchors(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                     lay.suffix_offsets, ranks)
        for r in range(ranks + 1):            # rank == ranks owns nothing: an empty batch
            got = q.shard_batch(lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets,
                                rank_of, r)
            ref = shard.sub_batch(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                  lay.suffix_offsets, rank_of, r)
            for key, val in ref.items():
                assert got[key].tolist() == val, (trial, r, key)


def test_sub_batch_rejects_bad_arguments():
    import ctypes
    ao = np.array([0, 3, 5], np.int32)
    asp = np.array([0, 1, 2], np.int32)
    so = np.array([0, 2, 4], np.int32)
    ro = np.array([0, 1], np.int32)
    sz = q.ShardSizes()
    p = lambda x: x.ctypes.data
    call = lambda A=2, ao=ao, asp=asp, so=so, ro=ro, rank=0, sizes=ctypes.byref(sz), arrays=(
        None,) * 6: q.lib.quail_shard_batch(A, p(ao), p(asp), p(so), p(ro), rank, sizes, *arrays)
    assert call() == q.QUAIL_OK and (sz.num_anchors, sz.num_suffixes) == (1, 1)
    assert (sz.anchor_tokens, sz.suffix_tokens) == (3, 2)
    assert call(rank=-1) == q.QUAIL_ERR_INVALID_ARG
    assert call(A=-1) == q.QUAIL_ERR_INVALID_ARG
    assert call(sizes=None) == q.QUAIL_ERR_INVALID_ARG
    assert call(ao=np.array([0, 3, 2], np.int32)) == q.QUAIL_ERR_INVALID_ARG   # length < 0
    assert call(asp=np.array([1, 1, 2], np.int32)) == q.QUAIL_ERR_INVALID_ARG  # CSR not from 0
    buf = np.zeros(8, np.int64)
    # some output arrays given, others not
    assert call(arrays=(p(buf), None, None, None, None, None)) == q.QUAIL_ERR_INVALID_ARG
