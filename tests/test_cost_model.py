"""Host-side checks of the cost model (no GPU): work formulas against hand-computed small
plans, the speed-of-light bound, the work-item enumeration against the schedule's
invariants, and the per-item MMA cycle count against a hand count."""
import math

import numpy as np

import workloads
from prefill_only_cascade_gb300 import cost_model as cm


def _layout(anchors, counts, lens):
    lay = workloads.layout_from_lengths(anchors, counts, lens)
    return lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets


def test_visible_pairs_by_hand():
    # anchor of 10 keys with suffixes of 3 and 1 tokens: 3*10 + (1+2+3) + 1*10 + 1 = 47
    w = cm.work(*_layout([10], [2], [3, 1]), hq=4, hkv=1, d=64)
    assert w["visible_pairs"] == 47
    assert w["flops"] == 4 * 64 * 4 * 47
    ts, ta = 4, 10
    assert w["bytes"] == ts * 4 * 64 * 4 + ts * 4 * 4 + ts * 1 * 64 * 4 + ta * 64 * 4 \
        + 4 * (2 * 2 + 2 + 1)


def test_sol_is_the_larger_bound():
    hw = cm.Hardware(bf16_tflops=1000.0, hbm_gbs=5000.0)
    assert cm.sol_seconds(1e12, 1e6, hw) == 1e12 / 1e15          # tensor-bound
    assert cm.sol_seconds(1e6, 5e9, hw) == 5e9 / 5e12            # HBM-bound


def test_work_items_follow_the_schedule():
    rng = np.random.default_rng(3)
    anchors = [300, 0, 1024, 77]
    counts = [5, 3, 7, 2]
    lens = rng.integers(1, 90, size=sum(counts))
    ao, asp, so = _layout(anchors, counts, lens)
    hq, hkv = 32, 8
    items = cm.work_items(ao, asp, so, hq, hkv)
    tok = 128 // (hq // hkv)
    per_anchor = [int(so[asp[a + 1]] - so[asp[a]]) for a in range(len(anchors))]
    assert items["la"].size == hkv * sum(math.ceil(n / (2 * tok)) for n in per_anchor)
    # anchors in decreasing anchor-tile order: 1024 keys first, then 300, then 77, then 0
    assert list(items["la"][:1]) == [1024] and items["la"][-1] == 0
    seg = np.repeat(so[:-1], np.diff(so))
    for ws, te in ((items["ws0"], items["tend0"]), (items["ws1"], items["tend1"])):
        nonempty = te > ws
        assert (ws[nonempty] <= te[nonempty]).all()
        # the window starts at the suffix start of a token of the tile
        assert np.isin(ws[nonempty], seg).all()


def test_item_mma_cycles_by_hand():
    hw = cm.Hardware()
    # 256 anchor keys (2 full tiles) and two 32-token query tiles whose windows are 32 keys:
    # per query tile 2 x (S 8 x 96 + PV 8 x 72) + one 64-key suffix tile (8 x 68 + 4 x 72)
    items = {"la": np.array([256]), "ws0": np.array([0]), "ws1": np.array([32]),
             "tend0": np.array([32]), "tend1": np.array([64]), "t0": np.array([0]),
             "t1": np.array([32]), "sl0": np.array([0]), "sl1": np.array([32])}
    per_q = 2 * (8 * 96 + 8 * 72) + (8 * 68 + 4 * 72)
    assert cm.item_mma_cycles(items, 128, hw)[0] == 2 * per_q
    assert cm.masked_tiles(items)[0] == 2 * 1        # the suffix tile; anchor tiles full


def test_masked_tiles_of_a_long_suffix():
    # one sequence of 1,024 tokens with no anchor (the causal-prefill shape), G = 4: a
    # query tile of 32 tokens starting at token t0 sees tiles below floor((t0 + 1) / 128)
    # whole; only the diagonal tile (and, for the item's shorter tile, the tile beyond
    # its own window) needs the mask
    ao, asp, so = _layout([0], [1], [1024])
    items = cm.work_items(ao, asp, so, 32, 8)
    m = cm.masked_tiles(items)
    assert m.size == 8 * 16
    for k in range(16):  # item k: query tiles at tokens 64k and 64k + 32
        t0, t1 = 64 * k, 64 * k + 32
        n = (t1 + 32 + 127) // 128                   # suffix tiles of the item
        whole0 = sum(1 for i in range(n) if 128 * i + 127 <= t0)
        whole1 = sum(1 for i in range(n) if 128 * i + 127 <= t1)
        assert m[k] == 2 * n - whole0 - whole1


def test_model_time_grows_with_work_and_beats_nothing_below_sol():
    ao, asp, so = _layout([1024] * 8, [256] * 8, [16] * 2048)
    small = cm.plan_report(ao, asp, so, 32, 8, 128)
    ao2, asp2, so2 = _layout([1024] * 8, [512] * 8, [16] * 4096)
    big = cm.plan_report(ao2, asp2, so2, 32, 8, 128)
    assert big["model_seconds"] > small["model_seconds"]
    for r in (small, big):
        assert r["model_seconds"] >= r["mma_floor_seconds"] >= 0.9 * r["sol_seconds"]
        assert r["bound"] == "tensor"


def test_visible_pairs_agree_across_bench_cost_model_and_oracle():
    # three independent countings of the visible (query, key) pairs: the bench's FLOP
    # count, the cost model's work, and the sharding oracle's per-anchor work
    import bench
    from oracle import shard
    rng = np.random.default_rng(31)
    for _ in range(10):
        A = int(rng.integers(1, 9))
        counts = rng.integers(0, 7, size=A)
        lay = workloads.layout_from_lengths(rng.integers(0, 500, size=A), counts,
                                            rng.integers(1, 70, size=int(counts.sum())))
        pairs = sum(shard.anchor_pairs(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                       lay.suffix_offsets))
        w = cm.work(lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets, 32, 8, 128)
        assert w["visible_pairs"] == pairs
        assert bench.attention_flops(lay, 32, 128) == 4 * 128 * 32 * pairs
