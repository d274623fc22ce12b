"""Pins of the sharding oracle (CPU): the visible-pair count against a brute-force count
from the attention mask, and longest-processing-time-first against Graham's bound, the
exhaustive optimum, a textbook worst case and its special cases."""
import numpy as np

import workloads
from oracle import shard


def _brute_pairs(ao, asp, so):
    """Count (query, key) pairs from the mask: a suffix token sees every key of its anchor
    and the tokens of its own suffix up to itself."""
    out = []
    for a in range(len(ao) - 1):
        n = 0
        for s in range(asp[a], asp[a + 1]):
            toks = range(so[s], so[s + 1])
            for qi, q in enumerate(toks):
                n += ao[a + 1] - ao[a]                                # anchor keys
                n += sum(1 for ki, _ in enumerate(toks) if ki <= qi)  # causal suffix keys
        out.append(n)
    return out


def test_pairs_match_a_count_from_the_mask():
    rng = np.random.default_rng(5)
    for _ in range(20):
        A = int(rng.integers(1, 6))
        anchors = rng.integers(0, 40, size=A)
        counts = rng.integers(0, 4, size=A)
        lens = rng.integers(0, 12, size=int(counts.sum()))
        lay = workloads.layout_from_lengths(anchors, counts, lens)
        assert shard.anchor_pairs(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                  lay.suffix_offsets) == \
            _brute_pairs(list(lay.anchor_offsets), list(lay.anchor_suffix_ptr),
                         list(lay.suffix_offsets))


def test_textbook_worst_case_of_lpt():
    # jobs 3, 3, 2, 2, 2 on two machines: LPT gives {3, 2, 2} and {3, 2} (makespan 7)
    # while {3, 3} and {2, 2, 2} give 6 - Graham's bound 4/3 - 1/(3m) = 7/6 is tight
    rank_of, loads = shard.lpt([3, 3, 2, 2, 2], 2)
    assert rank_of == [0, 1, 0, 1, 0]
    assert sorted(loads) == [5, 7]
    assert shard.optimal_makespan([3, 3, 2, 2, 2], 2) == 6


def test_lpt_within_graham_bound_of_the_optimum():
    rng = np.random.default_rng(9)
    for _ in range(60):
        n = int(rng.integers(1, 8))
        m = int(rng.integers(1, 4))
        costs = [int(x) for x in rng.integers(0, 50, size=n)]
        rank_of, loads = shard.lpt(costs, m)
        opt = shard.optimal_makespan(costs, m)
        assert max(loads) * 3 * m <= (4 * m - 1) * opt
        assert max(loads) >= opt
        assert sum(loads) == sum(costs)
        assert [sum(c for c, r in zip(costs, rank_of) if r == k) for k in range(m)] == loads


def test_special_cases():
    costs = [5, 1, 9, 9, 0]
    assert shard.lpt(costs, 1) == ([0] * 5, [24])
    # at least as many ranks as items: the largest items each go alone, in order
    rank_of, loads = shard.lpt(costs, 6)
    assert rank_of == [2, 3, 0, 1, 4] and max(loads) == 9
    # equal costs: round robin in index order
    assert shard.lpt([4] * 7, 3)[0] == [0, 1, 2, 0, 1, 2, 0]
    assert shard.lpt([], 2) == ([], [0, 0])


def test_sub_batch_hand_worked_and_partition():
    # anchors of 3, 0 and 2 tokens with 2, 1 and 1 suffixes of 1, 2, 0 and 4 tokens;
    # anchors 0 and 2 on rank 1
    ao, asp, so = [0, 3, 3, 5], [0, 2, 3, 4], [0, 1, 3, 3, 7]
    r1 = shard.sub_batch(ao, asp, so, [1, 0, 1], 1)
    assert r1 == {"anchor_offsets": [0, 3, 5], "anchor_suffix_ptr": [0, 2, 3],
                  "suffix_offsets": [0, 1, 3, 7], "anchors": [0, 2],
                  "anchor_rows": [0, 1, 2, 3, 4], "suffix_rows": [0, 1, 2, 3, 4, 5, 6]}
    r0 = shard.sub_batch(ao, asp, so, [1, 0, 1], 0)
    assert r0 == {"anchor_offsets": [0, 0], "anchor_suffix_ptr": [0, 1],
                  "suffix_offsets": [0, 0], "anchors": [1], "anchor_rows": [],
                  "suffix_rows": []}
    # random plans: the sub-batches partition the rows and keep every length
    rng = np.random.default_rng(12)
    for _ in range(30):
        A = int(rng.integers(1, 7))
        counts = rng.integers(0, 4, size=A)
        lay = workloads.layout_from_lengths(rng.integers(0, 20, size=A), counts,
                                            rng.integers(0, 9, size=int(counts.sum())))
        R = int(rng.integers(1, 4))
        rank_of = [int(x) for x in rng.integers(0, R, size=A)]
        a_rows, s_rows, anchors = [], [], []
        for r in range(R):
            sb = shard.sub_batch(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                 lay.suffix_offsets, rank_of, r)
            a_rows += sb["anchor_rows"]
            s_rows += sb["suffix_rows"]
            anchors += sb["anchors"]
            la = np.diff(sb["anchor_offsets"])
            assert list(la) == [int(lay.anchor_lens[a]) for a in sb["anchors"]]
            ls = np.diff(sb["suffix_offsets"])
            assert list(ls) == [int(x) for a in sb["anchors"]
                                for x in lay.suffix_lens[lay.suffix_anchor == a]]
        assert sorted(a_rows) == list(range(lay.total_anchor_tokens))
        assert sorted(s_rows) == list(range(lay.total_suffix_tokens))
        assert sorted(anchors) == list(range(A))
