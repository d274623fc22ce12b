"""Oracle for sharding one join batch over ranks by anchor. Test infrastructure.

Source: "Motor de inferência Quail atinge 1 bilhão de tokens por minuto por GPU", section
"Como funciona", cascade-attention bullet: a suffix attends only to its own anchor and to
itself, so an anchor together with its suffixes is an independent unit of work; and the
throughput-per-GPU framing of the key points of "Quail: یک میلیارد توکن در دقیقه روی یک
GPU". The pages give no multi-GPU scheme. Plainest reading: give every rank whole anchors
so that the ranks carry about the same attention work.

  * work of anchor a = its visible (query, key) pairs: for each suffix s of a and each of
    its tokens i, the L_a anchor keys and the i + 1 suffix keys up to itself, i.e.
    sum_s sum_{i < l_s} (L_a + i + 1) = sum_s (l_s L_a + l_s (l_s + 1) / 2) (attention
    FLOPs are 4 d Hq times this);
  * longest processing time first (R. L. Graham, "Bounds on multiprocessing timing
    anomalies", SIAM J. Appl. Math. 17, 1969): anchors in decreasing work (ties: lower
    index first), each to the rank with the least work so far (ties: lower rank).
`optimal_makespan` is the exact minimum over every assignment (tiny inputs only).
"""
from __future__ import annotations

import itertools


def anchor_pairs(anchor_offsets, anchor_suffix_ptr, suffix_offsets):
    """Visible (query, key) pairs of every anchor's suffix tokens (python ints)."""
    ao = [int(x) for x in anchor_offsets]
    asp = [int(x) for x in anchor_suffix_ptr]
    so = [int(x) for x in suffix_offsets]
    out = []
    for a in range(len(ao) - 1):
        la = ao[a + 1] - ao[a]
        total = 0
        for s in range(asp[a], asp[a + 1]):
            ls = so[s + 1] - so[s]
            total += ls * la + ls * (ls + 1) // 2
        out.append(total)
    return out


def lpt(costs, num_ranks):
    """Longest-processing-time-first assignment: (rank of each item, load of each rank)."""
    order = sorted(range(len(costs)), key=lambda a: (-costs[a], a))
    loads = [0] * num_ranks
    rank_of = [0] * len(costs)
    for a in order:
        r = min(range(num_ranks), key=lambda k: (loads[k], k))
        rank_of[a] = r
        loads[r] += costs[a]
    return rank_of, loads


def optimal_makespan(costs, num_ranks):
    """Smallest possible maximum rank load (exhaustive over num_ranks ** len(costs))."""
    best = None
    for assign in itertools.product(range(num_ranks), repeat=len(costs)):
        loads = [0] * num_ranks
        for c, r in zip(costs, assign):
            loads[r] += c
        m = max(loads)
        best = m if best is None else min(best, m)
    return best if best is not None else 0


def sub_batch(anchor_offsets, anchor_suffix_ptr, suffix_offsets, rank_of_anchor, rank):
    """One rank's sub-batch, written out plainly: the anchors assigned to `rank` in their
    original order, each with all of its suffixes; offsets are the prefix sums of the kept
    lengths, and rows list, in that order, the full batch's anchor rows and suffix rows
    that the sub-batch covers."""
    ao = [int(x) for x in anchor_offsets]
    asp = [int(x) for x in anchor_suffix_ptr]
    so = [int(x) for x in suffix_offsets]
    res = {"anchor_offsets": [0], "anchor_suffix_ptr": [0], "suffix_offsets": [0],
           "anchors": [], "anchor_rows": [], "suffix_rows": []}
    for a in range(len(ao) - 1):
        if int(rank_of_anchor[a]) != rank:
            continue
        res["anchors"].append(a)
        res["anchor_rows"].extend(range(ao[a], ao[a + 1]))
        res["anchor_offsets"].append(len(res["anchor_rows"]))
        for s in range(asp[a], asp[a + 1]):
            res["suffix_rows"].extend(range(so[s], so[s + 1]))
            res["suffix_offsets"].append(len(res["suffix_rows"]))
        res["anchor_suffix_ptr"].append(len(res["suffix_offsets"]) - 1)
    return res
