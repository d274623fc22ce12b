"""The native anchor-KV planner (quail_kv_plan, host code) against the oracle: every hit
flag and every statistic must match, for both policies, on random plans of all sizes
(CPU only: the planner does no GPU work)."""
import numpy as np
import pytest

import prefill_only_cascade_gb300 as q
from oracle import kv_plan as kp

POLICIES = [(q.KV_LRU, kp.LRU), (q.KV_FURTHEST_NEXT_USE, kp.BELADY)]


def _random_plan(rng, n_anchor, n_access, size_hi):
    # skewed reuse: a few anchors are accessed often, as when a join revisits a table
    weights = rng.pareto(1.2, size=n_anchor) + 0.05
    acc = rng.choice(n_anchor, size=n_access, p=weights / weights.sum())
    size = rng.integers(0, size_hi + 1, size=n_anchor)
    return acc.astype(np.int32), size.astype(np.int64)


@pytest.mark.parametrize("native,orc", POLICIES)
def test_matches_oracle_on_random_plans(native, orc):
    rng = np.random.default_rng(11 + native)
    for trial in range(200):
        n_anchor = int(rng.integers(1, 40))
        n_access = int(rng.integers(0, 300))
        acc, size = _random_plan(rng, n_anchor, n_access, int(rng.integers(1, 50)))
        cap = int(rng.integers(0, max(1, int(size.sum())) + 5))
        hit, st = q.kv_plan(acc, size, cap, native)
        o_hits, o_comp, o_regret, o_peak = kp.simulate(acc.tolist(), size.tolist(), cap, orc)
        assert hit.tolist() == o_hits, trial
        assert (st["compulsory_tokens"], st["regret_tokens"], st["peak_resident_tokens"]) == \
            (o_comp, o_regret, o_peak), trial
        assert st["hits"] == sum(o_hits) and st["hits"] + st["misses"] == n_access


def test_large_plan_matches_oracle():
    rng = np.random.default_rng(5)
    acc, size = _random_plan(rng, 400, 20000, 2000)
    cap = int(size.sum() // 5)
    for native, orc in POLICIES:
        hit, st = q.kv_plan(acc, size, cap, native)
        o_hits, _, o_regret, o_peak = kp.simulate(acc.tolist(), size.tolist(), cap, orc)
        assert hit.tolist() == o_hits
        assert st["regret_tokens"] == o_regret and st["peak_resident_tokens"] == o_peak


def test_rejects_bad_arguments():
    ok = np.array([0, 1], np.int32), np.array([3, 4], np.int64)
    with pytest.raises(q.QuailError):
        q.kv_plan(np.array([0, 2], np.int32), ok[1], 5)          # id out of range
    with pytest.raises(q.QuailError):
        q.kv_plan(ok[0], np.array([3, -1], np.int64), 5)         # negative size
    with pytest.raises(q.QuailError):
        q.kv_plan(ok[0], ok[1], -1)                               # negative capacity
    with pytest.raises(q.QuailError):
        q.kv_plan(ok[0], ok[1], 5, policy=7)                      # unknown policy
    hit, st = q.kv_plan(np.zeros(0, np.int32), np.zeros(0, np.int64), 0)
    assert hit.size == 0 and st["misses"] == 0
