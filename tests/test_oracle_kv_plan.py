"""Pins of the KV-plan oracle (CPU): a hand-worked cyclic plan, Belady's optimality for
equal sizes against the exhaustive minimum, bounds that hold for any plan."""
import numpy as np

from oracle import kv_plan as kp


def test_cyclic_plan_by_hand():
    # capacity for two of three equal anchors, accessed A B C A B C
    acc, size = [0, 1, 2, 0, 1, 2], [1, 1, 1]
    hits, comp, regret, peak = kp.simulate(acc, size, 2, kp.LRU)
    assert hits == [0, 0, 0, 0, 0, 0] and comp == 3 and regret == 3 and peak == 2
    hits, comp, regret, peak = kp.simulate(acc, size, 2, kp.BELADY)
    # C has the furthest next use at its first access: bypassed, A and B hit
    assert hits == [0, 0, 0, 1, 1, 0] and comp == 3 and regret == 1
    assert kp.min_regret(acc, size, 2) == 1


def test_belady_is_optimal_for_equal_sizes():
    rng = np.random.default_rng(7)
    for _ in range(300):
        n_anchor = int(rng.integers(2, 5))
        acc = [int(x) for x in rng.integers(0, n_anchor, size=int(rng.integers(1, 10)))]
        cap = int(rng.integers(1, n_anchor + 1))
        size = [1] * n_anchor
        _, _, regret, _ = kp.simulate(acc, size, cap, kp.BELADY)
        assert regret == kp.min_regret(acc, size, cap), (acc, cap)


def test_bounds_for_any_sizes():
    rng = np.random.default_rng(8)
    for _ in range(300):
        n_anchor = int(rng.integers(2, 5))
        acc = [int(x) for x in rng.integers(0, n_anchor, size=int(rng.integers(1, 9)))]
        size = [int(x) for x in rng.integers(1, 6, size=n_anchor)]
        cap = int(rng.integers(1, sum(size) + 1))
        opt = kp.min_regret(acc, size, cap)
        for pol in (kp.LRU, kp.BELADY):
            hits, comp, regret, peak = kp.simulate(acc, size, cap, pol)
            assert regret >= opt and peak <= cap
            assert comp == sum(size[a] for a in set(acc))
            # every miss prefills its anchor: misses cost compulsory + regret tokens
            assert sum(size[a] for a, h in zip(acc, hits) if not h) == comp + regret


def test_everything_fits_or_nothing_does():
    acc, size = [0, 1, 0, 2, 1, 0], [3, 4, 5]
    for pol in (kp.LRU, kp.BELADY):
        assert kp.simulate(acc, size, 12, pol)[2] == 0           # all fit: no regret
        # every anchor larger than the capacity: each repeat is regret
        assert kp.simulate(acc, size, 2, pol)[2] == 3 + 4 + 3
