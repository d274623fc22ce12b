"""Pins of the join-verdict oracle (CPU): a hand-worked batch, and the invariants that tie
the three outputs together on random batches."""
import numpy as np

from oracle import join


def test_hand_worked_batch():
    # anchors: 0 -> suffixes 0..2, 1 -> none, 2 -> suffixes 3..6; "true" is option 5
    argmax = [5, 0, 5, 7, 5, 5, 1]
    v, sel, cnt = join.join_select(argmax, [0, 3, 3, 7], 5)
    assert v.tolist() == [1, 0, 1, 0, 1, 1, 0]
    assert sel.tolist() == [0, 2, 4, 5]
    assert cnt.tolist() == [2, 0, 2]


def test_invariants_on_random_batches():
    rng = np.random.default_rng(2)
    for _ in range(30):
        A = int(rng.integers(0, 20))
        counts = rng.integers(0, 9, size=A)
        asp = np.concatenate([[0], np.cumsum(counts)])
        S = int(asp[-1])
        am = rng.integers(0, 8, size=S)
        t = int(rng.integers(0, 8))
        v, sel, cnt = join.join_select(am, asp, t)
        assert v.sum() == sel.size == cnt.sum()
        assert np.all(np.diff(sel) > 0) and np.all(am[sel] == t)
        assert np.all(am[v == 0] != t)
        # the selected ids of anchor a are exactly those inside its suffix range
        for a in range(A):
            inside = sel[(sel >= asp[a]) & (sel < asp[a + 1])]
            assert inside.size == cnt[a]
