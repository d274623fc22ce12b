"""GPU parity of quail_join_select (the join's verdicts from the head's argmax) against
the oracle, bit for bit: per-suffix verdicts, the passing suffix ids in order, their
number and the per-anchor counts, across chunk boundaries (4,096 suffixes per CTA) and
the empty cases."""
import numpy as np
import pytest
import torch

import oracle
import prefill_only_cascade_gb300 as q

pytestmark = pytest.mark.gpu


def _run(am_np, asp_np, t):
    dev = "cuda"
    S, A = am_np.size, asp_np.size - 1
    am = torch.from_numpy(am_np.astype(np.int32)).to(dev)
    asp = torch.from_numpy(asp_np.astype(np.int32)).to(dev)
    sel = torch.full((max(S, 1),), -7, dtype=torch.int32, device=dev)
    nsel = torch.full((1,), -7, dtype=torch.int32, device=dev)
    cnt = torch.full((max(A, 1),), -7, dtype=torch.int32, device=dev)
    verdict = torch.full((max(S, 1),), 9, dtype=torch.uint8, device=dev)
    ws = torch.empty(q.join_select_workspace_size(S), dtype=torch.uint8, device=dev)
    q.join_select(am, t, sel, nsel, ws, verdict=verdict, anchor_suffix_ptr=asp,
                  anchor_count=cnt)
    torch.cuda.synchronize()
    n = int(nsel.item())
    return (verdict.cpu().numpy()[:S], sel.cpu().numpy()[:n], n, cnt.cpu().numpy()[:A],
            sel.cpu().numpy()[n:S])


@pytest.mark.parametrize("S", [0, 1, 15, 4095, 4096, 4097, 33152, 1_000_003])
def test_matches_the_oracle(S):
    rng = np.random.default_rng(S)
    A = max(1, S // 500)
    cuts = np.sort(rng.integers(0, S + 1, size=A - 1))
    asp = np.concatenate([[0], cuts, [S]])
    am = rng.integers(0, 8, size=S)
    for t in (0, 5):
        v, sel, n, cnt, rest = _run(am, asp, t)
        rv, rsel, rcnt = oracle.join_select(am, asp, t)
        assert n == rsel.size
        np.testing.assert_array_equal(v, rv)
        np.testing.assert_array_equal(sel, rsel)
        np.testing.assert_array_equal(cnt, rcnt)
        assert (rest == -7).all()          # past the count, `selected` is untouched


def test_all_and_none_pass():
    S = 9000
    asp = np.array([0, 100, 100, 9000])
    v, sel, n, cnt, _ = _run(np.full(S, 3), asp, 3)
    assert n == S and np.array_equal(sel, np.arange(S)) and cnt.tolist() == [100, 0, 8900]
    v, sel, n, cnt, _ = _run(np.full(S, 3), asp, 2)
    assert n == 0 and not v.any() and cnt.tolist() == [0, 0, 0]
