"""One batch split over ranks by anchor, on one GPU: quail_shard_anchors plans the split,
shard_batch builds each rank's sub-batch, each sub-batch goes through quail_cascade_attn
in turn (as each rank would on its own GPU), and the reassembled rows must match the
float64 oracle on the whole batch."""
import numpy as np
import pytest
import torch

import workloads
from parity_util import check_full, layout_tensors, run_cascade

pytestmark = pytest.mark.gpu

DEVICE = "cuda"


def _sub_layout(sb):
    la = np.diff(sb["anchor_offsets"])
    counts = np.diff(sb["anchor_suffix_ptr"])
    ls = np.diff(sb["suffix_offsets"])
    return workloads.layout_from_lengths(la, counts, ls)


@pytest.mark.parametrize("ranks", [2, 3])
def test_sharded_batch_matches_the_oracle(ranks):
    import prefill_only_cascade_gb300 as q
    heads = (8, 2, 128)
    rng = np.random.default_rng(90 + ranks)
    anchors = [700, 0, 260, 129, 64, 300]
    counts = [5, 2, 6, 3, 4, 2]
    lay = workloads.layout_from_lengths(anchors, counts,
                                        rng.integers(1, 60, size=sum(counts)))
    cfg = workloads.AttnConfig("shard", lay.num_anchors, (0, 0), 0, (0, 0), *heads, False, 91)
    t = workloads.make_attention_inputs(cfg, lay, DEVICE)
    rank_of, pairs = q.shard_anchors(lay.anchor_offsets, lay.anchor_suffix_ptr,
                                     lay.suffix_offsets, ranks)
    assert (pairs > 0).all()                       # every rank gets work here
    out = torch.full((lay.total_suffix_tokens, heads[0], heads[2]), float("nan"),
                     dtype=torch.bfloat16, device=DEVICE)
    lse = torch.full((lay.total_suffix_tokens, heads[0]), float("nan"), dtype=torch.float32,
                     device=DEVICE)
    for r in range(ranks):
        sb = q.shard_batch(lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets,
                           rank_of, r)
        sub = _sub_layout(sb)
        ar = torch.from_numpy(sb["anchor_rows"]).to(DEVICE)
        sr = torch.from_numpy(sb["suffix_rows"]).to(DEVICE)
        ts = {"q_suf": t["q_suf"][sr], "k_anc": t["k_anc"][ar], "v_anc": t["v_anc"][ar],
              "k_suf": t["k_suf"][sr], "v_suf": t["v_suf"][sr], **layout_tensors(sub, DEVICE)}
        o, l_ = run_cascade(heads, sub, ts)
        out[sr] = o
        lse[sr] = l_
    check_full(heads, lay, t, out, lse)
