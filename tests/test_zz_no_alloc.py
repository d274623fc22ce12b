"""quail_cascade_attn_noalloc, the entry point for callers that may not allocate device
memory (fixed memory budgets, plugin hosts that pass only inputs and outputs): its output
must match the workspace entry point's, through the C ABI, on two calls in a row that
share the library's fixed scratch array. The second call uses a smaller batch, so any
state left in the array by the first call would show up as a mismatch.

Collected last on purpose (file name) so that a run that stops at its first failure has
already run every other test.
"""
import pytest
import torch

import workloads
from parity_util import compare, np64, run_cascade

pytestmark = pytest.mark.gpu


def _noalloc(heads, layout, t):
    import prefill_only_cascade_gb300 as q
    hq, hkv, d = heads
    desc = q.make_desc(layout.num_anchors, layout.num_suffixes, layout.total_anchor_tokens,
                       layout.total_suffix_tokens, layout.max_anchor_len, layout.max_suffix_len,
                       hq, hkv, d)
    out = torch.full((layout.total_suffix_tokens, hq, d), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((layout.total_suffix_tokens, hq), float("nan"), dtype=torch.float32,
                     device="cuda")
    q.cascade_attn_noalloc(desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
                           t["anchor_offsets"], t["anchor_suffix_ptr"], t["suffix_offsets"],
                           out, lse)
    torch.cuda.synchronize()
    assert q.get_device_error() == q.QUAIL_OK
    return out, lse


def _case(anchors, counts, lens, heads, seed):
    lay = workloads.layout_from_lengths(anchors, counts, lens)
    hq, hkv, d = heads
    cfg = workloads.AttnConfig("noalloc", lay.num_anchors, (0, 0), 0, (0, 0), hq, hkv, d,
                               False, seed)
    return lay, workloads.make_attention_inputs(cfg, lay, "cuda")


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    import numpy as np
    heads = (32, 8, 128)
    rng = np.random.default_rng(77)
    lay1, t1 = _case([1024, 300, 0, 129], [40, 25, 3, 30],
                     rng.integers(1, 40, size=98), heads, 21)
    lay2, t2 = _case([200, 64], [5, 4], rng.integers(1, 30, size=9), heads, 22)
    for lay, t in ((lay1, t1), (lay2, t2)):
        ref_out, ref_lse = run_cascade(heads, lay, t)
        out, lse = _noalloc(heads, lay, t)
        compare(np64(out), np64(lse), np64(ref_out), np64(ref_lse))


def test_noalloc_rejects_batches_beyond_the_scratch_array():
    import prefill_only_cascade_gb300 as q
    # 40M suffix tokens need far more than the fixed array: refused before any launch
    desc = q.make_desc(1, 1, 16, 40_000_000, 16, 40_000_000, 32, 8, 128)
    assert q.cascade_workspace_size(desc) > 64 * 1024 * 1024
    with pytest.raises(q.QuailError) as e:
        q.cascade_attn_noalloc(desc, *([None] * 8), out=None)
    assert e.value.status == q.QUAIL_ERR_UNSUPPORTED
