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
        # the same kernels on the same inputs: any difference (e.g. stale scratch) is a bug
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_batches_beyond_the_scratch_array():
    import prefill_only_cascade_gb300 as q
    # 40M suffix tokens need far more than the fixed array: refused before any launch
    desc = q.make_desc(1, 1, 16, 40_000_000, 16, 40_000_000, 32, 8, 128)
    assert q.cascade_workspace_size(desc) > 64 * 1024 * 1024
    with pytest.raises(q.QuailError) as e:
        q.cascade_attn_noalloc(desc, *([None] * 8), out=None)
    assert e.value.status == q.QUAIL_ERR_UNSUPPORTED


def test_noalloc_fp8_stages_the_anchors_in_the_scratch_array():
    # FP8 anchor KV: the bf16 staging of the anchor codes also lives in the fixed array
    import numpy as np
    import prefill_only_cascade_gb300 as q
    heads = (32, 8, 128)
    rng = np.random.default_rng(78)
    lay, t = _case([300, 129, 0], [6, 4, 2], rng.integers(1, 40, size=12), heads, 23)
    codes, scales = {}, {}
    for name in ("k_anc", "v_anc"):
        c = torch.empty(t[name].shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(lay.num_anchors, 8, dtype=torch.float32, device="cuda")
        q.quantize_kv_fp8(t[name], t["anchor_offsets"], c, sc)
        codes[name], scales[name] = c, sc
    t8 = dict(t, k_anc=codes["k_anc"], v_anc=codes["v_anc"])
    ref_out, ref_lse = run_cascade(heads, lay, t8, kv_fp8=True, k_scale=scales["k_anc"],
                                   v_scale=scales["v_anc"])
    desc = q.make_desc(lay.num_anchors, lay.num_suffixes, lay.total_anchor_tokens,
                       lay.total_suffix_tokens, lay.max_anchor_len, lay.max_suffix_len,
                       *heads, 0.0, True)
    assert q.cascade_workspace_size(desc) <= 64 * 1024 * 1024
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    q.cascade_attn_noalloc(desc, t8["q_suf"], t8["k_anc"], t8["v_anc"], t8["k_suf"],
                           t8["v_suf"], t8["anchor_offsets"], t8["anchor_suffix_ptr"],
                           t8["suffix_offsets"], out, lse, scales["k_anc"], scales["v_anc"])
    torch.cuda.synchronize()
    assert q.get_device_error() == q.QUAIL_OK
    compare(np64(out), np64(lse), np64(ref_out), np64(ref_lse))
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
