"""Bounded device-side waits: a KV-tile load that never arrives (host-side fault
injection: the producer skips issuing it) makes the consumer's wait run out; the launch
must end by itself and report QUAIL_ERR_TIMEOUT, and the context must stay usable."""
import pytest
import torch

import workloads
from parity_util import check_full, run_cascade

pytestmark = pytest.mark.gpu


def test_missing_load_times_out_cleanly_and_context_survives():
    import prefill_only_cascade_gb300 as q
    cfg = workloads.ATTN_CONFIGS["tiny"]
    lay = workloads.make_layout(cfg)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    heads = (cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim)
    desc = q.make_desc(lay.num_anchors, lay.num_suffixes, lay.total_anchor_tokens,
                       lay.total_suffix_tokens, lay.max_anchor_len, lay.max_suffix_len, *heads)
    ws = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty(lay.total_suffix_tokens, cfg.num_q_heads, cfg.head_dim,
                      dtype=torch.bfloat16, device="cuda")
    q.set_wait_timeout_ns(50_000_000)  # 50 ms
    q.debug_inject(True)
    try:
        q.cascade_attn(desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
                       t["anchor_offsets"], t["anchor_suffix_ptr"], t["suffix_offsets"], out,
                       None, ws)
        assert q.get_device_error() == q.QUAIL_ERR_TIMEOUT
    finally:
        q.debug_inject(False)
        q.set_wait_timeout_ns(0)
    assert q.get_device_error() == q.QUAIL_OK
    out2, lse2 = run_cascade(heads, lay, t)
    check_full(heads, lay, t, out2, lse2)


def test_missing_load_times_out_cleanly_on_cta_pairs():
    # the same on the CTA-pair kernel (forced): CTA 0 skips its half of the first K tile,
    # so its MMA warp's wait runs out; CTA 1's waits run out on their own. Both CTAs
    # exchange their abort state and let copies in flight land before they exit.
    import prefill_only_cascade_gb300 as q
    heads = (8, 2, 128)
    lay = workloads.layout_from_lengths([300, 5], [3, 2], [40, 7, 90, 12, 3])
    cfg = workloads.AttnConfig("pairs_timeout", lay.num_anchors, (0, 0), 0, (0, 0), *heads,
                               False, 5)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    desc = q.make_desc(lay.num_anchors, lay.num_suffixes, lay.total_anchor_tokens,
                       lay.total_suffix_tokens, lay.max_anchor_len, lay.max_suffix_len, *heads)
    ws = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty(lay.total_suffix_tokens, heads[0], heads[2], dtype=torch.bfloat16,
                      device="cuda")
    assert q.set_cta_pairs(q.CTA_PAIRS_ALWAYS) == q.QUAIL_OK
    q.set_wait_timeout_ns(50_000_000)  # 50 ms
    q.debug_inject(True)
    try:
        q.cascade_attn(desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
                       t["anchor_offsets"], t["anchor_suffix_ptr"], t["suffix_offsets"], out,
                       None, ws)
        assert q.get_device_error() == q.QUAIL_ERR_TIMEOUT
    finally:
        q.debug_inject(False)
        q.set_wait_timeout_ns(0)
    try:
        assert q.get_device_error() == q.QUAIL_OK
        out2, lse2 = run_cascade(heads, lay, t)  # the pair kernel again, without the fault
        check_full(heads, lay, t, out2, lse2)
    finally:
        q.set_cta_pairs(q.CTA_PAIRS_AUTO)
