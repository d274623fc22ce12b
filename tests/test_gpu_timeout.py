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
