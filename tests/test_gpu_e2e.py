"""GPU test of the end-to-end path through host buffers: the batch's inputs copied from
pinned host memory in anchor groups (two device buffer sets, copies on a second stream
overlapping the previous group's cascade and head calls) must give the same logits and
argmax for every suffix, and the same attention output, as one device-resident call."""
import sys
import os

import numpy as np
import pytest
import torch

import workloads

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv_fp8", [False, True])
def test_host_buffer_path_matches_resident_call(kv_fp8):
    import prefill_only_cascade_gb300 as q
    dev = torch.device("cuda", 0)
    cfg = workloads.AttnConfig("e2e_case", 12, (100, 900), 20, (4, 64), 32, 8, 128, kv_fp8, 21)
    lay = workloads.make_layout(cfg)
    t = workloads.make_attention_inputs(cfg, lay, dev)
    hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    k_scale = v_scale = None
    if kv_fp8:
        ka = torch.empty(t["k_anc"].shape, dtype=torch.uint8, device=dev)
        va = torch.empty_like(ka)
        k_scale = torch.empty(lay.num_anchors, hkv, dtype=torch.float32, device=dev)
        v_scale = torch.empty_like(k_scale)
        q.quantize_kv_fp8(t["k_anc"], t["anchor_offsets"], ka, k_scale)
        q.quantize_kv_fp8(t["v_anc"], t["anchor_offsets"], va, v_scale)
        t["k_anc"], t["v_anc"] = ka, va
    desc = q.make_desc(lay.num_anchors, lay.num_suffixes, lay.total_anchor_tokens,
                       lay.total_suffix_tokens, lay.max_anchor_len, lay.max_suffix_len,
                       hq, hkv, d, 0.0, kv_fp8)
    ws = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device=dev)
    out = torch.empty(lay.total_suffix_tokens, hq, d, dtype=torch.bfloat16, device=dev)
    hcfg = workloads.HEAD_CONFIGS["join_last_token"]
    hx = workloads.make_head_inputs(hcfg, dev, num_rows=lay.total_suffix_tokens)
    last = torch.from_numpy((lay.suffix_offsets[1:] - 1).astype(np.int32)).to(dev)
    logits = torch.empty(lay.num_suffixes, 8, dtype=torch.float32, device=dev)
    am = torch.empty(lay.num_suffixes, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()
    q.cascade_attn(desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
                   t["anchor_offsets"], t["anchor_suffix_ptr"], t["suffix_offsets"], out, None,
                   ws, k_scale, v_scale, stream=stream)
    q.restricted_head(hx["h"], hx["gamma"], hx["w8"], logits, am, eps=hcfg.eps, row_index=last,
                      stream=stream)
    torch.cuda.synchronize()
    assert q.get_device_error() == q.QUAIL_OK
    res = bench.run_e2e_chunked(q, cfg, lay, t, hx["h"], last, k_scale, v_scale, dev, stream,
                                1, steps=2, n_chunks=3, head_weights=(hx["gamma"], hx["w8"]),
                                check=(out, logits, am))
    print(res["vs_resident"], res["host_set_h2d_gbs"], res["anchor_groups"])
    assert res["anchor_groups"] == 3
    assert res["vs_resident"]["head_logits_argmax_identical"]
    assert res["vs_resident"]["last_group_attention_max_abs_diff"] == 0.0
