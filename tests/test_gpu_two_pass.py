"""GPU parity of quail_cascade_attn_two_pass: the cascade run as an anchor pass (A2, fp32
normalised partial and its LSE), a suffix pass (A3) and the LSE merge (A4) - folded into
the suffix pass's epilogue or run as its own kernel - against the float64 oracle on every
output element of the edge layouts (bf16 and FP8 anchor KV), and at the full join size
on sampled suffixes. The two-pass result must also stay within the bf16 bounds of the
fused kernel's output on the same inputs."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.fp8 import dequantize_kv_fp8
from parity_util import (FP8_REL_L2, check_full, check_sampled, compare, fp8_max_abs, np64,
                         run_cascade)
from test_gpu_parity import EDGE_CASES

pytestmark = pytest.mark.gpu


def _inputs(layout, heads, seed):
    hq, hkv, d = heads
    cfg = workloads.AttnConfig("two_pass", layout.num_anchors, (0, 0), 0, (0, 0), hq, hkv, d,
                               False, seed)
    return workloads.make_attention_inputs(cfg, layout, "cuda")


def run_two_pass(heads, layout, t, merge_in_suffix_pass, kv_fp8=False, k_scale=None,
                 v_scale=None, with_lse=True):
    import prefill_only_cascade_gb300 as q
    hq, hkv, d = heads
    desc = q.make_desc(layout.num_anchors, layout.num_suffixes, layout.total_anchor_tokens,
                       layout.total_suffix_tokens, layout.max_anchor_len, layout.max_suffix_len,
                       hq, hkv, d, 0.0, kv_fp8)
    need = q.cascade_two_pass_workspace_size(desc)
    assert need >= q.cascade_workspace_size(desc) + 4 * layout.total_suffix_tokens * hq * (d + 2)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    out = torch.full((layout.total_suffix_tokens, hq, d), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    lse = torch.full((layout.total_suffix_tokens, hq), float("nan"), dtype=torch.float32,
                     device="cuda") if with_lse else None
    q.cascade_attn_two_pass(desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
                            t["anchor_offsets"], t["anchor_suffix_ptr"], t["suffix_offsets"],
                            out, lse, ws, k_scale, v_scale,
                            merge_in_suffix_pass=merge_in_suffix_pass)
    torch.cuda.synchronize()
    st = q.get_device_error()
    assert st == q.QUAIL_OK, q.status_string(st)
    return out, lse


def _edge(name):
    anchors, counts, lens, heads = EDGE_CASES[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    if isinstance(lens, tuple):
        lens = rng.integers(lens[0], lens[1] + 1, size=sum(counts))
    lay = workloads.layout_from_lengths(anchors, counts, lens)
    return lay, heads, _inputs(lay, heads, zlib.crc32(name.encode()) % 1000)


@pytest.mark.parametrize("merge", [True, False], ids=["merge_in_suffix_pass", "merge_kernel"])
@pytest.mark.parametrize("name", sorted(EDGE_CASES))
def test_two_pass_edge_layouts_every_element(name, merge):
    lay, heads, t = _edge(name)
    out, lse = run_two_pass(heads, lay, t, merge)
    figs = check_full(heads, lay, t, out, lse)
    fused_out, fused_lse = run_cascade(heads, lay, t)
    compare(np64(out), np64(lse), np64(fused_out), np64(fused_lse))
    print(name, merge, figs)


@pytest.mark.parametrize("merge", [True, False], ids=["merge_in_suffix_pass", "merge_kernel"])
def test_two_pass_without_lse(merge):
    lay, heads, t = _edge("mixed_gqa4")
    out, _ = run_two_pass(heads, lay, t, merge, with_lse=False)
    check_full(heads, lay, t, out, None)


@pytest.mark.parametrize("merge", [True, False], ids=["merge_in_suffix_pass", "merge_kernel"])
@pytest.mark.parametrize("d", [128, 64])
def test_two_pass_fp8_every_element(d, merge):
    import prefill_only_cascade_gb300 as q
    heads = (32, 8, d)
    rng = np.random.default_rng(41 + d)
    lay = workloads.layout_from_lengths([513, 0, 40, 129], [5, 2, 6, 3],
                                        rng.integers(1, 90, size=16))
    t = _inputs(lay, heads, 41)
    codes, scales, kv = {}, {}, []
    for name in ("k_anc", "v_anc"):
        c = torch.empty(t[name].shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(lay.num_anchors, 8, dtype=torch.float32, device="cuda")
        q.quantize_kv_fp8(t[name], t["anchor_offsets"], c, sc)
        codes[name], scales[name] = c, sc
        oc, os_ = oracle.quantize_kv_fp8(np64(t[name]).astype(np.float32), lay.anchor_offsets)
        kv.append(dequantize_kv_fp8(oc, os_, lay.anchor_offsets))
    t8 = dict(t, k_anc=codes["k_anc"], v_anc=codes["v_anc"])
    out, lse = run_two_pass(heads, lay, t8, merge, kv_fp8=True, k_scale=scales["k_anc"],
                            v_scale=scales["v_anc"])
    check_full(heads, lay, t8, out, lse, kv=tuple(kv), rel_bound=FP8_REL_L2,
               max_abs=fp8_max_abs(t["v_anc"]))


@pytest.mark.parametrize("merge", [True, False], ids=["merge_in_suffix_pass", "merge_kernel"])
def test_two_pass_join_full_size_sampled(merge):
    cfg = workloads.ATTN_CONFIGS["join"]
    lay = workloads.make_layout(cfg)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    heads = (cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim)
    out, lse = run_two_pass(heads, lay, t, merge)
    ids = workloads.sample_suffixes(lay, 48, cfg.seed)
    print("join two-pass", merge, check_sampled(heads, lay, t, out, lse, ids))
    del t, out, lse
    torch.cuda.empty_cache()


def test_two_pass_rejects_bad_arguments():
    import ctypes
    import prefill_only_cascade_gb300 as q
    lay, heads, t = _edge("gqa2")
    desc = q.make_desc(lay.num_anchors, lay.num_suffixes, lay.total_anchor_tokens,
                       lay.total_suffix_tokens, lay.max_anchor_len, lay.max_suffix_len, *heads)
    need = q.cascade_two_pass_workspace_size(desc)
    small = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty(lay.total_suffix_tokens, heads[0], heads[2], dtype=torch.bfloat16,
                      device="cuda")
    with pytest.raises(q.QuailError) as e:          # the fused kernel's workspace is too small
        q.cascade_attn_two_pass(desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"],
                                t["v_suf"], t["anchor_offsets"], t["anchor_suffix_ptr"],
                                t["suffix_offsets"], out, workspace=small)
    assert e.value.status == q.QUAIL_ERR_INVALID_ARG
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    st = q.lib.quail_cascade_attn_two_pass(
        ctypes.byref(desc), *(ctypes.c_void_p(x.data_ptr()) for x in (
            t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"], t["anchor_offsets"],
            t["anchor_suffix_ptr"], t["suffix_offsets"])), None, None, 2,
        ctypes.c_void_p(out.data_ptr()), None, ctypes.c_void_p(ws.data_ptr()),
        ctypes.c_size_t(need), None)
    assert st == q.QUAIL_ERR_INVALID_ARG            # merge flag other than 0 or 1
