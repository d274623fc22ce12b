"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI and
compare with the float64 oracle under the stated tolerances."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import workloads

# Bounds (bf16 outputs): max |gpu - ref| <= 2e-2 and ||gpu - ref|| / ||ref|| <= 5e-3;
# LSE absolute <= 1e-3; FP8 KV relative L2 <= 3e-2 (max-abs: see fp8_max_abs); argmax
# exact where the oracle's top-2 margin > 1e-2.
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
LSE_ABS = 1e-3
FP8_REL_L2 = 3e-2
ARGMAX_MARGIN = 1e-2


def fp8_max_abs(v_anc):
    """Max-abs bound of the FP8 anchor-KV path (only its relative L2 bound is stated):
    the bf16 bound plus one more bf16 rounding (relative 2^-9) of the largest anchor
    value, since the anchor tiles' P carries v_scale (P * v_scale is rounded to bf16,
    where the bf16 path's dominant P = 1 is exact). v_anc: the anchor V before
    quantisation (its largest |value| is the largest amax)."""
    if v_anc.numel() == 0:
        return BF16_MAX_ABS
    return BF16_MAX_ABS + float(v_anc.abs().max()) * 2.0 ** -9


def layout_tensors(layout, device="cuda"):
    return {k: torch.from_numpy(getattr(layout, k).copy()).to(device)
            for k in ("anchor_offsets", "anchor_suffix_ptr", "suffix_offsets")}


def run_cascade(cfg_heads, layout, t, kv_fp8=False, k_scale=None, v_scale=None,
                softmax_scale=0.0, with_lse=True, keep_ws=False):
    """Call quail_cascade_attn on device tensors `t` (keys as in workloads). With keep_ws
    the workspace is returned too (its int32 at byte 4 counts the work items the fast
    kernel handed to the exact one)."""
    import prefill_only_cascade_gb300 as q
    hq, hkv, d = cfg_heads
    dev = t["q_suf"].device
    desc = q.make_desc(layout.num_anchors, layout.num_suffixes, layout.total_anchor_tokens,
                       layout.total_suffix_tokens, layout.max_anchor_len, layout.max_suffix_len,
                       hq, hkv, d, softmax_scale, kv_fp8)
    ws = torch.empty(max(q.cascade_workspace_size(desc), 16), dtype=torch.uint8, device=dev)
    out = torch.full((layout.total_suffix_tokens, hq, d), float("nan"), dtype=torch.bfloat16,
                     device=dev)
    lse = torch.full((layout.total_suffix_tokens, hq), float("nan"), dtype=torch.float32,
                     device=dev) if with_lse else None
    q.cascade_attn(desc, t["q_suf"], t.get("k_anc"), t.get("v_anc"), t["k_suf"], t["v_suf"],
                   t["anchor_offsets"], t["anchor_suffix_ptr"], t["suffix_offsets"], out, lse,
                   ws, k_scale, v_scale)
    torch.cuda.synchronize()
    st = q.get_device_error()
    assert st == q.QUAIL_OK, q.status_string(st)
    if keep_ws:
        return out, lse, ws
    return out, lse


def redo_count(ws):
    """Work items the fast kernel listed for the exact kernel in the last call."""
    return int(ws[4:8].view(torch.int32).item())


def np64(x):
    return x.detach().to("cpu", torch.float64).numpy()


def compare(out_gpu, lse_gpu, out_ref, lse_ref, rel_bound=BF16_REL_L2, max_abs=BF16_MAX_ABS):
    """Element-wise comparison; returns the error figures and asserts the bounds."""
    err = np.abs(out_gpu - out_ref)
    assert np.isfinite(out_gpu).all(), "non-finite output"
    rel = float(np.linalg.norm(out_gpu - out_ref) / max(np.linalg.norm(out_ref), 1e-30))
    figures = {"max_abs": float(err.max()) if err.size else 0.0, "rel_l2": rel}
    if lse_gpu is not None:
        figures["lse_abs"] = float(np.abs(lse_gpu - lse_ref).max()) if lse_ref.size else 0.0
    assert figures["max_abs"] <= max_abs, figures
    assert rel <= rel_bound, figures
    if lse_gpu is not None:
        assert figures["lse_abs"] <= LSE_ABS, figures
    return figures


def check_full(cfg_heads, layout, t, out, lse, scale=None, kv=None, rel_bound=BF16_REL_L2,
               max_abs=BF16_MAX_ABS):
    """Compare every output row with the oracle (small layouts only)."""
    hq, hkv, d = cfg_heads
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    k_anc, v_anc = kv if kv is not None else (np64(t["k_anc"]), np64(t["v_anc"]))
    ref_out, ref_lse = oracle.cascade_attention(
        np64(t["q_suf"]), k_anc, v_anc, np64(t["k_suf"]), np64(t["v_suf"]),
        layout.anchor_offsets, layout.anchor_suffix_ptr, layout.suffix_offsets, scale)
    return compare(np64(out), None if lse is None else np64(lse), ref_out,
                   None if lse is None else ref_lse, rel_bound=rel_bound, max_abs=max_abs)


def check_sampled(cfg_heads, layout, t, out, lse, suffix_ids, scale=None, kv_override=None,
                  rel_bound=BF16_REL_L2, max_abs=BF16_MAX_ABS):
    """Compare the rows of sampled suffixes with the oracle, one suffix at a time.
    kv_override(anchor) -> (k_anc, v_anc) float64 arrays replaces the anchor K/V (FP8)."""
    hq, hkv, d = cfg_heads
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    cases = workloads.gather_suffix_case(t, layout, suffix_ids)
    outs_g, outs_r, lses_g, lses_r = [], [], [], []
    for s, c in cases.items():
        r0, r1 = c["rows"]
        if r1 == r0:
            continue
        if kv_override is not None:
            ka, va = kv_override(c["anchor"])
        else:
            ka, va = c["k_anc"], c["v_anc"]
        o, l_ = oracle.suffix_attention(c["q_suf"], ka, va, c["k_suf"], c["v_suf"], scale)
        outs_r.append(o)
        lses_r.append(l_)
        outs_g.append(np64(out[r0:r1]))
        lses_g.append(np64(lse[r0:r1]))
    return compare(np.concatenate(outs_g), np.concatenate(lses_g), np.concatenate(outs_r),
                   np.concatenate(lses_r), rel_bound=rel_bound, max_abs=max_abs)


def check_head(h, gamma, w8, eps, logits, argmax, row_index=None):
    ref_logits, ref_arg = oracle.restricted_head(np64(h), np64(gamma), np64(w8), eps,
                                                 None if row_index is None else
                                                 row_index.cpu().numpy())
    lg = np64(logits)
    figs = compare(lg, None, ref_logits, None)
    margin = oracle.top2_margin(ref_logits)
    sure = margin > ARGMAX_MARGIN
    got = argmax.cpu().numpy()
    assert np.array_equal(got[sure], ref_arg[sure]), "argmax mismatch above the margin"
    # where the margin is small the kernel's pick must still be a (near-)maximum
    best = ref_logits.max(-1)
    picked = ref_logits[np.arange(len(got)), got]
    assert np.all(best - picked <= ARGMAX_MARGIN + 1e-9)
    figs["argmax_checked"] = int(sure.sum())
    return figs
