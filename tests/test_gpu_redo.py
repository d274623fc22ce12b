"""GPU parity of the exact recompute path.

The fast cascade kernel computes P = 2^(s c - m_ref) against a fixed reference m_ref, the
row max of the work item's first key tile (0 when the row sees no key of that tile), and
lists the item for the exact kernel when a valid row's sum of P leaves [2^-64, 2^32]
(with FP8 anchor KV also when the anchor's V scale is above 2^64). Seeded inputs whose
later tiles score far above the first one, rows whose first tile is empty and whose keys
score very low, or a huge V scale force that path, for all items or only some; every
output element is compared with the float64 oracle, and the workspace's redo counter
shows the exact kernel did run. Wide but ordinary logit ranges stay on the fast path."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.fp8 import dequantize_kv_fp8
from parity_util import (FP8_REL_L2, check_full, compare, fp8_max_abs, np64, redo_count,
                         run_cascade)

pytestmark = pytest.mark.gpu


def _case(anchors, counts, lens, heads, seed):
    rng = np.random.default_rng(seed)
    if isinstance(lens, tuple):
        lens = rng.integers(lens[0], lens[1] + 1, size=sum(counts))
    lay = workloads.layout_from_lengths(anchors, counts, lens)
    hq, hkv, d = heads
    cfg = workloads.AttnConfig("redo", lay.num_anchors, (0, 0), 0, (0, 0), hq, hkv, d, False,
                               seed)
    return lay, workloads.make_attention_inputs(cfg, lay, "cuda")


def test_normal_inputs_need_no_recompute():
    lay, t = _case([300, 40], [4, 3], (1, 40), (8, 2, 128), 3)
    out, lse, ws = run_cascade((8, 2, 128), lay, t, keep_ws=True)
    assert redo_count(ws) == 0
    check_full((8, 2, 128), lay, t, out, lse)


@pytest.mark.parametrize("heads", [(8, 2, 128), (16, 1, 64)])
def test_wide_logits_stay_on_the_fast_path(heads):
    # queries x 4: s c has a standard deviation of ~6 (log2 units); a later tile's row max
    # exceeds the first tile's by far less than 32, so nothing is recomputed (with the
    # fixed reference 0 of a plain fast kernel the largest P would pass 2^32 on some rows)
    lay, t = _case([300, 0, 129], [4, 2, 3], (1, 40), heads, 11)
    t["q_suf"] = (t["q_suf"].float() * 4).to(torch.bfloat16)
    out, lse, ws = run_cascade(heads, lay, t, keep_ws=True)
    assert redo_count(ws) == 0
    check_full(heads, lay, t, out, lse)


@pytest.mark.parametrize("heads", [(8, 2, 128), (16, 1, 64)])
def test_very_wide_logits_partly_recomputed(heads):
    # queries x 24: a standard deviation of ~35 in log2 units; rows whose later tiles
    # beat the first tile's max by more than 32 send their items to the exact kernel
    lay, t = _case([300, 0, 129], [4, 2, 3], (1, 40), heads, 11)
    t["q_suf"] = (t["q_suf"].float() * 24).to(torch.bfloat16)
    out, lse, ws = run_cascade(heads, lay, t, keep_ws=True)
    print("items recomputed:", redo_count(ws))
    check_full(heads, lay, t, out, lse)


@pytest.mark.parametrize("heads", [(8, 2, 128), (16, 1, 64)])
def test_later_tiles_far_above_the_first_every_item_recomputed(heads):
    # suffix keys x 40 (the last tiles of every item): their scores exceed the first
    # (anchor) tile's max by far more than 32 in log2 units
    lay, t = _case([300, 70, 129], [4, 2, 3], (2, 40), heads, 11)
    t["k_suf"] = (t["k_suf"].float() * 40).to(torch.bfloat16)
    out, lse, ws = run_cascade(heads, lay, t, keep_ws=True)
    assert redo_count(ws) > 0
    check_full(heads, lay, t, out, lse)


def test_one_anchor_recomputed_others_fast():
    lay, t = _case([200, 300, 150], [3, 3, 3], (2, 30), (8, 2, 128), 12)
    ao = lay.anchor_offsets
    # anchor 1's keys past its first tile x 40: only its items leave the bounds
    lo, hi = int(ao[1]) + 128, int(ao[2])
    t["k_anc"][lo:hi] = (t["k_anc"][lo:hi].float() * 40).to(torch.bfloat16)
    out, lse, ws = run_cascade((8, 2, 128), lay, t, keep_ws=True)
    # exactly anchor 1's items: 2 KV heads x ceil(tokens / 64) query-tile pairs (G = 4)
    so, asp = lay.suffix_offsets, lay.anchor_suffix_ptr
    ntok = int(so[asp[2]] - so[asp[1]])
    assert redo_count(ws) == 2 * ((ntok + 63) // 64)
    check_full((8, 2, 128), lay, t, out, lse)


def test_very_negative_scores_after_an_empty_first_tile_recomputed():
    # an empty anchor and a 200-token suffix followed by a 20-token one: the query tile
    # that holds the end of the first suffix and the start of the second has a 220-key
    # window, and the second suffix's rows see no key of its first tile (reference 0).
    # Their scores are all equal and very negative: keys v (|v| = 32), queries -0.75 v,
    # s c = -0.75 * 1024 * log2(e) / sqrt(128) ~ -98 < -64, so their sum of P falls
    # below 2^-64. (Uniformly low scores alone stay on the fast path: the first tile's
    # max is the reference.)
    lay, t = _case([0], [2], [200, 20], (8, 2, 128), 13)
    g = torch.Generator(device="cpu").manual_seed(13)
    v = torch.randn(128, generator=g)
    v = (v / v.norm() * 32).to(torch.bfloat16).to("cuda")
    t["k_suf"][200:] = v
    t["q_suf"][200:] = (-v.float() * 0.75).to(torch.bfloat16)
    out, lse, ws = run_cascade((8, 2, 128), lay, t, keep_ws=True)
    assert redo_count(ws) > 0
    check_full((8, 2, 128), lay, t, out, lse)


def test_uniformly_very_negative_scores_stay_fast():
    # every key v (|v| = 32), queries -0.75 v: all scores ~ -98 in log2 units; the first
    # tile's max is the reference, so every P is 1 and nothing is recomputed
    lay, t = _case([256], [4], (1, 20), (8, 2, 128), 13)
    g = torch.Generator(device="cpu").manual_seed(13)
    v = torch.randn(128, generator=g)
    v = (v / v.norm() * 32).to(torch.bfloat16).to("cuda")
    for name in ("k_anc", "k_suf"):
        t[name][:] = v
    t["q_suf"][:] = (-v.float() * 0.75).to(torch.bfloat16)
    out, lse, ws = run_cascade((8, 2, 128), lay, t, keep_ws=True)
    assert redo_count(ws) == 0
    check_full((8, 2, 128), lay, t, out, lse)


def _fp8_run(lay, t, heads):
    import prefill_only_cascade_gb300 as q
    hkv = heads[1]
    qz = {}
    for name in ("k_anc", "v_anc"):
        codes = torch.empty(t[name].shape, dtype=torch.uint8, device="cuda")
        scale = torch.empty(lay.num_anchors, hkv, dtype=torch.float32, device="cuda")
        q.quantize_kv_fp8(t[name], t["anchor_offsets"], codes, scale)
        qz[name] = (codes, scale)
    t8 = dict(t, k_anc=qz["k_anc"][0], v_anc=qz["v_anc"][0])
    return run_cascade(heads, lay, t8, kv_fp8=True, k_scale=qz["k_anc"][1],
                       v_scale=qz["v_anc"][1], keep_ws=True)


def _fp8_oracle_kv(t, lay):
    kv = []
    for name in ("k_anc", "v_anc"):
        codes, scales = oracle.quantize_kv_fp8(np64(t[name]).astype(np.float32),
                                               lay.anchor_offsets)
        kv.append(dequantize_kv_fp8(codes, scales, lay.anchor_offsets))
    return tuple(kv)


@pytest.mark.parametrize("d", [128, 64])
def test_fp8_large_logits_recomputed(d):
    lay, t = _case([513, 40], [6, 9], (2, 96), (32, 8, d), 14)
    # suffix keys (bf16) x 40: far above the first (e4m3 anchor) tile's max
    t["k_suf"] = (t["k_suf"].float() * 40).to(torch.bfloat16)
    out, lse, ws = _fp8_run(lay, t, (32, 8, d))
    assert redo_count(ws) > 0
    check_full((32, 8, d), lay, t, out, lse, kv=_fp8_oracle_kv(t, lay), rel_bound=FP8_REL_L2,
               max_abs=fp8_max_abs(t["v_anc"]))


def test_fp8_huge_v_scale_recomputed():
    # anchor and suffix V x 2^72 (exact in bf16; the codes are unchanged and v_scale grows
    # by 2^72, past 2^64): every item with anchor keys goes to the exact kernel, and the
    # output is 2^72 times the output for the unscaled V
    lay, t = _case([300, 0, 200], [4, 2, 3], (1, 40), (8, 2, 128), 15)
    big = dict(t)
    for name in ("v_anc", "v_suf"):
        big[name] = (t[name].float() * 2.0 ** 72).to(torch.bfloat16)
    out, lse, ws = _fp8_run(lay, big, (8, 2, 128))
    assert redo_count(ws) > 0
    k_anc, v_anc = _fp8_oracle_kv(t, lay)
    ref_out, ref_lse = oracle.cascade_attention(
        np64(t["q_suf"]), k_anc, v_anc, np64(t["k_suf"]), np64(t["v_suf"]),
        lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets, 1.0 / np.sqrt(128))
    compare(np64(out) / 2.0 ** 72, np64(lse), ref_out, ref_lse, rel_bound=FP8_REL_L2,
            max_abs=fp8_max_abs(t["v_anc"]))
