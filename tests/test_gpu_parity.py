"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Small layouts are compared on every output element; the full-size workloads are run at
their real sizes in the benchmark's launch configuration and compared on a seeded sample
of suffixes (always including the extreme anchor and suffix lengths).
"""
import math
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import (check_full, check_head, check_sampled, layout_tensors, np64,
                         run_cascade)

pytestmark = pytest.mark.gpu


def _inputs(layout, heads, seed, device="cuda"):
    hq, hkv, d = heads
    cfg = workloads.AttnConfig("case", layout.num_anchors, (0, 0), 0, (0, 0), hq, hkv, d, False,
                               seed)
    return workloads.make_attention_inputs(cfg, layout, device)


def test_tiny_workload_every_element():
    cfg = workloads.ATTN_CONFIGS["tiny"]
    lay = workloads.make_layout(cfg)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    heads = (cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim)
    out, lse = run_cascade(heads, lay, t)
    figs = check_full(heads, lay, t, out, lse)
    print("tiny", figs)


EDGE_CASES = {
    # name: (anchor lengths, suffixes per anchor, suffix lengths or (lo, hi), heads)
    "mixed_gqa4": ([0, 5, 130, 300, 256], [3, 0, 7, 2, 4], (0, 40), (8, 2, 128)),
    "mha_long_suffix": ([100, 257], [2, 3], [150, 1, 200, 30, 64], (2, 2, 64)),
    "gqa8_tile_edges": ([128, 129, 1], [5, 5, 5], (1, 50), (16, 2, 128)),
    "gqa16_d64": ([64, 383], [9, 4], (1, 24), (16, 1, 64)),
    "gqa2": ([77, 0, 12], [6, 2, 1], (1, 70), (4, 2, 128)),
    "no_anchor_keys": ([0, 0], [3, 2], [5, 1, 17, 33, 2], (8, 2, 128)),
    "single_token_suffixes": ([40, 1000], [40, 70], (1, 1), (32, 8, 128)),
    "one_suffix": ([513], [1], [97], (32, 8, 128)),
    # causal prefill: no anchor keys, one long sequence per anchor (shared suffix tiles)
    "causal_prefill": ([0, 0, 0], [1, 1, 1], [700, 1, 300], (8, 2, 128)),
    "causal_prefill_d64": ([0, 0], [1, 1], [513, 260], (16, 1, 64)),
}


@pytest.mark.parametrize("name", sorted(EDGE_CASES))
def test_edge_layouts_every_element(name):
    anchors, counts, lens, heads = EDGE_CASES[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    n = sum(counts)
    if isinstance(lens, tuple):
        lens = rng.integers(lens[0], lens[1] + 1, size=n)
    lay = workloads.layout_from_lengths(anchors, counts, lens)
    t = _inputs(lay, heads, seed=7)
    out, lse = run_cascade(heads, lay, t)
    figs = check_full(heads, lay, t, out, lse)
    print(name, figs)


def test_custom_softmax_scale_and_no_lse():
    lay = workloads.layout_from_lengths([200, 31], [4, 3], [10, 3, 25, 7, 1, 40, 8])
    heads = (8, 2, 128)
    t = _inputs(lay, heads, seed=9)
    out, _ = run_cascade(heads, lay, t, softmax_scale=0.05, with_lse=False)
    check_full(heads, lay, t, out, None, scale=0.05)


def test_empty_batch_is_a_no_op():
    lay = workloads.layout_from_lengths([10, 0], [0, 0], [])
    t = _inputs(lay, (8, 2, 128), seed=1)
    out, lse = run_cascade((8, 2, 128), lay, t)
    assert out.numel() == 0 and lse.numel() == 0


def test_inconsistent_offsets_are_reported_not_used():
    import prefill_only_cascade_gb300 as q
    lay = workloads.layout_from_lengths([16, 16], [2, 2], [3, 4, 5, 6])
    heads = (8, 2, 128)
    t = _inputs(lay, heads, seed=2)
    bad = t["suffix_offsets"].clone()
    bad[2] = 100  # not monotone, beyond the total
    desc = q.make_desc(2, 4, 32, 18, 16, 6, 8, 2, 128)
    ws = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.zeros(18, 8, 128, dtype=torch.bfloat16, device="cuda")
    q.cascade_attn(desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
                   t["anchor_offsets"], t["anchor_suffix_ptr"], bad, out, None, ws)
    assert q.get_device_error() == q.QUAIL_ERR_DEVICE_BOUNDS
    assert torch.count_nonzero(out) == 0   # no attention work ran
    assert q.get_device_error() == q.QUAIL_OK  # the word was cleared


@pytest.mark.parametrize("name", ["join", "ragged"])
def test_full_size_workload_sampled_rows(name):
    cfg = workloads.ATTN_CONFIGS[name]
    lay = workloads.make_layout(cfg)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    heads = (cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim)
    out, lse = run_cascade(heads, lay, t)
    # properties that hold at any size: every row written and finite; lse >= the log of the
    # number of... (lse >= max score, checked per sample by the oracle below)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    ids = workloads.sample_suffixes(lay, 64, cfg.seed)
    figs = check_sampled(heads, lay, t, out, lse, ids)
    print(name, figs)
    del t, out, lse
    torch.cuda.empty_cache()


# ----------------------------------------------------------------------------- head

def test_head_tiny_every_row_and_gather():
    cfg = workloads.HEAD_CONFIGS["tiny"]
    x = workloads.make_head_inputs(cfg, "cuda")
    n = x["h"].shape[0]
    logits = torch.empty(n, 8, dtype=torch.float32, device="cuda")
    am = torch.empty(n, dtype=torch.int32, device="cuda")
    import prefill_only_cascade_gb300 as q
    q.restricted_head(x["h"], x["gamma"], x["w8"], logits, am, eps=cfg.eps)
    torch.cuda.synchronize()
    print("head tiny", check_head(x["h"], x["gamma"], x["w8"], cfg.eps, logits, am))
    # gather: the last token of each of 64 suffixes of 32 tokens
    idx = torch.arange(31, 64 * 32, 32, dtype=torch.int32, device="cuda") % n
    lg2 = torch.empty(64, 8, dtype=torch.float32, device="cuda")
    am2 = torch.empty(64, dtype=torch.int32, device="cuda")
    q.restricted_head(x["h"], x["gamma"], x["w8"], lg2, am2, eps=cfg.eps, row_index=idx)
    torch.cuda.synchronize()
    check_head(x["h"], x["gamma"], x["w8"], cfg.eps, lg2, am2, row_index=idx)


def test_head_out_of_range_gather_index_is_reported_not_read():
    # indices -1 and h_rows are checked on the device: those rows get NaN logits and
    # argmax -1 and the call reports QUAIL_ERR_DEVICE_BOUNDS; the other rows are exact
    import prefill_only_cascade_gb300 as q
    cfg = workloads.HEAD_CONFIGS["tiny"]
    x = workloads.make_head_inputs(cfg, "cuda", num_rows=100)
    idx = torch.tensor([0, 5, -1, 99, 100, 7, 2**31 - 1, 42], dtype=torch.int32, device="cuda")
    logits = torch.zeros(8, 8, dtype=torch.float32, device="cuda")
    am = torch.zeros(8, dtype=torch.int32, device="cuda")
    q.restricted_head(x["h"], x["gamma"], x["w8"], logits, am, eps=cfg.eps, row_index=idx)
    assert q.get_device_error() == q.QUAIL_ERR_DEVICE_BOUNDS
    assert q.get_device_error() == q.QUAIL_OK          # reading the word clears it
    bad = np.array([False, False, True, False, True, False, True, False])
    lg, a = logits.cpu().numpy(), am.cpu().numpy()
    assert np.isnan(lg[bad]).all() and (a[bad] == -1).all()
    good = torch.from_numpy(np.flatnonzero(~bad)).cuda()
    check_head(x["h"], x["gamma"], x["w8"], cfg.eps, logits[good], am[good],
               row_index=idx[good])


def test_head_ragged_row_count_and_strided_rows():
    import prefill_only_cascade_gb300 as q
    g = torch.Generator(device="cuda").manual_seed(5)
    base = torch.randn(37, 512 + 64, generator=g, device="cuda").to(torch.bfloat16)
    h = base[:, :512]  # row stride 576 elements
    gamma = (torch.rand(512, generator=g, device="cuda") + 0.5).to(torch.bfloat16)
    w8 = (torch.randn(8, 512, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    logits = torch.empty(37, 8, dtype=torch.float32, device="cuda")
    am = torch.empty(37, dtype=torch.int32, device="cuda")
    q.restricted_head(h, gamma, w8, logits, am, eps=1e-6)
    torch.cuda.synchronize()
    check_head(h, gamma, w8, 1e-6, logits, am)


def test_head_full_size_sampled_rows():
    import prefill_only_cascade_gb300 as q
    cfg = workloads.HEAD_CONFIGS["head"]
    x = workloads.make_head_inputs(cfg, "cuda")
    n = cfg.num_rows
    logits = torch.empty(n, 8, dtype=torch.float32, device="cuda")
    am = torch.empty(n, dtype=torch.int32, device="cuda")
    q.restricted_head(x["h"], x["gamma"], x["w8"], logits, am, eps=cfg.eps)
    torch.cuda.synchronize()
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 8192)]))
    ridx = torch.from_numpy(rows).cuda()
    print("head full", check_head(x["h"][ridx], x["gamma"], x["w8"], cfg.eps, logits[ridx],
                                  am[ridx]))
    del x, logits, am
    torch.cuda.empty_cache()


# ----------------------------------------------------------------------------- fp8

def test_quantizer_bit_exact_small():
    import prefill_only_cascade_gb300 as q
    lay = workloads.layout_from_lengths([5, 0, 37, 128, 1], [0] * 5, [])
    g = torch.Generator(device="cuda").manual_seed(11)
    for d in (64, 128):
        kv = (torch.randn(lay.total_anchor_tokens, 3, d, generator=g, device="cuda") * 3).to(
            torch.bfloat16)
        kv[42:170, 1] = 0            # an all-zero (anchor, head) block
        kv[0, 0, 0] = -1e-30         # a value that rounds to a signed zero
        codes = torch.empty(kv.shape, dtype=torch.uint8, device="cuda")
        scale = torch.empty(5, 3, dtype=torch.float32, device="cuda")
        ao = torch.from_numpy(lay.anchor_offsets.copy()).cuda()
        q.quantize_kv_fp8(kv, ao, codes, scale)
        torch.cuda.synchronize()
        ref_codes, ref_scale = oracle.quantize_kv_fp8(np64(kv).astype(np.float32), lay.anchor_offsets)
        np.testing.assert_array_equal(scale.cpu().numpy(), ref_scale)
        np.testing.assert_array_equal(codes.cpu().numpy(), ref_codes)


@pytest.mark.parametrize("d,anchors", [(128, [4100, 3, 4096]), (64, [8300, 8192, 0])])
def test_quantizer_long_slices_bit_exact(d, anchors):
    # a cluster keeps 65,536 16-byte vectors of one (anchor, head) in registers: 4,096 rows
    # at d = 128, 8,192 at d = 64; longer slices are read twice
    import prefill_only_cascade_gb300 as q
    lay = workloads.layout_from_lengths(anchors, [0] * len(anchors), [])
    g = torch.Generator(device="cuda").manual_seed(5 + d)
    kv = (torch.randn(lay.total_anchor_tokens, 2, d, generator=g, device="cuda") * 2).to(
        torch.bfloat16)
    kv[int(lay.anchor_offsets[1]) - 1, 1, 3] = 300.0   # the max sits in the last row
    codes = torch.empty(kv.shape, dtype=torch.uint8, device="cuda")
    scale = torch.empty(len(anchors), 2, dtype=torch.float32, device="cuda")
    ao = torch.from_numpy(lay.anchor_offsets.copy()).cuda()
    q.quantize_kv_fp8(kv, ao, codes, scale)
    torch.cuda.synchronize()
    ref_codes, ref_scale = oracle.quantize_kv_fp8(np64(kv).astype(np.float32), lay.anchor_offsets)
    np.testing.assert_array_equal(scale.cpu().numpy(), ref_scale)
    np.testing.assert_array_equal(codes.cpu().numpy(), ref_codes)


def test_quantizer_full_size_scales_and_sampled_codes():
    import prefill_only_cascade_gb300 as q
    cfg = workloads.ATTN_CONFIGS["fp8_long"]
    lay = workloads.make_layout(cfg)
    g = torch.Generator(device="cuda").manual_seed(4)
    kv = workloads._randn_bf16((lay.total_anchor_tokens, cfg.num_kv_heads, cfg.head_dim), g, "cuda")
    codes = torch.empty(kv.shape, dtype=torch.uint8, device="cuda")
    scale = torch.empty(cfg.num_anchors, cfg.num_kv_heads, dtype=torch.float32, device="cuda")
    ao = torch.from_numpy(lay.anchor_offsets.copy()).cuda()
    q.quantize_kv_fp8(kv, ao, codes, scale)
    torch.cuda.synchronize()
    for a in (0, 17, cfg.num_anchors - 1):
        r = slice(int(lay.anchor_offsets[a]), int(lay.anchor_offsets[a + 1]))
        rc, rs = oracle.quantize_kv_fp8(np64(kv[r]).astype(np.float32),
                                        np.array([0, r.stop - r.start]))
        np.testing.assert_array_equal(scale[a].cpu().numpy(), rs[0])
        np.testing.assert_array_equal(codes[r].cpu().numpy(), rc)
