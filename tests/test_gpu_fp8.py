"""GPU parity of the FP8 (e4m3) anchor-KV cascade attention against the float64 oracle.

Anchor K/V are drawn in bf16 and quantised per (anchor, KV head) by
quail_quantize_kv_fp8; the oracle quantises the same bf16 values itself (bit-exact
agreement of the codes is checked too) and attends over the dequantised values
decode(code) * scale. Bounds: relative L2 <= 3e-2, the LSE bound of the bf16 path, and
max-abs <= 2e-2 + 2^-9 x the largest |V| (parity_util.fp8_max_abs)."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle.fp8 import dequantize_kv_fp8
from parity_util import FP8_REL_L2, check_full, check_sampled, fp8_max_abs, np64, run_cascade

pytestmark = pytest.mark.gpu


def _quantise(t, layout, hkv):
    import prefill_only_cascade_gb300 as q
    out = {}
    for name in ("k_anc", "v_anc"):
        codes = torch.empty(t[name].shape, dtype=torch.uint8, device="cuda")
        scale = torch.empty(layout.num_anchors, hkv, dtype=torch.float32, device="cuda")
        q.quantize_kv_fp8(t[name], t["anchor_offsets"], codes, scale)
        out[name] = (codes, scale)
    torch.cuda.synchronize()
    return out


def _oracle_kv(t, layout, name):
    codes, scales = oracle.quantize_kv_fp8(np64(t[name]).astype(np.float32), layout.anchor_offsets)
    return codes, scales, dequantize_kv_fp8(codes, scales, layout.anchor_offsets)


FP8_CASES = {
    "gqa4_mixed": ([0, 5, 130, 300, 256], [3, 0, 7, 2, 4], (0, 40), (8, 2)),
    "gqa4_qwen_heads": ([513, 40], [6, 9], (1, 96), (32, 8)),
    "mha": ([100, 257], [2, 3], [150, 1, 200, 30, 64], (2, 2)),
    "gqa8": ([128, 129, 1], [5, 5, 5], (1, 50), (16, 2)),
    "gqa16": ([64, 383], [9, 4], (1, 24), (16, 1)),
    "no_anchor_keys": ([0, 0], [3, 2], [5, 1, 17, 33, 2], (8, 2)),
    "d64_gqa4": ([0, 5, 130, 300, 256], [3, 0, 7, 2, 4], (0, 40), (8, 2), 64),
    "d64_gqa8_long": ([700, 129], [4, 6], (1, 90), (16, 2), 64),
}


@pytest.mark.parametrize("name", sorted(FP8_CASES))
def test_fp8_edge_layouts_every_element(name):
    anchors, counts, lens, (hq, hkv), *rest = FP8_CASES[name]
    d = rest[0] if rest else 128
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    if isinstance(lens, tuple):
        lens = rng.integers(lens[0], lens[1] + 1, size=sum(counts))
    lay = workloads.layout_from_lengths(anchors, counts, lens)
    cfg = workloads.AttnConfig("fp8case", lay.num_anchors, (0, 0), 0, (0, 0), hq, hkv, d,
                               True, 31)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    qz = _quantise(t, lay, hkv)
    kc, ks, kd = _oracle_kv(t, lay, "k_anc")
    vc, vs, vd = _oracle_kv(t, lay, "v_anc")
    np.testing.assert_array_equal(qz["k_anc"][0].cpu().numpy(), kc)
    np.testing.assert_array_equal(qz["v_anc"][1].cpu().numpy(), vs)
    t8 = dict(t, k_anc=qz["k_anc"][0], v_anc=qz["v_anc"][0])
    out, lse = run_cascade((hq, hkv, d), lay, t8, kv_fp8=True, k_scale=qz["k_anc"][1],
                           v_scale=qz["v_anc"][1])
    figs = check_full((hq, hkv, d), lay, t, out, lse, kv=(kd, vd), rel_bound=FP8_REL_L2,
                      max_abs=fp8_max_abs(t["v_anc"]))
    print(name, figs)


def test_fp8_full_size_workload_sampled_rows():
    cfg = workloads.ATTN_CONFIGS["fp8_long"]
    lay = workloads.make_layout(cfg)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    heads = (cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim)
    qz = _quantise(t, lay, cfg.num_kv_heads)
    t8 = dict(t, k_anc=qz["k_anc"][0], v_anc=qz["v_anc"][0])
    out, lse = run_cascade(heads, lay, t8, kv_fp8=True, k_scale=qz["k_anc"][1],
                           v_scale=qz["v_anc"][1])
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    ids = workloads.sample_suffixes(lay, 48, cfg.seed)
    ao = lay.anchor_offsets
    cache = {}

    def kv_for(a):
        # the oracle quantises this anchor's bf16 K/V itself and dequantises
        if a not in cache:
            r = slice(int(ao[a]), int(ao[a + 1]))
            pair = []
            for name in ("k_anc", "v_anc"):
                blk = np64(t[name][r]).astype(np.float32)
                codes, scales = oracle.quantize_kv_fp8(blk, np.array([0, r.stop - r.start]))
                pair.append(dequantize_kv_fp8(codes, scales, np.array([0, r.stop - r.start])))
            cache[a] = tuple(pair)
        return cache[a]

    figs = check_sampled(heads, lay, t, out, lse, ids, kv_override=kv_for, rel_bound=FP8_REL_L2,
                         max_abs=fp8_max_abs(t["v_anc"]))
    print("fp8_long", figs)
    del t, t8, out, lse, qz
    torch.cuda.empty_cache()


def test_fp8_missing_tile_times_out_cleanly():
    import prefill_only_cascade_gb300 as q
    lay = workloads.layout_from_lengths([300, 64], [5, 4], [3, 9, 27, 1, 16, 5, 5, 40, 2])
    cfg = workloads.AttnConfig("fp8to", 2, (0, 0), 0, (0, 0), 8, 2, 128, True, 5)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    qz = _quantise(t, lay, 2)
    t8 = dict(t, k_anc=qz["k_anc"][0], v_anc=qz["v_anc"][0])
    desc = q.make_desc(2, 9, lay.total_anchor_tokens, lay.total_suffix_tokens,
                       lay.max_anchor_len, lay.max_suffix_len, 8, 2, 128, 0.0, True)
    ws = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device="cuda")
    out = torch.empty(lay.total_suffix_tokens, 8, 128, dtype=torch.bfloat16, device="cuda")
    q.set_wait_timeout_ns(50_000_000)
    q.debug_inject(True)
    try:
        q.cascade_attn(desc, t8["q_suf"], t8["k_anc"], t8["v_anc"], t8["k_suf"], t8["v_suf"],
                       t8["anchor_offsets"], t8["anchor_suffix_ptr"], t8["suffix_offsets"], out,
                       None, ws, qz["k_anc"][1], qz["v_anc"][1])
        assert q.get_device_error() == q.QUAIL_ERR_TIMEOUT
    finally:
        q.debug_inject(False)
        q.set_wait_timeout_ns(0)
    out2, lse2 = run_cascade((8, 2, 128), lay, t8, kv_fp8=True, k_scale=qz["k_anc"][1],
                             v_scale=qz["v_anc"][1])
    kd = _oracle_kv(t, lay, "k_anc")[2]
    vd = _oracle_kv(t, lay, "v_anc")[2]
    check_full((8, 2, 128), lay, t, out2, lse2, kv=(kd, vd), rel_bound=FP8_REL_L2,
               max_abs=fp8_max_abs(t["v_anc"]))


@pytest.mark.parametrize("d", [128, 64])
def test_fp8_staged_anchor_copy_is_exact_for_every_code(d):
    """The attention reads the anchor codes widened to bf16 by the staging kernel: check
    that copy bit for bit against the oracle's decode, for all 256 codes (signed zeros,
    subnormals, the largest finite values and the two NaN codes). White-box: the two
    staged copies are the last 2 x T_A x Hkv x d x 2 bytes of the workspace (K, then V)."""
    hkv, hq = 2, 8
    lay = workloads.layout_from_lengths([512, 256], [1, 2], [8, 3, 5])
    cfg = workloads.AttnConfig("fp8stage", 2, (0, 0), 0, (0, 0), hq, hkv, d, True, 41)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    T_A = lay.total_anchor_tokens
    n = T_A * hkv * d
    k_codes = (torch.arange(n, dtype=torch.int64) % 256).to(torch.uint8).reshape(T_A, hkv, d)
    g = torch.Generator().manual_seed(41)
    v_codes = k_codes.flatten()[torch.randperm(n, generator=g)].reshape(T_A, hkv, d)
    ones = torch.ones(2, hkv, dtype=torch.float32, device="cuda")
    t8 = dict(t, k_anc=k_codes.cuda(), v_anc=v_codes.cuda())
    _, _, ws = run_cascade((hq, hkv, d), lay, t8, kv_fp8=True, k_scale=ones, v_scale=ones,
                           keep_ws=True)
    nbytes = n * 2
    staged = {"k": ws[ws.numel() - 2 * nbytes: ws.numel() - nbytes],
              "v": ws[ws.numel() - nbytes:]}
    for name, codes in (("k", k_codes), ("v", v_codes)):
        got = staged[name].view(torch.bfloat16).float().cpu().numpy().reshape(-1)
        ref = oracle.e4m3_decode(codes.numpy().reshape(-1))
        nan = np.isnan(ref)
        assert nan.sum() == 2 * n // 256                 # codes 0x7F and 0xFF
        np.testing.assert_array_equal(np.isnan(got), nan)
        np.testing.assert_array_equal(got[~nan], ref[~nan].astype(np.float32))
        # signed zeros: code 0x80 is -0
        neg_zero = codes.numpy().reshape(-1) == 0x80
        assert np.signbit(got[neg_zero]).all() and not np.signbit(got[codes.numpy().reshape(-1) == 0]).any()
