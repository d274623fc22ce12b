"""GPU parity of the E4M3 quantisers against the oracle, bit for bit (codes and scales).

quail_quantize_kv_fp8 keeps each (anchor, KV head) slab on an 8-CTA cluster's chips up to
16 chunks of 32 rows per CTA (4,096 tokens) and reads longer anchors twice, in rounds;
the cases cover empty anchors, chunk and part edges (31, 32, 33, 255, 256, 257 rows),
both sides of the on-chip limit, 128- and 256-byte rows (one or two heads per slab), and
KV head counts that are not powers of two.
quail_quantize_kv_fp8_with_scales takes the amax; quail_causal_prefill_attn can emit it
(k_amax / v_amax) from the K/V tiles it loads, which must equal max |x| exactly and leave
the attention output unchanged."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import np64

pytestmark = pytest.mark.gpu


def _kv(lens, hkv, d, seed, scale=1.0):
    lay = workloads.layout_from_lengths(lens, [0] * len(lens), [])
    g = torch.Generator(device="cuda").manual_seed(seed)
    kv = (torch.randn(lay.total_anchor_tokens, hkv, d, generator=g, device="cuda") *
          scale).to(torch.bfloat16)
    # per-anchor magnitudes differ, so each slab has its own scale
    ao = lay.anchor_offsets
    for a in range(len(lens)):
        kv[int(ao[a]):int(ao[a + 1])] *= 2.0 ** (a % 7 - 3)
    return lay, kv, torch.from_numpy(ao.copy()).cuda()


def _check(kv, lay, codes, scale):
    ref_codes, ref_scale = oracle.quantize_kv_fp8(np64(kv).astype(np.float32),
                                                  lay.anchor_offsets)
    np.testing.assert_array_equal(scale.cpu().numpy(), ref_scale)
    got = codes.cpu().numpy()
    assert np.array_equal(got, ref_codes), f"{int((got != ref_codes).sum())} codes differ"


CASES = {
    # name: (anchor lengths, Hkv, d)
    "edges_h8_d128": ([0, 1, 31, 32, 33, 255, 256, 257, 0, 1000], 8, 128),
    "on_chip_limit_h8_d128": ([6144, 6145, 6400], 8, 128),
    "long_streamed_h2_d128": ([9001, 13], 2, 128),
    "h1_d64_128_byte_rows": ([5, 300, 12345, 64], 1, 64),
    "h2_d64_two_heads_per_slab": ([7, 2048, 513], 2, 64),
    "h4_d128": ([4096, 777, 1], 4, 128),
    # KV heads not a power of two: token rows of 48 16-byte vectors do not divide the
    # given-scale stream's 256 vectors per step (its general index path)
    "h6_d64_uneven_rows": ([100, 37, 2049], 6, 64),
    "h3_d128_uneven_rows": ([50, 0, 300], 3, 128),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_quantize_bit_exact(name):
    import prefill_only_cascade_gb300 as q
    lens, hkv, d = CASES[name]
    lay, kv, ao = _kv(lens, hkv, d, seed=len(name))
    codes = torch.full(kv.shape, 0xAB, dtype=torch.uint8, device="cuda")
    scale = torch.full((len(lens), hkv), float("nan"), dtype=torch.float32, device="cuda")
    q.quantize_kv_fp8(kv, ao, codes, scale)
    torch.cuda.synchronize()
    assert q.get_device_error() == q.QUAIL_OK
    _check(kv, lay, codes, scale)
    # the same with the amax given
    amax = torch.from_numpy(np.stack([
        np.abs(np64(kv[int(lay.anchor_offsets[a]):int(lay.anchor_offsets[a + 1])])).reshape(
            -1, hkv, d).max(axis=(0, 2)) if lens[a] else np.zeros(hkv)
        for a in range(len(lens))]).astype(np.float32)).cuda()
    codes2 = torch.full(kv.shape, 0xCD, dtype=torch.uint8, device="cuda")
    scale2 = torch.full_like(scale, float("nan"))
    q.quantize_kv_fp8_with_scales(kv, ao, amax, codes2, scale2)
    torch.cuda.synchronize()
    assert torch.equal(codes2, codes) and torch.equal(scale2, scale)


def test_quantize_anchors_without_tokens():
    import prefill_only_cascade_gb300 as q
    ao = torch.zeros(4, dtype=torch.int32, device="cuda")
    kv = torch.empty(0, 8, 128, dtype=torch.bfloat16, device="cuda")
    codes = torch.empty(0, 8, 128, dtype=torch.uint8, device="cuda")
    scale = torch.zeros(3, 8, dtype=torch.float32, device="cuda")
    q.quantize_kv_fp8(kv, ao, codes, scale)
    torch.cuda.synchronize()
    assert (scale == 1.0).all()


@pytest.mark.parametrize("heads", [(8, 2, 128), (16, 1, 64), (32, 8, 128)])
def test_causal_prefill_emits_kv_amax(heads):
    import prefill_only_cascade_gb300 as q
    hq, hkv, d = heads
    lens = [700, 1, 300, 64, 65, 129, 2000]
    lay = workloads.layout_from_lengths([0] * len(lens), [1] * len(lens), lens)
    cfg = workloads.AttnConfig("amax", len(lens), (0, 0), 1, (0, 0), hq, hkv, d, False, 5)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    # uneven magnitudes per sequence and head
    so = lay.suffix_offsets
    for s in range(len(lens)):
        for name in ("k_suf", "v_suf"):
            t[name][int(so[s]):int(so[s + 1])] *= 2.0 ** ((s + (name == "v_suf")) % 5 - 2)
    T, S = lay.total_suffix_tokens, len(lens)
    ws = torch.empty(q.causal_prefill_workspace_size(S, T, max(lens), hq, hkv, d),
                     dtype=torch.uint8, device="cuda")
    out = torch.empty(T, hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(T, hq, dtype=torch.float32, device="cuda")
    k_amax = torch.full((S, hkv), float("nan"), dtype=torch.float32, device="cuda")
    v_amax = torch.full_like(k_amax, float("nan"))
    q.causal_prefill_attn(t["q_suf"], t["k_suf"], t["v_suf"], t["suffix_offsets"], out,
                          max(lens), lse=lse, workspace=ws, k_amax=k_amax, v_amax=v_amax)
    torch.cuda.synchronize()
    assert q.get_device_error() == q.QUAIL_OK
    for name, am in (("k_suf", k_amax), ("v_suf", v_amax)):
        x = np64(t[name])
        ref = np.stack([np.abs(x[int(so[s]):int(so[s + 1])]).max(axis=(0, 2))
                        for s in range(S)]).astype(np.float32)
        np.testing.assert_array_equal(am.cpu().numpy(), ref)
    # the attention output is the same as without the amax
    out2, lse2 = torch.empty_like(out), torch.empty_like(lse)
    q.causal_prefill_attn(t["q_suf"], t["k_suf"], t["v_suf"], t["suffix_offsets"], out2,
                          max(lens), lse=lse2, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    # prefill amax -> quantise with those scales == the oracle's quantisation
    for name, am in (("k_suf", k_amax), ("v_suf", v_amax)):
        codes = torch.empty(t[name].shape, dtype=torch.uint8, device="cuda")
        scale = torch.empty(S, hkv, dtype=torch.float32, device="cuda")
        q.quantize_kv_fp8_with_scales(t[name], t["suffix_offsets"], am, codes, scale)
        torch.cuda.synchronize()
        _check(t[name], workloads.layout_from_lengths(lens, [0] * S, []), codes, scale)
