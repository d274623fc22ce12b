"""Pins of the float64 CPU oracle against things other than itself (CPU only).

Each test checks the oracle against brute force, a closed form, an invariant, a library
routine (torch SDPA / rms_norm / float8_e4m3fn) or the OCP E4M3 definition, chosen so that
a dropped term, a wrong sign or index, or a transposed operand fails at least one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle.fp8 import dequantize_kv_fp8
from workloads import layout_from_lengths


def _rand(rng, *shape):
    return rng.standard_normal(shape)


def _brute_force(q, k_anc, v_anc, k_suf, v_suf, scale):
    """Pure-Python loops: one (token, head) at a time."""
    l, hq, d = q.shape
    la, hkv = k_anc.shape[0], k_anc.shape[1]
    group = hq // hkv
    out = np.zeros((l, hq, d))
    lse = np.zeros((l, hq))
    for i in range(l):
        for h in range(hq):
            g = h // group
            keys = [k_anc[j, g] for j in range(la)] + [k_suf[j, g] for j in range(i + 1)]
            vals = [v_anc[j, g] for j in range(la)] + [v_suf[j, g] for j in range(i + 1)]
            z = [scale * sum(float(q[i, h, c]) * float(kk[c]) for c in range(d)) for kk in keys]
            tot = math.fsum(math.exp(x) for x in z)
            lse[i, h] = math.log(tot)
            for j, vv in enumerate(vals):
                w = math.exp(z[j] - lse[i, h])
                for c in range(d):
                    out[i, h, c] += w * float(vv[c])
    return out, lse


@pytest.mark.parametrize("la,l,hq,hkv", [(5, 3, 4, 2), (0, 4, 2, 1), (7, 1, 4, 4), (3, 2, 8, 2)])
def test_attention_brute_force(la, l, hq, hkv):
    rng = np.random.default_rng(la * 100 + l)
    d = 6
    q, ka, va = _rand(rng, l, hq, d), _rand(rng, la, hkv, d), _rand(rng, la, hkv, d)
    ks, vs = _rand(rng, l, hkv, d), _rand(rng, l, hkv, d)
    scale = 1 / math.sqrt(d)
    o_ref, lse_ref = _brute_force(q, ka, va, ks, vs, scale)
    o, lse = oracle.suffix_attention(q, ka, va, ks, vs, scale)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_ragged_batch_matches_per_suffix_brute_force():
    rng = np.random.default_rng(7)
    lay = layout_from_lengths([3, 0, 5], [2, 1, 3], [2, 1, 3, 1, 4, 2])
    hq, hkv, d = 4, 2, 4
    T_A, T_S = lay.total_anchor_tokens, lay.total_suffix_tokens
    q, ks, vs = _rand(rng, T_S, hq, d), _rand(rng, T_S, hkv, d), _rand(rng, T_S, hkv, d)
    ka, va = _rand(rng, T_A, hkv, d), _rand(rng, T_A, hkv, d)
    out, lse = oracle.cascade_attention(q, ka, va, ks, vs, lay.anchor_offsets,
                                        lay.anchor_suffix_ptr, lay.suffix_offsets)
    ao, so = lay.anchor_offsets, lay.suffix_offsets
    for s in range(lay.num_suffixes):
        a = int(lay.suffix_anchor[s])
        r = slice(so[s], so[s + 1])
        o_ref, l_ref = _brute_force(q[r], ka[ao[a]:ao[a + 1]], va[ao[a]:ao[a + 1]], ks[r], vs[r],
                                    1 / math.sqrt(d))
        np.testing.assert_allclose(out[r], o_ref, atol=1e-12)
        np.testing.assert_allclose(lse[r], l_ref, atol=1e-12)


@pytest.mark.parametrize("la,l", [(0, 1), (0, 5), (1, 1), (9, 1), (16, 7), (64, 32)])
def test_cascade_merge_equals_monolithic(la, l):
    rng = np.random.default_rng(la + 31 * l)
    hq, hkv, d = 8, 2, 16
    q, ka, va = _rand(rng, l, hq, d) * 2, _rand(rng, la, hkv, d), _rand(rng, la, hkv, d)
    ks, vs = _rand(rng, l, hkv, d), _rand(rng, l, hkv, d)
    o1, l1 = oracle.suffix_attention(q, ka, va, ks, vs, 0.25)
    o2, l2 = oracle.cascade_suffix(q, ka, va, ks, vs, 0.25)
    np.testing.assert_allclose(o2, o1, atol=1e-12)
    np.testing.assert_allclose(l2, l1, atol=1e-12)
    oa, lsa = oracle.anchor_partial(q, ka, va, 0.25)
    if la == 0:
        assert np.all(np.isneginf(lsa)) and np.all(oa == 0)


def test_zero_query_gives_mean_of_visible_values():
    rng = np.random.default_rng(1)
    la, l, hq, hkv, d = 6, 4, 4, 2, 5
    q = np.zeros((l, hq, d))
    ka, va, ks, vs = (_rand(rng, n, hkv, d) for n in (la, la, l, l))
    o, lse = oracle.suffix_attention(q, ka, va, ks, vs, 0.3)
    for i in range(l):
        n = la + i + 1
        np.testing.assert_allclose(lse[i], np.log(n), atol=1e-13)
        for h in range(hq):
            g = h // (hq // hkv)
            mean = (va[:, g].sum(0) + vs[:i + 1, g].sum(0)) / n
            np.testing.assert_allclose(o[i, h], mean, atol=1e-13)


def test_single_visible_key_copies_value():
    rng = np.random.default_rng(2)
    hq, hkv, d = 4, 1, 8
    q, ks, vs = _rand(rng, 1, hq, d), _rand(rng, 1, hkv, d), _rand(rng, 1, hkv, d)
    empty = np.zeros((0, hkv, d))
    o, lse = oracle.suffix_attention(q, empty, empty, ks, vs, 0.7)
    for h in range(hq):
        np.testing.assert_allclose(o[0, h], vs[0, 0], atol=1e-14)
        np.testing.assert_allclose(lse[0, h], 0.7 * q[0, h] @ ks[0, 0], atol=1e-13)


def test_identical_queries_in_a_group_give_identical_outputs():
    rng = np.random.default_rng(3)
    hq, hkv, d, la, l = 8, 2, 8, 5, 3
    q = _rand(rng, l, hkv, d)[:, np.repeat(np.arange(hkv), hq // hkv), :]
    ka, va, ks, vs = (_rand(rng, n, hkv, d) for n in (la, la, l, l))
    o, lse = oracle.suffix_attention(q, ka, va, ks, vs, 0.3)
    for g in range(hkv):
        for h in range(g * 4, g * 4 + 4):
            np.testing.assert_array_equal(o[:, h], o[:, g * 4])
    assert not np.allclose(o[:, 0], o[:, 4])  # different KV heads differ


def test_anchor_row_permutation_invariance():
    rng = np.random.default_rng(4)
    hq, hkv, d, la, l = 4, 2, 8, 11, 4
    q, ka, va, ks, vs = (_rand(rng, *s) for s in
                         [(l, hq, d), (la, hkv, d), (la, hkv, d), (l, hkv, d), (l, hkv, d)])
    perm = rng.permutation(la)
    o1, l1 = oracle.suffix_attention(q, ka, va, ks, vs, 0.3)
    o2, l2 = oracle.suffix_attention(q, ka[perm], va[perm], ks, vs, 0.3)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(l2, l1, atol=1e-13)
    # but suffix order matters (causality): reversing the suffix changes the result
    o3, _ = oracle.suffix_attention(q, ka, va, ks[::-1], vs[::-1], 0.3)
    assert not np.allclose(o3, o1)


def test_dominant_anchor_key_selects_its_value():
    rng = np.random.default_rng(5)
    hq, hkv, d, la, l = 2, 1, 8, 6, 2
    q = _rand(rng, l, hq, d)
    ka, va, ks, vs = (_rand(rng, n, hkv, d) * 0.01 for n in (la, la, l, l))
    ka[3, 0] = 0
    va[3, 0] = _rand(rng, d)
    # key 3 aligned with every query direction: huge score
    ka[3, 0] = q.reshape(-1, d).sum(0) * 1e3
    o, _ = oracle.suffix_attention(q, ka, va, ks, vs, 1.0)
    for i in range(l):
        for h in range(hq):
            if q[i, h] @ ka[3, 0] > 50:
                np.testing.assert_allclose(o[i, h], va[3, 0], atol=1e-9)


def test_matches_library_sdpa_with_explicit_mask():
    """Reduction to a textbook routine: torch SDPA (float64, CPU) with a boolean mask over
    [anchor ; suffix] and torch's own GQA head mapping."""
    rng = np.random.default_rng(6)
    hq, hkv, d, la, l = 8, 2, 16, 13, 9
    q, ka, va, ks, vs = (_rand(rng, *s) for s in
                         [(l, hq, d), (la, hkv, d), (la, hkv, d), (l, hkv, d), (l, hkv, d)])
    scale = 1 / math.sqrt(d)
    o, lse = oracle.suffix_attention(q, ka, va, ks, vs, scale)
    K = torch.from_numpy(np.concatenate([ka, ks])).permute(1, 0, 2)[None]   # [1, Hkv, n, d]
    V = torch.from_numpy(np.concatenate([va, vs])).permute(1, 0, 2)[None]
    Q = torch.from_numpy(q).permute(1, 0, 2)[None]                          # [1, Hq, l, d]
    mask = torch.zeros(l, la + l, dtype=torch.bool)
    mask[:, :la] = True
    mask[:, la:] = torch.tril(torch.ones(l, l, dtype=torch.bool))
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale,
                                                           enable_gqa=True)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), atol=1e-12)
    Kx = K.repeat_interleave(hq // hkv, dim=1)
    z = (Q @ Kx.transpose(-1, -2)) * scale
    ref_lse = torch.logsumexp(z.masked_fill(~mask, float("-inf")), dim=-1)[0].T.numpy()
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


# ----------------------------------------------------------------------------- head

def test_rmsnorm_constant_row_closed_form():
    gamma = np.linspace(0.5, 1.5, 32)
    for c in (1e-3, 0.5, -3.0):
        y = oracle.rmsnorm(np.full((1, 32), c), gamma, 1e-6)
        np.testing.assert_allclose(y[0], c / np.sqrt(c * c + 1e-6) * gamma, rtol=1e-14)


def test_rmsnorm_unit_gamma_zero_eps_has_norm_sqrt_hidden():
    rng = np.random.default_rng(8)
    h = _rand(rng, 5, 48) * 3
    y = oracle.rmsnorm(h, np.ones(48), 0.0)
    np.testing.assert_allclose((y * y).sum(-1), 48.0, rtol=1e-13)


def test_rmsnorm_matches_library():
    rng = np.random.default_rng(9)
    h, gamma = _rand(rng, 7, 40), rng.uniform(0.5, 1.5, 40)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(h), (40,), torch.from_numpy(gamma), eps=1e-6)
    np.testing.assert_allclose(oracle.rmsnorm(h, gamma, 1e-6), ref.numpy(), rtol=1e-13)


def test_head_one_hot_columns_select_normalised_features():
    rng = np.random.default_rng(10)
    hidden = 24
    h, gamma = _rand(rng, 6, hidden), rng.uniform(0.5, 1.5, hidden)
    cols = [3, 0, 7, 11, 23, 5, 9, 1]
    w8 = np.zeros((8, hidden))
    w8[np.arange(8), cols] = 1.0
    logits, am = oracle.restricted_head(h, gamma, w8, 1e-6)
    y = oracle.rmsnorm(h, gamma, 1e-6)
    np.testing.assert_allclose(logits, y[:, cols], rtol=1e-14)
    np.testing.assert_array_equal(am, np.argmax(y[:, cols], -1))


def test_head_row_index_and_argmax_ties():
    hidden = 8
    h = np.eye(hidden)[:4] + 0.5
    w8 = np.zeros((8, hidden))
    w8[2] = w8[5] = 1.0          # columns 2 and 5 tie on every row
    logits, am = oracle.restricted_head(h, np.ones(hidden), w8, 1e-6, row_index=[3, 1])
    np.testing.assert_array_equal(am, [2, 2])   # lowest index among the maxima
    full, _ = oracle.restricted_head(h, np.ones(hidden), w8, 1e-6)
    np.testing.assert_array_equal(logits, full[[3, 1]])
    np.testing.assert_allclose(oracle.top2_margin(logits), 0.0)


# ----------------------------------------------------------------------------- fp8

def test_e4m3_known_points():
    # OCP 8-bit floating point specification, E4M3: bias 7, max normal 448 (S.1111.110),
    # min normal 2^-6, min subnormal 2^-9, NaN = S.1111.111, no infinities.
    dec = oracle.e4m3_decode
    assert dec(0x7E) == 448.0 and dec(0xFE) == -448.0
    assert dec(0x08) == 2.0 ** -6 and dec(0x01) == 2.0 ** -9 and dec(0x07) == 7 * 2.0 ** -9
    assert dec(0x38) == 1.0 and dec(0x39) == 1.125 and dec(0x40) == 2.0
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))
    assert dec(0x00) == 0.0 and dec(0x80) == 0.0 and np.signbit(dec(0x80))


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = oracle.e4m3_decode(codes)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(ours), nan)
    np.testing.assert_array_equal(ours[~nan], ref[~nan])


def test_e4m3_round_trip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes)), codes)


def test_e4m3_rounding_ties_and_saturation():
    enc = oracle.e4m3_encode
    assert enc(1.0625) == 0x38          # halfway 1.0 / 1.125 -> even code 0x38
    assert enc(1.1875) == 0x3A          # halfway 1.125 / 1.25 -> even code 0x3A
    assert enc(1.07) == 0x39
    assert enc(2.0 ** -10) == 0x00      # halfway 0 / 2^-9 -> 0
    assert enc(3 * 2.0 ** -10) == 0x02  # halfway 2^-9 / 2^-8 -> even code 0x02
    assert enc(1e6) == 0x7E and enc(-1e6) == 0xFE and enc(460.0) == 0x7E
    assert enc(-1e-9) == 0x80           # sign kept on underflow


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.standard_normal(20000) * 50, rng.standard_normal(2000) * 1e-2])
    x = x.astype(np.float32).astype(np.float64)
    x = x[np.abs(x) <= 448]
    ref = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(x), ref)


def test_quantize_kv_scales_and_error():
    rng = np.random.default_rng(12)
    ao = np.array([0, 5, 5, 17], dtype=np.int32)   # the middle anchor is empty
    kv = rng.standard_normal((17, 3, 16)).astype(np.float32)
    kv[5:17, 1] = 0.0                               # an all-zero (anchor, head) block
    codes, scales = oracle.quantize_kv_fp8(kv, ao)
    assert scales[1].tolist() == [1.0, 1.0, 1.0] and scales[2, 1] == 1.0
    assert np.all(codes[5:17, 1] == 0)
    np.testing.assert_allclose(scales[0, 0], np.abs(kv[0:5, 0]).max() / 448, rtol=1e-7)
    deq = dequantize_kv_fp8(codes, scales, ao)
    for a in (0, 2):
        for g in range(3):
            blk = slice(ao[a], ao[a + 1])
            amax = np.abs(kv[blk, g]).max()
            if amax == 0:
                continue
            j = np.unravel_index(np.argmax(np.abs(kv[blk, g])), kv[blk, g].shape)
            assert abs(oracle.e4m3_decode(codes[blk, g][j])) == 448.0
            err = np.abs(deq[blk, g] - kv[blk, g])
            # half an E4M3 step: relative 2^-4 for normals, absolute 2^-10 * scale below
            bound = np.maximum(np.abs(kv[blk, g]) * 2.0 ** -4, 2.0 ** -10 * scales[a, g])
            assert np.all(err <= bound * (1 + 1e-6))


# ----------------------------------------------------------------------------- tolerances

def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def test_tolerance_bounds_are_reachable_by_a_bf16_kernel():
    """Emulate a kernel that rounds what a tensor-core kernel rounds (fp32 scores, bf16 P,
    fp32 sums, bf16 output) on a tiny-workload-sized suffix and check the stated bounds:
    max abs <= 2e-2, relative L2 <= 5e-3, LSE abs <= 1e-3."""
    rng = np.random.default_rng(13)
    hq, hkv, d, la, l = 4, 1, 64, 64, 32
    q, ka, va, ks, vs = (_bf16(_rand(rng, *s)) for s in
                         [(l, hq, d), (la, hkv, d), (la, hkv, d), (l, hkv, d), (l, hkv, d)])
    scale = 1 / 8
    o_ref, lse_ref = oracle.suffix_attention(q, ka, va, ks, vs, scale)
    K = np.concatenate([ka, ks])[:, 0]
    V = np.concatenate([va, vs])[:, 0]
    o = np.zeros_like(o_ref)
    lse = np.zeros_like(lse_ref)
    for i in range(l):
        n = la + i + 1
        z = (q[i] @ K[:n].T).astype(np.float32) * np.float32(scale)    # [hq, n]
        m = z.max(-1, keepdims=True)
        p = np.exp2((z - m) * np.float32(np.log2(np.e))).astype(np.float32)
        lsum = p.sum(-1, dtype=np.float32)
        acc = (_bf16(p) @ V[:n]).astype(np.float32)
        o[i] = _bf16(acc / lsum[:, None])
        lse[i] = (m[:, 0] + np.log(lsum)).astype(np.float32)
    err = np.abs(o - o_ref)
    assert err.max() <= 2e-2
    assert np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref) <= 5e-3
    assert np.abs(lse - lse_ref).max() <= 1e-3
