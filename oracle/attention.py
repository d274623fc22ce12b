"""Oracle for the simplified cascade attention (float64, numpy, CPU). Test infrastructure.

Definition followed: [P1] "Motor de inferência Quail atinge 1 bilhão de tokens por minuto
por GPU", section "Como funciona", cascade-attention bullet: for a join, the suffix
tokens attend to the anchor (cross-attention) and then to themselves, and the two
results are combined by LSE rescaling. With the prompt of the AI.IF example on "Quail:
یک میلیارد توکن در دقیقه روی یک GPU" (a shared anchor text followed by the per-pair
text), this is exactly causal softmax attention over the concatenated prompt
[anchor ; suffix], restricted to the suffix rows: every anchor key is visible, and suffix
token i sees suffix tokens 0..i of its own suffix only.

`suffix_attention` is that plain definition. `anchor_partial`, `suffix_partial` and
`lse_merge` are the three cascade steps written separately; the tests check that they
reproduce the plain definition (the cascade is exact up to rounding).
"""
from __future__ import annotations

import numpy as np


def _expand_kv(kv: np.ndarray, num_q_heads: int) -> np.ndarray:
    """[L, Hkv, d] -> [L, Hq, d]: query head h reads KV head h // (Hq / Hkv)."""
    hkv = kv.shape[1]
    if num_q_heads % hkv:
        raise ValueError("num_q_heads must be a multiple of num_kv_heads")
    group = num_q_heads // hkv
    return kv[:, np.arange(num_q_heads) // group, :]


def _scores(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """q [l, H, d], k [n, H, d] -> z [H, l, n] with z[h, i, j] = <q[i, h], k[j, h]>."""
    return np.matmul(q.transpose(1, 0, 2), k.transpose(1, 2, 0))


def _softmax_attend(z: np.ndarray, v: np.ndarray):
    """z [H, l, n] scores with -inf for hidden keys, v [n, H, d] -> out [l, H, d], lse [l, H].

    lse = log(sum_j exp(z_j)) (natural log), out = sum_j exp(z_j - lse) v_j. A row with no
    visible key has lse = -inf and out = 0.
    """
    m = np.max(z, axis=-1, keepdims=True) if z.shape[-1] else np.full(z.shape[:-1] + (1,), -np.inf)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(z - m_safe)
    s = e.sum(axis=-1, keepdims=True)
    with np.errstate(divide="ignore"):
        lse = (np.log(s) + m_safe)[..., 0]
        w = np.where(s > 0, e / np.where(s > 0, s, 1.0), 0.0)
    out = np.matmul(w, v.transpose(1, 0, 2)).transpose(1, 0, 2)  # sum_j w[h,i,j] v[j,h,:]
    return out, lse.T


def suffix_attention(q, k_anc, v_anc, k_suf, v_suf, scale):
    """Monolithic attention of one suffix over [anchor ; suffix].

    q [l, Hq, d]; k_anc, v_anc [L_a, Hkv, d]; k_suf, v_suf [l, Hkv, d]. Returns
    out [l, Hq, d] and lse [l, Hq] in float64.
    """
    q = np.asarray(q, np.float64)
    l, hq, _ = q.shape
    la = k_anc.shape[0]
    k = _expand_kv(np.concatenate([np.asarray(k_anc, np.float64), np.asarray(k_suf, np.float64)]), hq)
    v = _expand_kv(np.concatenate([np.asarray(v_anc, np.float64), np.asarray(v_suf, np.float64)]), hq)
    z = scale * _scores(q, k)
    visible = np.zeros((l, la + l), dtype=bool)
    visible[:, :la] = True
    visible[:, la:] = np.tril(np.ones((l, l), dtype=bool))
    z = np.where(visible[None], z, -np.inf)
    return _softmax_attend(z, v)


def anchor_partial(q, k_anc, v_anc, scale):
    """Cascade step 1: non-causal cross-attention of the suffix queries to the anchor.
    With an empty anchor the partial is out = 0, lse = -inf."""
    q = np.asarray(q, np.float64)
    hq = q.shape[1]
    k = _expand_kv(np.asarray(k_anc, np.float64), hq)
    v = _expand_kv(np.asarray(v_anc, np.float64), hq)
    z = scale * _scores(q, k)
    return _softmax_attend(z, v)


def suffix_partial(q, k_suf, v_suf, scale):
    """Cascade step 2: causal self-attention of the suffix over its own tokens."""
    q = np.asarray(q, np.float64)
    l, hq, _ = q.shape
    k = _expand_kv(np.asarray(k_suf, np.float64), hq)
    v = _expand_kv(np.asarray(v_suf, np.float64), hq)
    z = scale * _scores(q, k)
    z = np.where(np.tril(np.ones((l, l), dtype=bool))[None], z, -np.inf)
    return _softmax_attend(z, v)


def lse_merge(out_a, lse_a, out_s, lse_s):
    """Cascade step 3: combine two softmax partials by LSE rescaling.

    lse = log(e^lse_a + e^lse_s); out = e^(lse_a - lse) out_a + e^(lse_s - lse) out_s.
    """
    lse = np.logaddexp(lse_a, lse_s)
    fin = np.isfinite(lse)
    wa = np.where(fin, np.exp(np.where(fin, lse_a - lse, -np.inf)), 0.0)
    ws = np.where(fin, np.exp(np.where(fin, lse_s - lse, -np.inf)), 0.0)
    return wa[..., None] * out_a + ws[..., None] * out_s, lse


def cascade_suffix(q, k_anc, v_anc, k_suf, v_suf, scale):
    """The three cascade steps in order for one suffix."""
    oa, la = anchor_partial(q, k_anc, v_anc, scale)
    os_, ls = suffix_partial(q, k_suf, v_suf, scale)
    return lse_merge(oa, la, os_, ls)


def cascade_attention(q_suf, k_anc, v_anc, k_suf, v_suf, anchor_offsets, anchor_suffix_ptr,
                      suffix_offsets, scale=None, suffix_ids=None):
    """Plain definition over a whole ragged batch (or over the listed suffixes).

    Arrays are numpy (bf16 inputs already widened). Returns (out [T_S, Hq, d],
    lse [T_S, Hq]) with NaN in rows of suffixes that were not requested.
    """
    q_suf = np.asarray(q_suf, np.float64)
    T_S, hq, d = q_suf.shape
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    ao = np.asarray(anchor_offsets, np.int64)
    asp = np.asarray(anchor_suffix_ptr, np.int64)
    so = np.asarray(suffix_offsets, np.int64)
    S = so.size - 1
    ids = range(S) if suffix_ids is None else suffix_ids
    out = np.full((T_S, hq, d), np.nan)
    lse = np.full((T_S, hq), np.nan)
    for s in ids:
        a = int(np.searchsorted(asp, s, side="right") - 1)
        r0, r1 = so[s], so[s + 1]
        if r1 == r0:
            continue
        o, l_ = suffix_attention(q_suf[r0:r1], k_anc[ao[a]:ao[a + 1]], v_anc[ao[a]:ao[a + 1]],
                                 k_suf[r0:r1], v_suf[r0:r1], scale)
        out[r0:r1], lse[r0:r1] = o, l_
    return out, lse
