"""Oracle for the FP8 (E4M3) anchor KV format. Test infrastructure.

The pages say only that the model runs in FP8 ("qwen3-4b-fp8" in the key points of
"Quail: یک میلیارد توکن در دقیقه روی یک GPU"; "Qwen3 4B FP8" on the BIO-4 paragraph of
"Quail, il motore di inferenza che supera il miliardo di token al minuto su una H100").
Reading taken: OCP 8-bit floating point, E4M3FN variant (exponent bias 7, no infinities,
codes 0x7F/0xFF are NaN, largest finite 448), with one fp32 scale per (anchor, KV head).

Encoding rule (both sides take it in fp32): scale = fp32(amax) / 448 rounded to fp32
(1.0 when amax == 0); y = fp32(x) / scale rounded to fp32; code = y rounded to the
nearest E4M3 value, ties to the even code, magnitudes above 448 saturated to 448, the
sign kept (so a negative value that rounds to zero gives 0x80).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3FN code from the OCP formula, float64 (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    val = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where((e == 0xF) & (m == 7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(0x7F, dtype=np.int64)      # 0x00..0x7E: the 127 non-negative finite codes
_POS_VALUES = e4m3_decode(_POS_CODES)             # strictly increasing


def e4m3_encode(x) -> np.ndarray:
    """Round values (float64 holding the fp32 quotients) to E4M3 codes: nearest value,
    ties to the even code, saturating at 448, sign kept. NaN is not expected."""
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN input")
    mag = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, mag, side="left")   # first value >= mag
    hi = np.minimum(hi, _POS_VALUES.size - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    code = np.where(mag == _POS_VALUES[hi], _POS_CODES[hi], code)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)


def quantize_kv_fp8(kv, anchor_offsets):
    """Per-(anchor, KV head) quantisation of anchor K or V.

    kv [T_A, Hkv, d] (bf16 values widened), anchor_offsets [A+1]. Returns codes uint8
    [T_A, Hkv, d] and scales float32 [A, Hkv]; dequantised value = decode(code) * scale.
    """
    kv = np.asarray(kv, np.float32)
    ao = np.asarray(anchor_offsets, np.int64)
    A, hkv = ao.size - 1, kv.shape[1]
    codes = np.zeros(kv.shape, np.uint8)
    scales = np.ones((A, hkv), np.float32)
    for a in range(A):
        for g in range(hkv):
            blk = kv[ao[a]:ao[a + 1], g, :]
            amax = np.float32(np.abs(blk).max()) if blk.size else np.float32(0)
            scale = np.float32(amax / np.float32(E4M3_MAX)) if amax > 0 else np.float32(1.0)
            scales[a, g] = scale
            y = (blk / scale).astype(np.float32)   # fp32 quotient, correctly rounded
            codes[ao[a]:ao[a + 1], g, :] = e4m3_encode(y.astype(np.float64))
    return codes, scales


def dequantize_kv_fp8(codes, scales, anchor_offsets):
    """decode(code) * scale in float64 (exact: 4 x 24 significant bits fit in 53)."""
    ao = np.asarray(anchor_offsets, np.int64)
    out = e4m3_decode(codes)
    for a in range(ao.size - 1):
        out[ao[a]:ao[a + 1]] *= np.asarray(scales[a], np.float64)[None, :, None]
    return out
