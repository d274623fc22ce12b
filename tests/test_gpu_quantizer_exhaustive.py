"""Bit-exact check of the E4M3 quantiser's division over every finite bf16 input.

The kernel forms x / scale as RN(x r) with one FMA correction (r = RN(1/scale)) instead of
an IEEE division per element. Here 256 (anchor, head) slices, each holding every finite
bf16 value up to a random amax (2^-20 .. 2^20, so 256 different scales), go through
quail_quantize_kv_fp8, and every code and scale must equal the oracle's (numpy fp32
division, correctly rounded, then E4M3 round-to-nearest-even with saturation)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import np64

pytestmark = pytest.mark.gpu


def test_quantizer_every_bf16_input_256_scales():
    import prefill_only_cascade_gb300 as q
    pats = np.arange(1 << 16, dtype=np.uint32)
    vals = (pats << 16).view(np.float32)                     # every bf16 value, widened
    finite = vals[np.isfinite(vals)]
    rng = np.random.default_rng(2024)
    d = 128
    slices, lens = [], []
    for _ in range(256):
        m = np.float32(2.0 ** rng.uniform(-20, 20))
        m = (np.array([m], np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)[0]
        part = finite[np.abs(finite) <= m]                   # contains +-m, so amax == m
        rows = -(-part.size // d)
        blk = np.zeros(rows * d, np.float32)
        blk[:part.size] = rng.permutation(part)
        slices.append(blk.reshape(rows, 1, d))
        lens.append(rows)
    kv32 = np.concatenate(slices, axis=0)
    lay = workloads.layout_from_lengths(lens, [0] * len(lens), [])
    kv = torch.from_numpy(kv32).to("cuda").to(torch.bfloat16)   # exact: values are bf16
    codes = torch.empty(kv.shape, dtype=torch.uint8, device="cuda")
    scale = torch.empty(len(lens), 1, dtype=torch.float32, device="cuda")
    ao = torch.from_numpy(lay.anchor_offsets.copy()).cuda()
    q.quantize_kv_fp8(kv, ao, codes, scale)
    torch.cuda.synchronize()
    ref_codes, ref_scale = oracle.quantize_kv_fp8(np64(kv).astype(np.float32), lay.anchor_offsets)
    np.testing.assert_array_equal(scale.cpu().numpy(), ref_scale)
    got = codes.cpu().numpy()
    diff = np.nonzero(got.reshape(-1) != ref_codes.reshape(-1))[0]
    if diff.size:
        xs = np64(kv).reshape(-1)[diff[:8]]
        rows = diff[:8] // d
        anc = np.searchsorted(lay.anchor_offsets, rows, side="right") - 1
        sc = ref_scale.reshape(-1)[anc]
        raise AssertionError(
            f"{diff.size} of {got.size} codes differ; x={xs.tolist()} scale={sc.tolist()} "
            f"x/scale={(xs.astype(np.float32) / sc).tolist()} "
            f"got={got.reshape(-1)[diff[:8]].tolist()} ref={ref_codes.reshape(-1)[diff[:8]].tolist()}")
