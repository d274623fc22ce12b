"""GPU parity of quail_causal_prefill_attn (causal self-attention over packed sequences,
the anchors' own prefill) against the float64 oracle: the oracle's cascade with anchors of
length 0 is exactly causal attention within each sequence. Every element is compared."""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_util import compare, np64

pytestmark = pytest.mark.gpu

CASES = {
    "gqa4_d128": ([700, 1, 300, 129], (8, 2, 128)),
    "gqa16_d64": ([513, 260, 64], (16, 1, 64)),
    "mha_d128": ([250, 3, 131], (2, 2, 128)),
}


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("with_lse", [True, False])
def test_causal_prefill_every_element(name, with_lse):
    import prefill_only_cascade_gb300 as q
    lens, (hq, hkv, d) = CASES[name]
    seed = zlib.crc32(name.encode()) & 0xFFFF
    g = torch.Generator(device="cuda").manual_seed(seed)
    T = sum(lens)
    qx = workloads._randn_bf16((T, hq, d), g, "cuda")
    kx = workloads._randn_bf16((T, hkv, d), g, "cuda")
    vx = workloads._randn_bf16((T, hkv, d), g, "cuda")
    so = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    so_d = torch.from_numpy(so).cuda()
    ws = torch.empty(q.causal_prefill_workspace_size(len(lens), T, max(lens), hq, hkv, d),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((T, hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((T, hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse \
        else None
    q.causal_prefill_attn(qx, kx, vx, so_d, out, max(lens), lse=lse, workspace=ws)
    torch.cuda.synchronize()
    assert q.get_device_error() == q.QUAIL_OK
    empty = np.zeros((0, hkv, d))
    ref_out, ref_lse = oracle.cascade_attention(
        np64(qx), empty, empty, np64(kx), np64(vx), np.array([0, 0]), np.array([0, len(lens)]),
        so, 1.0 / np.sqrt(d))
    figs = compare(np64(out), np64(lse) if with_lse else None, ref_out,
                   ref_lse if with_lse else None)
    print(name, figs)


def test_causal_prefill_bad_offsets_reported():
    import prefill_only_cascade_gb300 as q
    lens = [40, 30]
    T = sum(lens)
    qx = torch.zeros(T, 8, 128, dtype=torch.bfloat16, device="cuda")
    kx = torch.zeros(T, 2, 128, dtype=torch.bfloat16, device="cuda")
    so_d = torch.tensor([0, 50, T - 1], dtype=torch.int32, device="cuda")  # ends before T
    ws = torch.empty(q.causal_prefill_workspace_size(2, T, 50, 8, 2, 128), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(T, 8, 128, dtype=torch.bfloat16, device="cuda")
    q.causal_prefill_attn(qx, kx, kx, so_d, out, 50, workspace=ws)
    torch.cuda.synchronize()
    assert q.get_device_error() == q.QUAIL_ERR_DEVICE_BOUNDS
