"""GPU parity of the two head_dim-128 kernels: query-tile quads on SM pairs and query-tile
pairs on single SMs, each forced by quail_set_cta_pairs (the other GPU tests run the
automatic choice).

Layouts that stress the quad bookkeeping (anchor lengths around the 64-key halves of a
key tile, quads whose second half is empty, pair tiles whose rows start in different
suffixes, long shared suffix windows) and the edge layouts run on both kernels, each
compared element by element with the float64 oracle.
"""
import zlib

import numpy as np
import pytest
import torch

import workloads
from parity_util import check_full, check_sampled, redo_count, run_cascade
from test_gpu_parity import EDGE_CASES, _inputs

pytestmark = pytest.mark.gpu


def _force(mode):
    import prefill_only_cascade_gb300 as q
    assert q.set_cta_pairs(mode) == q.QUAIL_OK
    yield
    q.set_cta_pairs(q.CTA_PAIRS_AUTO)


@pytest.fixture
def pairs_off():
    yield from _force(0)


@pytest.fixture
def pairs_always():
    yield from _force(2)


QUAD_CASES = {
    # name: (anchor lengths, suffixes per anchor, suffix lengths or (lo, hi), heads)
    # anchor lengths across the 64-key halves and 128-key tiles
    "anchor_halves": ([1, 63, 64, 65, 127, 128, 129, 191, 192, 255, 257], [2] * 11, (1, 90),
                      (8, 2, 128)),
    # 1..7 query tiles per anchor and KV head (G = 8: 16 tokens a tile): every quad tail
    "quad_tails": ([100, 40, 300, 7, 0, 500, 64], [1, 2, 3, 4, 5, 6, 7], (1, 20), (16, 2, 128)),
    # G = 16, one-token suffixes: the four query tiles of a quad start in different suffixes
    "many_suffixes_g16": ([130, 1, 700], [60, 33, 64], (1, 3), (16, 1, 128)),
    # one long suffix per anchor (windows of many key tiles, shared by both pair tiles)
    "long_windows": ([0, 200, 0], [1, 1, 2], [900, 650, 300, 420], (8, 2, 128)),
    # G = 1 (MHA): 128 tokens a tile, quads over 512 tokens
    "mha_quads": ([300, 5], [3, 2], [600, 1, 129, 512, 77], (2, 2, 128)),
}


def _layout(name, cases):
    anchors, counts, lens, heads = cases[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    n = sum(counts)
    if isinstance(lens, tuple):
        lens = rng.integers(lens[0], lens[1] + 1, size=n)
    return workloads.layout_from_lengths(anchors, counts, lens), heads


@pytest.mark.parametrize("name", sorted(QUAD_CASES))
def test_quad_layouts_every_element(name, pairs_always):
    lay, heads = _layout(name, QUAD_CASES)
    t = _inputs(lay, heads, seed=11)
    out, lse, ws = run_cascade(heads, lay, t, keep_ws=True)
    figs = check_full(heads, lay, t, out, lse)
    print(name, figs, "redo", redo_count(ws))


@pytest.mark.parametrize("name", sorted(QUAD_CASES))
def test_quad_layouts_fp8_every_element(name, pairs_always):
    from parity_util import FP8_REL_L2, fp8_max_abs
    from test_gpu_fp8 import _oracle_kv, _quantise
    lay, (hq, hkv, d) = _layout(name, QUAD_CASES)
    cfg = workloads.AttnConfig("fp8case", lay.num_anchors, (0, 0), 0, (0, 0), hq, hkv, d,
                               True, 13)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    qz = _quantise(t, lay, hkv)
    kd = _oracle_kv(t, lay, "k_anc")[2]
    vd = _oracle_kv(t, lay, "v_anc")[2]
    t8 = dict(t, k_anc=qz["k_anc"][0], v_anc=qz["v_anc"][0])
    out, lse = run_cascade((hq, hkv, d), lay, t8, kv_fp8=True, k_scale=qz["k_anc"][1],
                           v_scale=qz["v_anc"][1])
    figs = check_full((hq, hkv, d), lay, t, out, lse, kv=(kd, vd), rel_bound=FP8_REL_L2,
                      max_abs=fp8_max_abs(t["v_anc"]))
    print(name, figs)


D128_EDGE = sorted(k for k, v in EDGE_CASES.items() if v[3][2] == 128)


@pytest.mark.parametrize("name", D128_EDGE)
def test_edge_layouts_pair_kernel_every_element(name, pairs_always):
    lay, heads = _layout(name, EDGE_CASES)
    t = _inputs(lay, heads, seed=11)
    out, lse = run_cascade(heads, lay, t)
    print(name, check_full(heads, lay, t, out, lse))


@pytest.mark.parametrize("name", sorted(set(QUAD_CASES) | set(D128_EDGE)))
def test_single_sm_kernel_every_element(name, pairs_off):
    cases = QUAD_CASES if name in QUAD_CASES else EDGE_CASES
    lay, heads = _layout(name, cases)
    t = _inputs(lay, heads, seed=11)
    out, lse = run_cascade(heads, lay, t)
    figs = check_full(heads, lay, t, out, lse)
    print(name, figs)


@pytest.mark.parametrize("name", ["join", "ragged"])
def test_full_size_both_kernels_sampled_rows(name):
    import prefill_only_cascade_gb300 as q
    cfg = workloads.ATTN_CONFIGS[name]
    lay = workloads.make_layout(cfg)
    t = workloads.make_attention_inputs(cfg, lay, "cuda")
    heads = (cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim)
    ids = workloads.sample_suffixes(lay, 32, cfg.seed + 1)
    res = []
    try:
        for mode in (q.CTA_PAIRS_OFF, q.CTA_PAIRS_ALWAYS):
            q.set_cta_pairs(mode)
            res.append(run_cascade(heads, lay, t))
    finally:
        q.set_cta_pairs(q.CTA_PAIRS_AUTO)
    (out1, lse1), (out2, lse2) = res
    for out, lse in ((out1, lse1), (out2, lse2)):
        assert torch.isfinite(out).all() and torch.isfinite(lse).all()
        print(name, check_sampled(heads, lay, t, out, lse, ids))
    # the two kernels differ only in rounding (tile boundaries of the key windows)
    diff = 0.0
    step = 1 << 20
    for i in range(0, out1.shape[0], step):
        diff = max(diff, (out1[i:i + step].float() - out2[i:i + step].float()).abs().max().item())
    assert diff < 3e-2, diff
    del t, out1, out2, lse1, lse2, res
    torch.cuda.empty_cache()



@pytest.mark.parametrize("seed", range(32))
def test_random_layouts_both_kernels_every_element(seed):
    # seeded random layouts: 1-6 anchors of 0-700 tokens, 0-12 suffixes each of 1-150
    # tokens, G in {1, 2, 4, 8, 16}; both kernels forced, every element against the oracle
    import prefill_only_cascade_gb300 as q
    rng = np.random.default_rng(1000 + seed)
    na = int(rng.integers(1, 7))
    anchors = [int(x) for x in rng.integers(0, 701, size=na)]
    counts = [int(x) for x in rng.integers(0, 13, size=na)]
    if sum(counts) == 0:
        counts[0] = 1
    lens = [int(x) for x in rng.integers(1, 151, size=sum(counts))]
    g = int(rng.choice([1, 2, 4, 8, 16]))
    hkv = int(rng.choice([1, 2]))
    heads = (g * hkv, hkv, 128)
    lay = workloads.layout_from_lengths(anchors, counts, lens)
    t = _inputs(lay, heads, seed=seed)
    try:
        for mode in (q.CTA_PAIRS_ALWAYS, q.CTA_PAIRS_OFF):
            q.set_cta_pairs(mode)
            out, lse = run_cascade(heads, lay, t)
            print(seed, mode, heads, anchors, counts, check_full(heads, lay, t, out, lse))
    finally:
        q.set_cta_pairs(q.CTA_PAIRS_AUTO)


@pytest.mark.parametrize("lens", [(1, 30), (40, 200)])
def test_pair_kernel_redo_lists_quad_halves(lens, pairs_always):
    # anchor 1's keys past its first tile x 40: its quads leave the fast bounds and hand
    # their non-empty halves (two-tile items) to the exact kernel; the other anchors stay
    # fast. Count: 2 KV heads x ceil(tokens / 64) halves (G = 4: 32 tokens a query tile).
    from test_gpu_redo import _case
    lay, t = _case([200, 300, 150], [3, 3, 3], lens, (8, 2, 128), 12)
    ao = lay.anchor_offsets
    lo, hi = int(ao[1]) + 128, int(ao[2])
    t["k_anc"][lo:hi] = (t["k_anc"][lo:hi].float() * 40).to(torch.bfloat16)
    out, lse, ws = run_cascade((8, 2, 128), lay, t, keep_ws=True)
    so, asp = lay.suffix_offsets, lay.anchor_suffix_ptr
    ntok = int(so[asp[2]] - so[asp[1]])
    assert redo_count(ws) == 2 * ((ntok + 63) // 64)
    print(lens, check_full((8, 2, 128), lay, t, out, lse))
