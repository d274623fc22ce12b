"""Speed-of-light and kernel-level cost model of a join plan's cascade attention.

Host-side planning aid (no GPU work): given the ragged layout of a batch (the offset
arrays of quail_cascade_attn) it gives
  * the algorithmic work - FLOPs of the visible (query, key) pairs, 4 d Hq sum_s sum_i
    (L_a + i + 1), and the bytes that must move (Q, out, lse, suffix K/V, anchor K/V once,
    offsets) - and the speed-of-light time max(FLOPs / tensor peak, bytes / HBM peak);
  * a model of the library's single-CTA kernel: the work items its schedule builds
    (anchor, KV head, two 128-row query tiles), each costed in tensor-core cycles from
    measured single-CTA tcgen05.mma rates, plus the steady-state efficiency and the
    per-item overhead measured by a clock64 trace of the kernel, split over the persistent
    CTAs in the kernel's order. For head_dim 128 the library runs the CTA-pair kernel,
    which measures 3-6 % below this model (it moves half the operand bytes per SM).

The method it models: "Motor de inferência Quail atinge 1 bilhão de tokens por minuto por
GPU", section "Como funciona" (simplified cascade attention over a shared anchor and its
suffixes); the roofline view follows "Quail: یک میلیارد توکن در دقیقه روی یک GPU", key
points (throughput per GPU).
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass

import numpy as np

ROWS = 128        # query rows per tile (tcgen05.mma M)
KEYS = 128        # keys per KV tile


@dataclass(frozen=True)
class Hardware:
    bf16_tflops: float = 1902.4          # measured dense bf16 (cuBLAS burst)
    hbm_gbs: float = 6657.0              # measured copy bandwidth
    sm_count: int = 152
    sm_clock_ghz: float = 2.07
    # cycles per tcgen05.mma kind::f16, M = 128, K = 16, one CTA (probe on GB300):
    # A and B from shared memory (SS) or A from tensor memory (TS), by N
    ss_n128: float = 96.0
    ss_n64: float = 68.0
    ts_n128: float = 72.0
    ts_n64: float = 40.0
    # clock64 trace of the kernel (join): ~2,900 wall cycles per k-step of both query tiles
    # against 2,688 cycles of MMA work, and ~3,500 cycles per work-item boundary
    step_efficiency: float = 2688.0 / 2900.0
    item_overhead_cycles: float = 3500.0
    # extra cycles per query tile and masked KV tile (suffix tiles and a partial last anchor
    # tile: the softmax's per-column mask lengthens the critical loop); calibrated on the
    # causal-prefill workload (64 x 4,096 tokens, all tiles masked)
    masked_tile_cycles: float = 680.0
    launch_overhead_us: float = 20.0     # the three schedule kernels and two launches

    @classmethod
    def from_measured(cls, path: str) -> "Hardware":
        """Peaks from a MEASURED_PEAKS-style JSON file (keys bf16_tflops, hbm_gbs,
        sm_max_mhz); the other constants keep their defaults."""
        with open(path) as f:
            m = json.load(f)
        return cls(bf16_tflops=float(m["bf16_tflops"]), hbm_gbs=float(m["hbm_gbs"]),
                   sm_clock_ghz=float(m.get("sm_max_mhz", 2070.0)) / 1e3)


def _lengths(offsets) -> np.ndarray:
    o = np.asarray(offsets, dtype=np.int64)
    return o[1:] - o[:-1]


def work(anchor_offsets, anchor_suffix_ptr, suffix_offsets, hq: int, hkv: int, d: int,
         kv_bytes: int = 2) -> dict:
    """Algorithmic FLOPs and bytes of one cascade call (visible pairs only)."""
    la = _lengths(anchor_offsets)
    ls = _lengths(suffix_offsets)
    counts = _lengths(anchor_suffix_ptr)
    la_of_s = np.repeat(la, counts).astype(np.float64)
    pairs = float(np.sum(ls * la_of_s + ls * (ls + 1) / 2.0))
    ts, ta = int(np.sum(ls)), int(np.sum(la))
    A, S = la.size, ls.size
    flops = 4.0 * d * hq * pairs
    bytes_ = float(ts * hq * d * 2 * 2 + ts * hq * 4 + ts * hkv * d * 2 * 2
                   + ta * hkv * d * kv_bytes * 2 + 4 * (2 * (A + 1) + S + 1))
    return {"flops": flops, "bytes": bytes_, "visible_pairs": pairs, "suffix_tokens": ts}


def sol_seconds(flops: float, bytes_: float, hw: Hardware = Hardware()) -> float:
    """Speed-of-light time: the larger of the tensor-bound and the HBM-bound times."""
    return max(flops / (hw.bf16_tflops * 1e12), bytes_ / (hw.hbm_gbs * 1e9))


def work_items(anchor_offsets, anchor_suffix_ptr, suffix_offsets, hq: int, hkv: int) -> dict:
    """The work items the kernel's schedule builds, in its order: anchors by decreasing
    anchor-tile count (ties in index order), then per anchor KV head g major and query-tile
    pairs minor. Each item: anchor length, and for its two query tiles the first token,
    the suffix-key window start (the first token of the suffix that holds the tile's first
    token), the end, and the start of the suffix that holds its last token."""
    ao = np.asarray(anchor_offsets, dtype=np.int64)
    asp = np.asarray(anchor_suffix_ptr, dtype=np.int64)
    so = np.asarray(suffix_offsets, dtype=np.int64)
    la = ao[1:] - ao[:-1]
    G = hq // hkv
    tok = ROWS // G                       # suffix tokens per query tile
    seg = np.repeat(so[:-1], so[1:] - so[:-1])   # suffix start of every token
    tiles = (la + KEYS - 1) // KEYS
    order = np.argsort(-tiles, kind="stable")
    cols = {k: [] for k in ("la", "ws0", "ws1", "tend0", "tend1", "t0", "t1", "sl0", "sl1")}
    for a in order:
        s_begin, s_end = int(so[asp[a]]), int(so[asp[a + 1]])
        ntok = s_end - s_begin
        if ntok <= 0:
            continue
        pairs = (ntok + 2 * tok - 1) // (2 * tok)
        t0 = s_begin + np.arange(pairs, dtype=np.int64) * 2 * tok
        t1 = t0 + tok
        has1 = t1 < s_end
        tend0 = np.minimum(t0 + tok, s_end)
        tend1 = np.where(has1, np.minimum(t1 + tok, s_end), t1)
        ws0 = seg[t0]
        ws1 = np.where(has1, seg[np.minimum(t1, s_end - 1)], t1)
        sl0 = seg[tend0 - 1]
        sl1 = np.where(has1, seg[np.minimum(tend1, s_end) - 1], t1)
        for _ in range(hkv):
            cols["la"].append(np.full(pairs, la[a]))
            cols["ws0"].append(ws0)
            cols["ws1"].append(ws1)
            cols["tend0"].append(tend0)
            cols["tend1"].append(tend1)
            cols["t0"].append(t0)
            cols["t1"].append(t1)
            cols["sl0"].append(sl0)
            cols["sl1"].append(sl1)
    return {k: (np.concatenate(v) if v else np.zeros(0, np.int64)) for k, v in cols.items()}


def item_mma_cycles(items: dict, d: int, hw: Hardware = Hardware()) -> np.ndarray:
    """Tensor-core cycles of each work item: for each of its two query tiles, every anchor
    tile and every suffix tile costs S = Q K^T (SS, N = keys) and PV (TS, N = d), d / 16 and
    keys / 16 MMA steps."""
    la = items["la"]
    n_anchor = (la + KEYS - 1) // KEYS
    window = np.maximum(items["tend0"] - items["ws0"], items["tend1"] - items["ws1"])
    n_sfx = (window + KEYS - 1) // KEYS
    nk64 = (n_sfx == 1) & (window <= 64)
    pv_step = hw.ts_n128 if d == 128 else hw.ts_n64
    s128 = (d // 16) * hw.ss_n128
    s64 = (d // 16) * hw.ss_n64
    pv128 = (KEYS // 16) * pv_step
    pv64 = (64 // 16) * pv_step
    per_q = n_anchor * (s128 + pv128) + np.where(nk64, n_sfx * (s64 + pv64),
                                                 n_sfx * (s128 + pv128))
    return 2.0 * per_q


def masked_tiles(items: dict) -> np.ndarray:
    """Masked KV tiles of each item, counted per query tile: the last anchor tile when the
    anchor length is not a multiple of 128, and every suffix tile that some row of the
    query tile does not see whole (a row sees keys from the start of its suffix up to
    itself; the kernel skips the mask per warp, this counts per query tile)."""
    la = items["la"]
    window = np.maximum(items["tend0"] - items["ws0"], items["tend1"] - items["ws1"])
    n_sfx = (window + KEYS - 1) // KEYS
    nk = np.where((n_sfx == 1) & (window <= 64), 64, KEYS)
    count = 2 * (la % KEYS != 0).astype(np.int64)
    for q in (0, 1):
        ws, t0, sl = items[f"ws{q}"], items[f"t{q}"], items[f"sl{q}"]
        # tile i covers keys ws + i*128 .. + nk - 1; whole for every row iff
        # its last key <= t0 (first row's token) and sl <= its first key
        i_max = int(n_sfx.max()) if n_sfx.size else 0
        for i in range(i_max):
            base = ws + i * KEYS
            live = i < n_sfx
            whole = (base + nk - 1 <= t0) & (sl <= base)
            count += (live & ~whole).astype(np.int64)
    return count


def staging_seconds(anchor_offsets, hkv: int, d: int, hw: Hardware = Hardware()) -> float:
    """FP8 anchor KV: time of the pass that widens the e4m3 anchor K and V codes to bf16
    (1 byte read and 2 written per code) at the HBM peak."""
    ta = int(np.asarray(anchor_offsets, dtype=np.int64)[-1])
    return 2.0 * ta * hkv * d * 3 / (hw.hbm_gbs * 1e9)


def kernel_seconds(anchor_offsets, anchor_suffix_ptr, suffix_offsets, hq: int, hkv: int,
                   d: int, hw: Hardware = Hardware(), fp8: bool = False) -> dict:
    """Modelled time of one quail_cascade_attn call: items round-robin over
    min(items, SMs) persistent CTAs; each costs its MMA cycles / step_efficiency, the
    per-item overhead and the masked-tile cost; the call takes the slowest CTA plus the
    launch overhead (and, with FP8 anchor KV, the bf16 staging pass: the attention
    kernel is then the BF16 one)."""
    items = work_items(anchor_offsets, anchor_suffix_ptr, suffix_offsets, hq, hkv)
    n = items["la"].size
    extra = staging_seconds(anchor_offsets, hkv, d, hw) if fp8 else 0.0
    if n == 0:
        return {"seconds": hw.launch_overhead_us * 1e-6 + extra, "items": 0, "mma_cycles": 0.0}
    mma = item_mma_cycles(items, d, hw)
    cyc = (mma / hw.step_efficiency + hw.item_overhead_cycles
           + masked_tiles(items) * hw.masked_tile_cycles)
    grid = min(n, hw.sm_count)
    per_cta = np.bincount(np.arange(n) % grid, weights=cyc, minlength=grid)
    seconds = (float(per_cta.max()) / (hw.sm_clock_ghz * 1e9) + hw.launch_overhead_us * 1e-6
               + extra)
    return {"seconds": seconds, "items": int(n), "mma_cycles": float(mma.sum()),
            "mma_floor_seconds": float(np.bincount(np.arange(n) % grid, weights=mma,
                                                   minlength=grid).max())
            / (hw.sm_clock_ghz * 1e9)}


def plan_report(anchor_offsets, anchor_suffix_ptr, suffix_offsets, hq: int, hkv: int, d: int,
                hw: Hardware = Hardware(), kv_bytes: int = 2) -> dict:
    """Work, speed-of-light time and modelled kernel time of one call, in one dict."""
    w = work(anchor_offsets, anchor_suffix_ptr, suffix_offsets, hq, hkv, d, kv_bytes)
    k = kernel_seconds(anchor_offsets, anchor_suffix_ptr, suffix_offsets, hq, hkv, d, hw,
                       fp8=kv_bytes == 1)
    sol = sol_seconds(w["flops"], w["bytes"], hw)
    return {**w, "sol_seconds": sol, "model_seconds": k["seconds"], "items": k["items"],
            "mma_floor_seconds": k.get("mma_floor_seconds", 0.0),
            "bound": "tensor" if w["flops"] / (hw.bf16_tflops * 1e12) >=
                     w["bytes"] / (hw.hbm_gbs * 1e9) else "hbm"}


def default_hardware() -> Hardware:
    """Peaks from MEASURED_PEAKS.json at the repository root when present."""
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "MEASURED_PEAKS.json")
    return Hardware.from_measured(path) if os.path.exists(path) else Hardware()
