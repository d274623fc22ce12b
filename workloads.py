"""Seeded synthetic inputs for the prefill-only cascade attention and the restricted head.

This module is shared by the oracle's tests, the GPU parity tests and the benchmark. It
holds none of the method's arithmetic: it draws lengths, turns them into offset arrays
(prefix sums of the lengths) and fills tensors with seeded random values.

Shapes follow the workloads of the Quail pages (Qwen3-4B attention heads: 32 query heads,
8 KV heads, head dimension 128; hidden size 2560; an AI.IF join in which one anchor prompt
is shared by thousands of per-pair suffixes, e.g. 4,144 reaction terms per report in the
BIO-4 query of "Quail, il motore di inferenza che supera il miliardo di token al minuto
su una H100", paragraph on BIO-4). The pages' datasets are not used: every value here is
random.

Layouts (all row-major):
  q_suf              [T_S, Hq, d]   bf16   suffix queries, already rotated
  k_anc, v_anc       [T_A, Hkv, d]  bf16   anchor keys/values (FP8 configs quantise them)
  k_suf, v_suf       [T_S, Hkv, d]  bf16   suffix keys/values
  anchor_offsets     [A+1]          int32  token prefix sums into k_anc/v_anc
  anchor_suffix_ptr  [A+1]          int32  suffixes of anchor a are anchor_suffix_ptr[a]..[a+1]-1
  suffix_offsets     [S+1]          int32  token prefix sums into q_suf/k_suf/v_suf/out
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class AttnConfig:
    name: str
    num_anchors: int
    anchor_len: tuple  # inclusive (lo, hi); lo == hi for a fixed length
    suffixes_per_anchor: int
    suffix_len: tuple  # inclusive (lo, hi)
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    kv_fp8: bool
    seed: int


@dataclass(frozen=True)
class HeadConfig:
    name: str
    num_rows: int
    hidden: int
    eps: float
    seed: int


# The five workloads. "tiny" is small enough for the float64 oracle to check in full.
ATTN_CONFIGS = {
    "tiny": AttnConfig("tiny", 4, (64, 64), 16, (32, 32), 4, 1, 64, False, 0),
    "join": AttnConfig("join", 8, (1024, 1024), 4144, (8, 24), 32, 8, 128, False, 1),
    "ragged": AttnConfig("ragged", 256, (128, 2048), 512, (4, 64), 32, 8, 128, False, 2),
    "fp8_long": AttnConfig("fp8_long", 64, (4096, 4096), 1024, (16, 96), 32, 8, 128, True, 4),
    # causal prefill of the anchors themselves: no anchor keys, one 4,096-token sequence
    # per "anchor" (the suffix), Qwen3-4B heads
    "prefill": AttnConfig("prefill", 64, (0, 0), 1, (4096, 4096), 32, 8, 128, False, 6),
}
HEAD_CONFIGS = {
    # 64 last-token rows of the tiny attention workload plus 4,096 more rows
    "tiny": HeadConfig("tiny", 64 + 4096, 256, 1e-6, 0),
    "head": HeadConfig("head", 2_000_000, 2560, 1e-6, 3),
    # the last-token rows of the "join" workload (one per suffix), Qwen3-4B hidden size
    "join_last_token": HeadConfig("join_last_token", 8 * 4144, 2560, 1e-6, 5),
}


@dataclass
class RaggedLayout:
    anchor_lens: np.ndarray       # [A] int64
    suffix_lens: np.ndarray       # [S] int64
    suffix_anchor: np.ndarray     # [S] int64, the anchor of each suffix
    anchor_offsets: np.ndarray    # [A+1] int32
    anchor_suffix_ptr: np.ndarray  # [A+1] int32
    suffix_offsets: np.ndarray    # [S+1] int32

    @property
    def num_anchors(self) -> int:
        return int(self.anchor_lens.shape[0])

    @property
    def num_suffixes(self) -> int:
        return int(self.suffix_lens.shape[0])

    @property
    def total_anchor_tokens(self) -> int:
        return int(self.anchor_offsets[-1])

    @property
    def total_suffix_tokens(self) -> int:
        return int(self.suffix_offsets[-1])

    @property
    def max_anchor_len(self) -> int:
        return int(self.anchor_lens.max()) if self.anchor_lens.size else 0

    @property
    def max_suffix_len(self) -> int:
        return int(self.suffix_lens.max()) if self.suffix_lens.size else 0


def _prefix(lens) -> np.ndarray:
    out = np.zeros(len(lens) + 1, dtype=np.int64)
    np.cumsum(np.asarray(lens, dtype=np.int64), out=out[1:])
    if out[-1] >= 2**31:
        raise ValueError("token count does not fit int32 offsets")
    return out.astype(np.int32)


def layout_from_lengths(anchor_lens, suffixes_per_anchor_list, suffix_lens) -> RaggedLayout:
    """Build offset arrays from explicit lengths (used by the edge-case tests)."""
    anchor_lens = np.asarray(anchor_lens, dtype=np.int64)
    counts = np.asarray(suffixes_per_anchor_list, dtype=np.int64)
    suffix_lens = np.asarray(suffix_lens, dtype=np.int64)
    if counts.sum() != suffix_lens.size or counts.size != anchor_lens.size:
        raise ValueError("suffix counts do not match the suffix lengths")
    suffix_anchor = np.repeat(np.arange(anchor_lens.size, dtype=np.int64), counts)
    return RaggedLayout(anchor_lens, suffix_lens, suffix_anchor, _prefix(anchor_lens),
                        _prefix(counts), _prefix(suffix_lens))


def make_layout(cfg: AttnConfig) -> RaggedLayout:
    """Seeded anchor/suffix lengths for a workload (lengths uniform, bounds inclusive)."""
    rng = np.random.default_rng(cfg.seed)
    A = cfg.num_anchors
    anchor_lens = rng.integers(cfg.anchor_len[0], cfg.anchor_len[1] + 1, size=A)
    S = A * cfg.suffixes_per_anchor
    suffix_lens = rng.integers(cfg.suffix_len[0], cfg.suffix_len[1] + 1, size=S)
    return layout_from_lengths(anchor_lens, [cfg.suffixes_per_anchor] * A, suffix_lens)


def _randn_bf16(shape, gen: torch.Generator, device, chunk=1 << 27) -> torch.Tensor:
    """N(0,1) values drawn in fp32 and rounded to bf16 (round-to-nearest-even)."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    flat = out.view(-1)
    for start in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - start)
        flat[start:start + n] = torch.randn(n, generator=gen, device=device,
                                            dtype=torch.float32).to(torch.bfloat16)
    return out


def make_attention_inputs(cfg: AttnConfig, layout: RaggedLayout, device="cpu") -> dict:
    """Seeded bf16 Q/K/V for a layout. Values are drawn on `device` with a torch generator."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + cfg.seed)
    T_S, T_A = layout.total_suffix_tokens, layout.total_anchor_tokens
    Hq, Hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    t = {
        "q_suf": _randn_bf16((T_S, Hq, d), gen, dev),
        "k_anc": _randn_bf16((T_A, Hkv, d), gen, dev),
        "v_anc": _randn_bf16((T_A, Hkv, d), gen, dev),
        "k_suf": _randn_bf16((T_S, Hkv, d), gen, dev),
        "v_suf": _randn_bf16((T_S, Hkv, d), gen, dev),
    }
    for key in ("anchor_offsets", "anchor_suffix_ptr", "suffix_offsets"):
        t[key] = torch.from_numpy(getattr(layout, key).copy()).to(dev)
    return t


def make_head_inputs(cfg: HeadConfig, device="cpu", num_rows=None) -> dict:
    """h ~ N(0,1), gamma ~ U(0.5, 1.5), W8 ~ N(0, 0.02), all rounded to bf16."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(2000 + cfg.seed)
    n = cfg.num_rows if num_rows is None else num_rows
    h = _randn_bf16((n, cfg.hidden), gen, dev)
    gamma = (torch.rand(cfg.hidden, generator=gen, device=dev) + 0.5).to(torch.bfloat16)
    w8 = (torch.randn((8, cfg.hidden), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    return {"h": h, "gamma": gamma, "w8": w8}


def sample_suffixes(layout: RaggedLayout, count: int, seed: int) -> np.ndarray:
    """A seeded sample of suffix indices for row-sampled parity checks.

    Always includes a suffix of the shortest and of the longest anchor, the shortest and the
    longest suffix, the first and last suffix overall, and one suffix from every block of 8
    anchors; the rest are uniform draws. Anchors without suffixes are skipped.
    """
    rng = np.random.default_rng(10_000 + seed)
    S = layout.num_suffixes
    if S == 0:
        return np.zeros(0, dtype=np.int64)
    ptr = layout.anchor_suffix_ptr.astype(np.int64)
    chosen = {0, S - 1, int(np.argmin(layout.suffix_lens)), int(np.argmax(layout.suffix_lens))}
    has = np.nonzero(ptr[1:] > ptr[:-1])[0]
    if has.size:
        lens = layout.anchor_lens[has]
        for a in (has[np.argmin(lens)], has[np.argmax(lens)]):
            chosen.add(int(rng.integers(ptr[a], ptr[a + 1])))
        for blk in range(0, layout.num_anchors, 8):
            cand = has[(has >= blk) & (has < blk + 8)]
            if cand.size:
                a = int(rng.choice(cand))
                chosen.add(int(rng.integers(ptr[a], ptr[a + 1])))
    while len(chosen) < min(count, S):
        chosen.add(int(rng.integers(0, S)))
    return np.array(sorted(chosen), dtype=np.int64)


def gather_suffix_case(tensors: dict, layout: RaggedLayout, suffix_ids) -> dict:
    """Copy the rows that the sampled suffixes read (their Q/K/V and their anchors' K/V) to
    host numpy arrays, keyed by suffix id. Used to hand a bounded slice of a large
    workload to the CPU oracle."""
    so = layout.suffix_offsets.astype(np.int64)
    ao = layout.anchor_offsets.astype(np.int64)
    out, anchors = {}, {}
    for s in suffix_ids:
        s = int(s)
        a = int(layout.suffix_anchor[s])
        r0, r1 = int(so[s]), int(so[s + 1])
        case = {"anchor": a, "rows": (r0, r1)}
        for key in ("q_suf", "k_suf", "v_suf"):
            case[key] = _to_np(tensors[key][r0:r1])
        if a not in anchors:  # one host copy per anchor, shared by its suffixes
            a0, a1 = int(ao[a]), int(ao[a + 1])
            anchors[a] = {key: _to_np(tensors[key][a0:a1]) for key in ("k_anc", "v_anc")
                          if tensors.get(key) is not None}
        case.update(anchors[a])
        out[s] = case
    return out


def _to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.to(torch.float32).numpy()
    return t.numpy()


@dataclass(frozen=True)
class KvPlanConfig:
    name: str
    num_anchors: int
    anchor_tokens: tuple   # inclusive (lo, hi)
    kind: str              # "two_pass" or "zipf"
    accesses: int          # zipf only
    capacity_frac: float   # anchor-KV capacity as a fraction of all anchors' tokens
    seed: int


KV_PLAN_CONFIGS = {
    # the join of the BIO-4 shape: every anchor's KV is needed in two passes over the
    # anchors (the second list read twice), same order both times
    "two_pass": KvPlanConfig("two_pass", 5000, (256, 1024), "two_pass", 0, 0.15, 7),
    # several queries over shared tables: anchor popularity Zipf(1.1)
    "zipf": KvPlanConfig("zipf", 2000, (256, 1024), "zipf", 40000, 0.15, 8),
}


def make_kv_plan(cfg: KvPlanConfig):
    """Seeded anchor sizes (tokens), access sequence and capacity of a synthetic plan."""
    rng = np.random.default_rng(cfg.seed)
    size = rng.integers(cfg.anchor_tokens[0], cfg.anchor_tokens[1] + 1, size=cfg.num_anchors)
    if cfg.kind == "two_pass":
        order = np.arange(cfg.num_anchors)
        acc = np.concatenate([order, order])
    else:
        ranks = np.arange(1, cfg.num_anchors + 1, dtype=np.float64)
        p = ranks ** -1.1
        acc = rng.choice(cfg.num_anchors, size=cfg.accesses, p=p / p.sum())
    capacity = int(cfg.capacity_frac * size.sum())
    return acc.astype(np.int32), size.astype(np.int64), capacity

