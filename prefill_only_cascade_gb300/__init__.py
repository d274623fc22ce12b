"""Python binding of libquail: the GB300 (sm_103a) prefill-only cascade attention and
restricted head of Quail's AI.IF / AI_JOIN step.

This module only marshals arguments (tensor pointers, sizes, the current CUDA stream) to
the C ABI declared in include/quail.h; every step of the computation runs in the
library's CUDA kernels. PyTorch supplies device memory and streams. There is no CPU or
PyTorch fallback: importing fails loudly when libquail.so has not been built.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libquail.so")

QUAIL_OK = 0
QUAIL_ERR_INVALID_ARG = 1
QUAIL_ERR_UNSUPPORTED = 2
QUAIL_ERR_CUDA = 3
QUAIL_ERR_TIMEOUT = 4
QUAIL_ERR_DEVICE_BOUNDS = 5
QUAIL_BF16 = 0
QUAIL_FP8_E4M3 = 1

# Every symbol include/quail.h declares.
EXPORTED_SYMBOLS = (
    "quail_cascade_attn", "quail_cascade_workspace_size", "quail_restricted_head",
    "quail_quantize_kv_fp8", "quail_status_string", "quail_get_device_error",
    "quail_set_wait_timeout_ns", "quail_debug_inject", "quail_set_cta_pairs", "quail_version",
    "quail_cascade_attn_noalloc", "quail_causal_prefill_attn",
    "quail_causal_prefill_workspace_size", "quail_kv_plan", "quail_shard_anchors",
    "quail_join_select", "quail_join_select_workspace_size", "quail_shard_batch",
    "quail_cascade_attn_two_pass", "quail_cascade_two_pass_workspace_size",
    "quail_quantize_kv_fp8_with_scales",
)


class QuailError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class ShardSizes(ctypes.Structure):
    _fields_ = [("num_anchors", ctypes.c_int32), ("num_suffixes", ctypes.c_int32),
                ("anchor_tokens", ctypes.c_int64), ("suffix_tokens", ctypes.c_int64)]


class KvPlanStats(ctypes.Structure):
    _fields_ = [("hits", ctypes.c_int64), ("misses", ctypes.c_int64),
                ("compulsory_tokens", ctypes.c_int64), ("regret_tokens", ctypes.c_int64),
                ("peak_resident_tokens", ctypes.c_int64)]


KV_LRU, KV_FURTHEST_NEXT_USE = 0, 1


class CascadeDesc(ctypes.Structure):
    _fields_ = [
        ("num_anchors", ctypes.c_int32),
        ("num_suffixes", ctypes.c_int32),
        ("total_anchor_tokens", ctypes.c_int64),
        ("total_suffix_tokens", ctypes.c_int64),
        ("max_anchor_len", ctypes.c_int32),
        ("max_suffix_len", ctypes.c_int32),
        ("num_q_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("softmax_scale", ctypes.c_float),
        ("kv_anchor_dtype", ctypes.c_int32),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python prefill_only_cascade_gb300/build.py` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    lib.quail_cascade_attn.argtypes = [ctypes.POINTER(CascadeDesc), vp, vp, vp, vp, vp, i32p,
                                       i32p, i32p, f32p, f32p, vp, f32p, vp, ctypes.c_size_t, vp]
    lib.quail_cascade_attn.restype = ctypes.c_int
    lib.quail_cascade_attn_noalloc.argtypes = [ctypes.POINTER(CascadeDesc), vp, vp, vp, vp, vp,
                                               i32p, i32p, i32p, f32p, f32p, vp, f32p, vp]
    lib.quail_cascade_attn_noalloc.restype = ctypes.c_int
    lib.quail_cascade_workspace_size.argtypes = [ctypes.POINTER(CascadeDesc)]
    lib.quail_cascade_workspace_size.restype = ctypes.c_size_t
    lib.quail_cascade_attn_two_pass.argtypes = [ctypes.POINTER(CascadeDesc), vp, vp, vp, vp,
                                                vp, i32p, i32p, i32p, f32p, f32p,
                                                ctypes.c_int32, vp, f32p, vp, ctypes.c_size_t,
                                                vp]
    lib.quail_cascade_attn_two_pass.restype = ctypes.c_int
    lib.quail_cascade_two_pass_workspace_size.argtypes = [ctypes.POINTER(CascadeDesc)]
    lib.quail_cascade_two_pass_workspace_size.restype = ctypes.c_size_t
    lib.quail_restricted_head.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_float, vp,
                                          ctypes.c_int64, ctypes.c_int64, i32p, vp, vp, f32p,
                                          i32p, vp]
    lib.quail_restricted_head.restype = ctypes.c_int
    lib.quail_quantize_kv_fp8.argtypes = [ctypes.c_int32, i32p, ctypes.c_int64, ctypes.c_int32,
                                          ctypes.c_int32, vp, vp, f32p, vp]
    lib.quail_quantize_kv_fp8.restype = ctypes.c_int
    lib.quail_quantize_kv_fp8_with_scales.argtypes = [ctypes.c_int32, i32p, ctypes.c_int64,
                                                      ctypes.c_int32, ctypes.c_int32, vp, f32p,
                                                      vp, f32p, vp]
    lib.quail_quantize_kv_fp8_with_scales.restype = ctypes.c_int
    lib.quail_status_string.argtypes = [ctypes.c_int]
    lib.quail_status_string.restype = ctypes.c_char_p
    lib.quail_get_device_error.argtypes = [vp]
    lib.quail_get_device_error.restype = ctypes.c_int
    lib.quail_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.quail_set_wait_timeout_ns.restype = None
    lib.quail_debug_inject.argtypes = [ctypes.c_int32]
    lib.quail_debug_inject.restype = None
    lib.quail_set_cta_pairs.argtypes = [ctypes.c_int32]
    lib.quail_set_cta_pairs.restype = ctypes.c_int
    lib.quail_version.argtypes = []
    lib.quail_version.restype = ctypes.c_char_p
    i32, i64 = ctypes.c_int32, ctypes.c_int64
    lib.quail_causal_prefill_attn.argtypes = [i32, i64, i32, i32, i32, i32, ctypes.c_float, vp,
                                              vp, vp, i32p, vp, f32p, f32p, f32p, vp,
                                              ctypes.c_size_t, vp]
    lib.quail_causal_prefill_attn.restype = ctypes.c_int
    lib.quail_causal_prefill_workspace_size.argtypes = [i32, i64, i32, i32, i32, i32]
    lib.quail_causal_prefill_workspace_size.restype = ctypes.c_size_t
    lib.quail_kv_plan.argtypes = [i32, vp, i64, vp, i64, i32, vp, ctypes.POINTER(KvPlanStats)]
    lib.quail_kv_plan.restype = ctypes.c_int
    lib.quail_shard_anchors.argtypes = [i32, vp, vp, vp, i32, vp, vp]
    lib.quail_shard_anchors.restype = ctypes.c_int
    lib.quail_shard_batch.argtypes = [i32, vp, vp, vp, vp, i32, ctypes.POINTER(ShardSizes),
                                      vp, vp, vp, vp, vp, vp]
    lib.quail_shard_batch.restype = ctypes.c_int
    lib.quail_join_select_workspace_size.argtypes = [i32]
    lib.quail_join_select_workspace_size.restype = ctypes.c_size_t
    lib.quail_join_select.argtypes = [i32, i32, vp, vp, i32, vp, vp, vp, vp, vp,
                                      ctypes.c_size_t, vp]
    lib.quail_join_select.restype = ctypes.c_int
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.quail_status_string(int(status)).decode()


def version() -> str:
    return lib.quail_version().decode()


def _check(status: int, what: str):
    if status != QUAIL_OK:
        raise QuailError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_desc(num_anchors, num_suffixes, total_anchor_tokens, total_suffix_tokens,
              max_anchor_len, max_suffix_len, num_q_heads, num_kv_heads, head_dim,
              softmax_scale=0.0, kv_fp8=False) -> CascadeDesc:
    return CascadeDesc(int(num_anchors), int(num_suffixes), int(total_anchor_tokens),
                       int(total_suffix_tokens), int(max_anchor_len), int(max_suffix_len),
                       int(num_q_heads), int(num_kv_heads), int(head_dim), float(softmax_scale),
                       QUAIL_FP8_E4M3 if kv_fp8 else QUAIL_BF16)


def cascade_workspace_size(desc: CascadeDesc) -> int:
    return int(lib.quail_cascade_workspace_size(ctypes.byref(desc)))


def cascade_attn(desc: CascadeDesc, q_suf, k_anc, v_anc, k_suf, v_suf, anchor_offsets,
                 anchor_suffix_ptr, suffix_offsets, out, lse=None, workspace=None,
                 k_scale=None, v_scale=None, stream=None):
    """quail_cascade_attn on torch CUDA tensors (see include/quail.h for layouts)."""
    if workspace is None:
        raise ValueError("workspace is required (size: cascade_workspace_size(desc))")
    st = lib.quail_cascade_attn(
        ctypes.byref(desc), _ptr(q_suf), _ptr(k_anc), _ptr(v_anc), _ptr(k_suf), _ptr(v_suf),
        _ptr(anchor_offsets), _ptr(anchor_suffix_ptr), _ptr(suffix_offsets), _ptr(k_scale),
        _ptr(v_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(stream))
    _check(st, "quail_cascade_attn")


def cascade_two_pass_workspace_size(desc: CascadeDesc) -> int:
    return int(lib.quail_cascade_two_pass_workspace_size(ctypes.byref(desc)))


def cascade_attn_two_pass(desc: CascadeDesc, q_suf, k_anc, v_anc, k_suf, v_suf,
                          anchor_offsets, anchor_suffix_ptr, suffix_offsets, out, lse=None,
                          workspace=None, k_scale=None, v_scale=None, merge_in_suffix_pass=True,
                          stream=None):
    """quail_cascade_attn_two_pass: anchor pass, suffix pass and LSE merge run apart
    (workspace size: cascade_two_pass_workspace_size(desc))."""
    if workspace is None:
        raise ValueError("workspace is required (size: cascade_two_pass_workspace_size(desc))")
    st = lib.quail_cascade_attn_two_pass(
        ctypes.byref(desc), _ptr(q_suf), _ptr(k_anc), _ptr(v_anc), _ptr(k_suf), _ptr(v_suf),
        _ptr(anchor_offsets), _ptr(anchor_suffix_ptr), _ptr(suffix_offsets), _ptr(k_scale),
        _ptr(v_scale), 1 if merge_in_suffix_pass else 0, _ptr(out), _ptr(lse), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(stream))
    _check(st, "quail_cascade_attn_two_pass")


def cascade_attn_noalloc(desc: CascadeDesc, q_suf, k_anc, v_anc, k_suf, v_suf, anchor_offsets,
                         anchor_suffix_ptr, suffix_offsets, out, lse=None, k_scale=None,
                         v_scale=None, stream=None):
    """quail_cascade_attn_noalloc: the same computation with the library's fixed device
    scratch array instead of a caller workspace (for callers that may not allocate).
    Calls must not overlap on the GPU; the first call on a device must precede any
    stream capture."""
    st = lib.quail_cascade_attn_noalloc(
        ctypes.byref(desc), _ptr(q_suf), _ptr(k_anc), _ptr(v_anc), _ptr(k_suf), _ptr(v_suf),
        _ptr(anchor_offsets), _ptr(anchor_suffix_ptr), _ptr(suffix_offsets), _ptr(k_scale),
        _ptr(v_scale), _ptr(out), _ptr(lse), _stream(stream))
    _check(st, "quail_cascade_attn_noalloc")


def causal_prefill_workspace_size(num_seqs, total_tokens, max_seq_len, num_q_heads,
                                  num_kv_heads, head_dim):
    return int(lib.quail_causal_prefill_workspace_size(num_seqs, total_tokens, max_seq_len,
                                                       num_q_heads, num_kv_heads, head_dim))


def causal_prefill_attn(q, k, v, seq_offsets, out, max_seq_len, lse=None, workspace=None,
                        softmax_scale=0.0, k_amax=None, v_amax=None, stream=None):
    """quail_causal_prefill_attn: causal self-attention over packed sequences
    (q [T, Hq, d], k/v [T, Hkv, d] bf16, seq_offsets [S+1] int32 on the device); with
    k_amax / v_amax ([S, Hkv] fp32) also the max |k| and |v| per (sequence, KV head)."""
    if workspace is None:
        raise ValueError("workspace is required (size: causal_prefill_workspace_size(...))")
    st = lib.quail_causal_prefill_attn(
        int(seq_offsets.numel() - 1), int(q.shape[0]), int(max_seq_len), int(q.shape[1]),
        int(k.shape[1]), int(q.shape[2]), float(softmax_scale), _ptr(q), _ptr(k), _ptr(v),
        _ptr(seq_offsets), _ptr(out), _ptr(lse), _ptr(k_amax), _ptr(v_amax), _ptr(workspace),
        ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream(stream))
    _check(st, "quail_causal_prefill_attn")


def kv_plan(access_anchor, anchor_tokens, capacity_tokens, policy=KV_FURTHEST_NEXT_USE):
    """quail_kv_plan on host arrays: returns (hit flags uint8 [accesses], stats dict)."""
    import numpy as np
    acc = np.ascontiguousarray(access_anchor, dtype=np.int32)
    size = np.ascontiguousarray(anchor_tokens, dtype=np.int64)
    hit = np.zeros(acc.size, dtype=np.uint8)
    st = KvPlanStats()
    code = lib.quail_kv_plan(int(size.size), size.ctypes.data, int(acc.size), acc.ctypes.data,
                             int(capacity_tokens), int(policy), hit.ctypes.data,
                             ctypes.byref(st))
    _check(code, "quail_kv_plan")
    return hit, {f: getattr(st, f) for f, _ in KvPlanStats._fields_}


def shard_anchors(anchor_offsets, anchor_suffix_ptr, suffix_offsets, num_ranks):
    """quail_shard_anchors on host arrays: returns (rank of each anchor int32 [A], visible
    (query, key) pairs per rank int64 [num_ranks])."""
    import numpy as np
    ao = np.ascontiguousarray(anchor_offsets, dtype=np.int32)
    asp = np.ascontiguousarray(anchor_suffix_ptr, dtype=np.int32)
    so = np.ascontiguousarray(suffix_offsets, dtype=np.int32)
    rank_of = np.zeros(max(ao.size - 1, 0), dtype=np.int32)
    pairs = np.zeros(int(num_ranks), dtype=np.int64)
    code = lib.quail_shard_anchors(int(ao.size - 1), ao.ctypes.data, asp.ctypes.data,
                                   so.ctypes.data, int(num_ranks), rank_of.ctypes.data,
                                   pairs.ctypes.data)
    _check(code, "quail_shard_anchors")
    return rank_of, pairs


def shard_batch(anchor_offsets, anchor_suffix_ptr, suffix_offsets, rank_of_anchor, rank):
    """quail_shard_batch on host arrays: one rank's sub-batch (its anchors in their original
    order with their suffixes). Returns int32 offset arrays rebased to the sub-batch
    (anchor_offsets, anchor_suffix_ptr, suffix_offsets, as quail_cascade_attn takes them),
    the kept anchors' ids and int64 row indices into the full batch: anchor_rows (rows of
    k_anc / v_anc) and suffix_rows (rows of q_suf / k_suf / v_suf and of out / lse)."""
    import numpy as np
    ao = np.ascontiguousarray(anchor_offsets, dtype=np.int32)
    asp = np.ascontiguousarray(anchor_suffix_ptr, dtype=np.int32)
    so = np.ascontiguousarray(suffix_offsets, dtype=np.int32)
    ro = np.ascontiguousarray(rank_of_anchor, dtype=np.int32)
    A = int(ao.size - 1)
    sz = ShardSizes()
    args = (A, ao.ctypes.data, asp.ctypes.data, so.ctypes.data, ro.ctypes.data, int(rank))
    _check(lib.quail_shard_batch(*args, ctypes.byref(sz), None, None, None, None, None, None),
           "quail_shard_batch")
    out = {"anchor_offsets": np.zeros(sz.num_anchors + 1, np.int32),
           "anchor_suffix_ptr": np.zeros(sz.num_anchors + 1, np.int32),
           "suffix_offsets": np.zeros(sz.num_suffixes + 1, np.int32),
           "anchors": np.zeros(sz.num_anchors, np.int32),
           "anchor_rows": np.zeros(sz.anchor_tokens, np.int64),
           "suffix_rows": np.zeros(sz.suffix_tokens, np.int64)}
    _check(lib.quail_shard_batch(*args, ctypes.byref(sz), *(out[k].ctypes.data for k in (
        "anchor_offsets", "anchor_suffix_ptr", "suffix_offsets", "anchors", "anchor_rows",
        "suffix_rows"))), "quail_shard_batch")
    return out


def restricted_head(h, gamma, w8, logits, argmax, eps=1e-6, row_index=None, n_rows=None,
                    stream=None):
    """quail_restricted_head: RMSNorm + 8-column head + argmax over rows of h (or over
    h[row_index]; indices outside h's rows are reported on the device, not read)."""
    if n_rows is None:
        n_rows = row_index.numel() if row_index is not None else h.shape[0]
    st = lib.quail_restricted_head(int(n_rows), int(h.shape[-1]), float(eps), _ptr(h),
                                   int(h.shape[0]), int(h.stride(0)), _ptr(row_index),
                                   _ptr(gamma), _ptr(w8), _ptr(logits), _ptr(argmax),
                                   _stream(stream))
    _check(st, "quail_restricted_head")


def join_select_workspace_size(num_suffixes) -> int:
    return int(lib.quail_join_select_workspace_size(int(num_suffixes)))


def join_select(argmax, true_index, selected, num_selected, workspace, verdict=None,
                anchor_suffix_ptr=None, anchor_count=None, stream=None):
    """quail_join_select on torch CUDA tensors: verdicts of the head's argmax, the passing
    suffix ids in increasing order, their number, and (optionally) a count per anchor."""
    num_anchors = 0 if anchor_suffix_ptr is None else int(anchor_suffix_ptr.numel() - 1)
    st = lib.quail_join_select(num_anchors, int(argmax.numel()), _ptr(anchor_suffix_ptr),
                               _ptr(argmax), int(true_index), _ptr(verdict), _ptr(selected),
                               _ptr(num_selected), _ptr(anchor_count), _ptr(workspace),
                               int(workspace.numel() * workspace.element_size()),
                               _stream(stream))
    _check(st, "quail_join_select")


def quantize_kv_fp8(kv_bf16, anchor_offsets, codes, scale, stream=None):
    """quail_quantize_kv_fp8: per-(anchor, KV head) E4M3 codes and fp32 scales."""
    T, hkv, d = kv_bf16.shape
    st = lib.quail_quantize_kv_fp8(int(anchor_offsets.numel() - 1), _ptr(anchor_offsets), int(T),
                                   int(hkv), int(d), _ptr(kv_bf16), _ptr(codes), _ptr(scale),
                                   _stream(stream))
    _check(st, "quail_quantize_kv_fp8")


def quantize_kv_fp8_with_scales(kv_bf16, anchor_offsets, amax, codes, scale, stream=None):
    """quail_quantize_kv_fp8_with_scales: the same codes and scales given the max |x| of
    every (anchor, KV head) (e.g. the causal prefill's k_amax / v_amax)."""
    T, hkv, d = kv_bf16.shape
    st = lib.quail_quantize_kv_fp8_with_scales(
        int(anchor_offsets.numel() - 1), _ptr(anchor_offsets), int(T), int(hkv), int(d),
        _ptr(kv_bf16), _ptr(amax), _ptr(codes), _ptr(scale), _stream(stream))
    _check(st, "quail_quantize_kv_fp8_with_scales")


def get_device_error(stream=None) -> int:
    return int(lib.quail_get_device_error(_stream(stream)))


def set_wait_timeout_ns(ns: int):
    lib.quail_set_wait_timeout_ns(int(ns))


def debug_inject(skip_first_kv_load: bool):
    lib.quail_debug_inject(1 if skip_first_kv_load else 0)


CTA_PAIRS_OFF, CTA_PAIRS_AUTO, CTA_PAIRS_ALWAYS = 0, 1, 2


def set_cta_pairs(mode: int) -> int:
    """head_dim 128 kernel choice: CTA_PAIRS_OFF (single-SM kernel), CTA_PAIRS_AUTO (the
    default: SM pairs for every fused call, except with the fault-injection switch on) or
    CTA_PAIRS_ALWAYS. Returns the status."""
    return lib.quail_set_cta_pairs(int(mode))


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
