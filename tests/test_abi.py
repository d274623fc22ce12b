"""Host-only checks of the C ABI: the library loads, exports every function that
include/quail.h declares, and rejects bad arguments on the host (no kernel launch)."""
import ctypes
import os
import re

import pytest

import prefill_only_cascade_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "quail.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(quail_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    declared = _declared_functions()
    assert len(declared) >= 9
    assert sorted(q.EXPORTED_SYMBOLS) == declared
    for name in declared:
        assert hasattr(q.lib, name), name
        assert ctypes.cast(getattr(q.lib, name), ctypes.c_void_p).value


def test_status_strings_and_version():
    assert q.status_string(0) == "QUAIL_OK"
    assert q.status_string(4) == "QUAIL_ERR_TIMEOUT"
    assert q.status_string(5) == "QUAIL_ERR_DEVICE_BOUNDS"
    assert q.status_string(99) == "QUAIL_ERR_UNKNOWN"
    assert q.version().startswith("quail-gb300")


def test_desc_layout_matches_header():
    # int32 x2, int64 x2, int32 x5, float, int32 -> 8 + 16 + 20 + 4 + 4 = 52 -> 56 aligned
    assert ctypes.sizeof(q.CascadeDesc) == 56
    assert q.CascadeDesc.total_anchor_tokens.offset == 8


def test_workspace_size():
    d = q.make_desc(8, 33152, 8192, 530000, 1024, 24, 32, 8, 128)
    assert q.cascade_workspace_size(d) >= (2 * 8 + 1) * 4
    assert q.cascade_workspace_size(d) % 256 == 0
    assert q.lib.quail_cascade_workspace_size(None) == 0
    # FP8 anchor KV: the workspace also holds the anchor codes widened to bf16, two
    # [T_A, Hkv, d] copies (each placed on a 256-byte boundary)
    d8 = q.make_desc(8, 33152, 8192, 530000, 1024, 24, 32, 8, 128, kv_fp8=True)
    extra = q.cascade_workspace_size(d8) - q.cascade_workspace_size(d)
    assert 4 * 8192 * 8 * 128 <= extra <= 4 * 8192 * 8 * 128 + 512


def _call_attn(desc, fake=0x10000, ws_bytes=1 << 20, **over):
    args = dict(q_suf=fake, k_anc=fake, v_anc=fake, k_suf=fake, v_suf=fake, ao=fake,
                asp=fake, so=fake, ks=None, vs=None, out=fake, lse=None, ws=fake)
    args.update(over)
    v = lambda x: None if x is None else ctypes.c_void_p(x)
    return q.lib.quail_cascade_attn(
        ctypes.byref(desc) if desc is not None else None, v(args["q_suf"]), v(args["k_anc"]),
        v(args["v_anc"]), v(args["k_suf"]), v(args["v_suf"]), v(args["ao"]), v(args["asp"]),
        v(args["so"]), v(args["ks"]), v(args["vs"]), v(args["out"]), v(args["lse"]),
        v(args["ws"]), ctypes.c_size_t(ws_bytes), None)


def _good_desc(**kw):
    base = dict(num_anchors=2, num_suffixes=4, total_anchor_tokens=100, total_suffix_tokens=40,
                max_anchor_len=60, max_suffix_len=20, num_q_heads=32, num_kv_heads=8,
                head_dim=128)
    base.update(kw)
    return q.make_desc(**base)


@pytest.mark.parametrize("change,expect", [
    (dict(num_q_heads=30), q.QUAIL_ERR_INVALID_ARG),          # not a multiple of Hkv
    (dict(num_kv_heads=0), q.QUAIL_ERR_INVALID_ARG),
    (dict(num_anchors=-1), q.QUAIL_ERR_INVALID_ARG),
    (dict(total_suffix_tokens=1 << 31), q.QUAIL_ERR_INVALID_ARG),  # int32 offsets overflow
    (dict(head_dim=96), q.QUAIL_ERR_UNSUPPORTED),
    (dict(num_q_heads=64, num_kv_heads=2), q.QUAIL_ERR_UNSUPPORTED),  # group of 32
    (dict(softmax_scale=-1.0), q.QUAIL_ERR_INVALID_ARG),
    (dict(softmax_scale=float("inf")), q.QUAIL_ERR_INVALID_ARG),
    (dict(num_suffixes=0), q.QUAIL_ERR_INVALID_ARG),           # tokens without suffixes
])
def test_cascade_rejects_bad_descriptors(change, expect):
    assert _call_attn(_good_desc(**change)) == expect


def test_cascade_rejects_bad_pointers():
    d = _good_desc()
    assert _call_attn(None) == q.QUAIL_ERR_INVALID_ARG
    assert _call_attn(d, q_suf=None) == q.QUAIL_ERR_INVALID_ARG
    assert _call_attn(d, out=0x10008) == q.QUAIL_ERR_INVALID_ARG          # not 16-byte aligned
    assert _call_attn(d, out=0x10010) == q.QUAIL_ERR_INVALID_ARG          # not 32-byte aligned
    assert _call_attn(d, so=None) == q.QUAIL_ERR_INVALID_ARG
    assert _call_attn(d, ws=None) == q.QUAIL_ERR_INVALID_ARG
    assert _call_attn(d, ws_bytes=8) == q.QUAIL_ERR_INVALID_ARG           # workspace too small
    assert _call_attn(d, ks=0x10000) == q.QUAIL_ERR_INVALID_ARG           # scales with bf16
    fp8 = _good_desc(kv_fp8=True)
    assert _call_attn(fp8) == q.QUAIL_ERR_INVALID_ARG                     # fp8 without scales
    assert _call_attn(_good_desc(kv_fp8=True, head_dim=96), ks=0x10000, vs=0x10000) == \
        q.QUAIL_ERR_UNSUPPORTED
    # FP8 needs room for the staged bf16 anchors: the BF16-sized workspace is too small
    bf16_bytes = q.cascade_workspace_size(_good_desc())
    assert _call_attn(fp8, ks=0x10000, vs=0x10000, ws_bytes=bf16_bytes) == \
        q.QUAIL_ERR_INVALID_ARG


def test_head_rejects_bad_arguments():
    f = ctypes.c_void_p(0x10000)
    call = lambda n, hid, eps=1e-6, stride=None, h=f, lg=f, rows=4, idx=None: \
        q.lib.quail_restricted_head(n, hid, eps, h, rows, hid if stride is None else stride,
                                    idx, f, f, lg, f, None)
    assert call(-1, 256) == q.QUAIL_ERR_INVALID_ARG
    assert call(4, 250) == q.QUAIL_ERR_INVALID_ARG            # not a multiple of 32
    assert call(4, 256, eps=-1.0) == q.QUAIL_ERR_INVALID_ARG
    assert call(4, 256, stride=255) == q.QUAIL_ERR_INVALID_ARG
    assert call(4, 256, stride=260) == q.QUAIL_ERR_INVALID_ARG  # row stride not 16-byte multiple
    assert call(4, 256, h=None) == q.QUAIL_ERR_INVALID_ARG
    assert call(4, 256, lg=ctypes.c_void_p(0x10004)) == q.QUAIL_ERR_INVALID_ARG
    assert call(4, 8192) == q.QUAIL_ERR_UNSUPPORTED
    assert call(4, 256, rows=3) == q.QUAIL_ERR_INVALID_ARG   # more output rows than h has
    assert call(4, 256, rows=-1) == q.QUAIL_ERR_INVALID_ARG
    # with a gather the row count of h only bounds the indices (checked on the device)
    assert call(4, 256, rows=3, idx=ctypes.c_void_p(0x10002)) == q.QUAIL_ERR_INVALID_ARG


def test_quantize_rejects_bad_arguments():
    f = ctypes.c_void_p(0x10000)
    assert q.lib.quail_quantize_kv_fp8(-1, f, 10, 8, 128, f, f, f, None) == q.QUAIL_ERR_INVALID_ARG
    assert q.lib.quail_quantize_kv_fp8(2, f, 10, 8, 96, f, f, f, None) == q.QUAIL_ERR_UNSUPPORTED
    assert q.lib.quail_quantize_kv_fp8(2, None, 10, 8, 128, f, f, f, None) == q.QUAIL_ERR_INVALID_ARG
    assert q.lib.quail_quantize_kv_fp8(2, f, 10, 8, 128, ctypes.c_void_p(0x10001), f, f, None) == \
        q.QUAIL_ERR_INVALID_ARG


def test_causal_prefill_rejects_bad_arguments():
    f = 0x10000
    v = lambda x: None if x is None else ctypes.c_void_p(x)

    def call(S=3, T=100, L=60, hq=8, hkv=2, d=128, scale=0.0, q=f, k=f, v_=f, so=f, out=f,
             lse=None, ws=f, ws_bytes=1 << 20, ka=None, va=None):
        return q_lib().quail_causal_prefill_attn(S, T, L, hq, hkv, d, scale, v(q), v(k), v(v_),
                                                 v(so), v(out), v(lse), v(ka), v(va), v(ws),
                                                 ctypes.c_size_t(ws_bytes), None)

    def q_lib():
        return q.lib
    assert call(S=-1) == q.QUAIL_ERR_INVALID_ARG
    assert call(S=0, T=5) == q.QUAIL_ERR_INVALID_ARG
    assert call(S=0, T=0) == q.QUAIL_OK                     # empty: nothing to do
    assert call(hq=7) == q.QUAIL_ERR_INVALID_ARG            # not a multiple of Hkv
    assert call(hq=6) == q.QUAIL_ERR_UNSUPPORTED            # group of 3
    assert call(d=96) == q.QUAIL_ERR_UNSUPPORTED
    assert call(hq=64, hkv=2) == q.QUAIL_ERR_UNSUPPORTED    # group of 32
    assert call(scale=float("nan")) == q.QUAIL_ERR_INVALID_ARG
    assert call(so=None) == q.QUAIL_ERR_INVALID_ARG
    assert call(out=0x10010) == q.QUAIL_ERR_INVALID_ARG     # not 32-byte aligned
    assert call(k=0x10008) == q.QUAIL_ERR_INVALID_ARG       # not 16-byte aligned
    assert call(ws=0x10080) == q.QUAIL_ERR_INVALID_ARG      # workspace not 256-byte aligned
    assert call(ws_bytes=64) == q.QUAIL_ERR_INVALID_ARG     # workspace too small
    assert call(ka=0x10000) == q.QUAIL_ERR_INVALID_ARG      # k_amax without v_amax
    assert call(ka=0x10000, va=0x10002) == q.QUAIL_ERR_INVALID_ARG   # misaligned
    assert q.causal_prefill_workspace_size(3, 100, 60, 8, 2, 128) > 256
    assert q.causal_prefill_workspace_size(-1, 100, 60, 8, 2, 128) == 0


def test_join_select_rejects_bad_arguments():
    f = ctypes.c_void_p(0x10000)
    ws_need = q.join_select_workspace_size(10)
    assert ws_need >= 16 and q.join_select_workspace_size(-1) == 0
    call = lambda **kw: q.lib.quail_join_select(
        kw.get("A", 2), kw.get("S", 10), kw.get("asp", f), kw.get("am", f), kw.get("t", 3),
        kw.get("v", None), kw.get("sel", f), kw.get("n", f), kw.get("cnt", None),
        kw.get("ws", f), ctypes.c_size_t(kw.get("ws_bytes", ws_need)), None)
    assert call(t=8) == q.QUAIL_ERR_INVALID_ARG            # only 8 options
    assert call(t=-1) == q.QUAIL_ERR_INVALID_ARG
    assert call(S=-1) == q.QUAIL_ERR_INVALID_ARG
    assert call(n=None) == q.QUAIL_ERR_INVALID_ARG         # the count is always written
    assert call(am=None) == q.QUAIL_ERR_INVALID_ARG
    assert call(sel=ctypes.c_void_p(0x10002)) == q.QUAIL_ERR_INVALID_ARG   # misaligned
    assert call(cnt=f, asp=None) == q.QUAIL_ERR_INVALID_ARG  # per-anchor counts need the CSR
    assert call(ws_bytes=ws_need - 4) == q.QUAIL_ERR_INVALID_ARG


def test_two_pass_workspace_and_argument_checks():
    d = _good_desc()
    base = q.cascade_workspace_size(d)
    two = q.cascade_two_pass_workspace_size(d)
    rows = d.total_suffix_tokens * d.num_q_heads
    assert two >= base + 4 * rows * (d.head_dim + 2) and two % 256 == 0
    assert q.cascade_two_pass_workspace_size(_good_desc(head_dim=96)) == 0
    f = ctypes.c_void_p(0x10000)
    call = lambda desc, merge: q.lib.quail_cascade_attn_two_pass(
        desc, f, f, f, f, f, f, f, f, None, None, merge, ctypes.c_void_p(0x10020), None, f,
        ctypes.c_size_t(two), None)
    assert call(None, 1) == q.QUAIL_ERR_INVALID_ARG
    assert call(ctypes.byref(d), 2) == q.QUAIL_ERR_INVALID_ARG         # merge flag 0 or 1
    assert q.lib.quail_cascade_attn_two_pass(
        ctypes.byref(d), f, f, f, f, f, f, f, f, None, None, 1, ctypes.c_void_p(0x10020), None,
        f, ctypes.c_size_t(base), None) == q.QUAIL_ERR_INVALID_ARG     # workspace too small


def test_quantize_with_scales_rejects_bad_arguments():
    f = ctypes.c_void_p(0x10000)
    call = lambda A=2, ao=f, T=10, hkv=8, d=128, x=f, amax=f, c=f, sc=f: \
        q.lib.quail_quantize_kv_fp8_with_scales(A, ao, T, hkv, d, x, amax, c, sc, None)
    assert call(A=-1) == q.QUAIL_ERR_INVALID_ARG
    assert call(d=96) == q.QUAIL_ERR_UNSUPPORTED
    assert call(amax=None) == q.QUAIL_ERR_INVALID_ARG
    assert call(amax=ctypes.c_void_p(0x10002)) == q.QUAIL_ERR_INVALID_ARG
    assert call(x=ctypes.c_void_p(0x10008)) == q.QUAIL_ERR_INVALID_ARG


def test_cta_pair_mode_values_checked():
    # host-only: the mode switch validates its argument (no kernel runs)
    assert q.set_cta_pairs(3) == q.QUAIL_ERR_INVALID_ARG
    assert q.set_cta_pairs(-1) == q.QUAIL_ERR_INVALID_ARG
    for mode in (q.CTA_PAIRS_OFF, q.CTA_PAIRS_ALWAYS, q.CTA_PAIRS_AUTO):
        assert q.set_cta_pairs(mode) == q.QUAIL_OK
