"""Benchmark of the prefill-only AI.IF / AI_JOIN hot path on GB300.

One step = one pass of the whole path over one batch: the cascade attention over every
suffix token of the workload, then the restricted head (RMSNorm + 8 columns + argmax) on
the last token of every suffix (gathered by row index from the hidden states of all
suffix tokens). Default workload: the largest one that fits one GPU, "ragged" (256
anchors of U[128, 2048] tokens, 512 suffixes each of U[4, 64] tokens, 32 query / 8 KV
heads, d = 128; hidden size 2,560 for the head). Inputs are synthetic and seeded and
already resident in HBM; they are larger than L2, so L2 is not flushed between steps.

Prints ONE JSON line (metric: suffix tokens per second). The line also carries, measured
in the same process after the headline: `sub.join` (the Qwen3-4B join), `sub.fp8_long`
(e4m3 anchor KV), `sub.head` (2 M head rows) and `sub.softmax_stress` (the join with
queries scaled x4 and x8), each with its own roofline, oracle baseline and parity.
Each attention workload also carries `fused_vs_two_pass`: the same batch through the
two-pass entry point (anchor pass, suffix pass, LSE merge) timed against the fused call.
`--impl reference` times the float64 CPU oracle on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "suffix tokens/sec (cascade prefill attn) and % of GB300 BF16 tensor/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
ATTN_WORKLOADS = ("ragged", "join", "fp8_long")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="ragged",
                    choices=["ragged", "join", "fp8_long", "head", "quantize", "prefill",
                             "kvplan"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub", action="store_true",
                    help="only the headline workload (no sub-objects)")
    ap.add_argument("--strong", action="store_true",
                    help="N > 1: split ONE batch of the workload over the ranks (strong "
                         "scaling) instead of N batches (weak scaling)")
    ap.add_argument("--head-rows", type=int, default=None,
                    help="fewer rows for --workload head (profiling only)")
    ap.add_argument("--suffixes-per-anchor", type=int, default=None,
                    help="smaller case of the same workload (profiling only)")
    ap.add_argument("--sequences", type=int, default=None,
                    help="fewer sequences for --workload prefill (profiling only)")
    return ap.parse_args(argv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def attention_flops(layout, hq, d) -> float:
    """4 d Hq sum_s sum_{i < l_s} (L_a + i + 1): only visible (query, key) pairs count."""
    la = layout.anchor_lens[layout.suffix_anchor].astype(np.float64)
    ls = layout.suffix_lens.astype(np.float64)
    pairs = ls * la + ls * (ls + 1) / 2
    return float(4.0 * d * hq * pairs.sum())


def attention_bytes(layout, hq, hkv, d, kv_bytes=2) -> float:
    """Algorithmic bytes: Q + out + lse + suffix K/V once + anchor K/V once + offsets."""
    ts, ta = layout.total_suffix_tokens, layout.total_anchor_tokens
    return float(ts * hq * d * 2 * 2 + ts * hq * 4 + ts * hkv * d * 2 * 2
                 + ta * hkv * d * kv_bytes * 2
                 + 4 * (2 * (layout.num_anchors + 1) + layout.num_suffixes + 1))


def pair_kernel(layout, hq, hkv, d) -> bool:
    """Whether quail_cascade_attn's automatic choice runs the CTA-pair kernel for this
    layout: every head_dim-128 fused call (the rule the library states for
    QUAIL_CTA_PAIRS_AUTO)."""
    return d == 128


def work_items(layout, hkv, group) -> int:
    """Work items of one cascade call: per anchor and KV head, one per pair of 128-row
    query tiles over the anchor's suffix tokens (bench bookkeeping for the redo rate; a
    CTA-pair quad counts as its two halves, as the exact kernel's list does)."""
    pair_tok = 2 * (128 // group)
    so, asp = layout.suffix_offsets.astype(np.int64), layout.anchor_suffix_ptr.astype(np.int64)
    ntok = so[asp[1:]] - so[asp[:-1]]
    return int(hkv * ((ntok + pair_tok - 1) // pair_tok).sum())


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)  # let the sampler start
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def code_digest(path: str) -> str:
    """sha256 of a source file's code: `//` comments, trailing blanks and empty lines
    removed, so that a comment edit does not disown a profile taken on the same code."""
    lines = []
    for line in open(path, encoding="utf-8"):
        i = line.find("//")
        if i >= 0:
            line = line[:i]
        line = line.rstrip()
        if line:
            lines.append(line)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()


def traffic_from_profile(kernel_file: str, profile_md: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel code (the summary records `kernel_code_sha256`, the code_digest of the source,
    or an older whole-file `kernel_source_sha256`)."""
    path = os.path.join(ROOT, "profiles", profile_md)
    src = os.path.join(ROOT, "prefill_only_cascade_gb300", "csrc", kernel_file)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if "kernel_code_sha256" in vals:
        ok = vals["kernel_code_sha256"] == code_digest(src)
    else:
        ok = vals.get("kernel_source_sha256") == hashlib.sha256(open(src, "rb").read()).hexdigest()
    if not ok:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------- ranks

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value: float, device="cuda") -> float:
    """Largest value over the ranks (the job's time is its slowest rank's time)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(world, value: float, device="cuda") -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def global_layout(cfg, copies: int):
    """The job's batch: `copies` seeded batches of the workload's shape side by side (copy r
    drawn with seed cfg.seed + 7919 r), as one ragged batch."""
    lays = [workloads.make_layout(dataclasses.replace(cfg, seed=cfg.seed + 7919 * r))
            for r in range(copies)]
    return workloads.layout_from_lengths(
        np.concatenate([l.anchor_lens for l in lays]),
        np.concatenate([np.diff(l.anchor_suffix_ptr) for l in lays]),
        np.concatenate([l.suffix_lens for l in lays]))


def rank_layout(cfg, world: int, rank: int, strong: bool = False):
    """This rank's share of the job (the path partitions by anchor and has no exchange
    step). Weak scaling: the job is `world` batches of the workload's shape; strong: one
    batch. Anchors go to ranks by quail_shard_anchors (longest processing time first on
    visible (query, key) pairs) and quail_shard_batch gives the rank's sub-batch. Returns
    (layout, plan) with plan = the ranks' loads in visible pairs."""
    if world == 1:
        return workloads.make_layout(cfg), None
    import prefill_only_cascade_gb300 as q
    g = global_layout(cfg, 1 if strong else world)
    rank_of, pairs = q.shard_anchors(g.anchor_offsets, g.anchor_suffix_ptr, g.suffix_offsets,
                                     world)
    sb = q.shard_batch(g.anchor_offsets, g.anchor_suffix_ptr, g.suffix_offsets, rank_of, rank)
    lay = workloads.layout_from_lengths(np.diff(sb["anchor_offsets"]),
                                        np.diff(sb["anchor_suffix_ptr"]),
                                        np.diff(sb["suffix_offsets"]))
    return lay, {"rank_pairs": [int(x) for x in pairs], "global_anchors": g.num_anchors}


# ---------------------------------------------------------------------------- oracle timing

def _oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        return max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:  # threadpoolctl is not installed everywhere
        return len(os.sched_getaffinity(0))


def cpu_oracle_sample(layout, cfg, t_host_fn, budget_s=15.0, max_suffixes=1024, kv_for=None,
                      with_head=True, results=None, q_scale=1.0):
    """Time the float64 oracle (attention of each suffix + its head row) on host cores over a
    seeded sample of suffixes until `budget_s` is spent. kv_for(anchor) -> (k, v) float64
    replaces the anchor K/V (FP8: the oracle quantises and dequantises the anchor itself,
    once per anchor, inside the timed loop). With a dict `results`, each sampled suffix's
    oracle (out, lse) is stored under its id. Returns tokens/s and details."""
    import oracle
    threads = _oracle_threads()
    ids = workloads.sample_suffixes(layout, max_suffixes, cfg.seed + 100)
    cases = t_host_fn(ids)
    hx = workloads.make_head_inputs(workloads.HEAD_CONFIGS["join_last_token"], "cpu",
                                    num_rows=len(ids))
    h64 = hx["h"].to(torch.float64).numpy()
    g64, w64 = hx["gamma"].to(torch.float64).numpy(), hx["w8"].to(torch.float64).numpy()
    scale = 1.0 / np.sqrt(cfg.head_dim)
    tokens, n = 0, 0
    kv_cache = {}
    t0 = time.perf_counter()
    for j, s in enumerate(ids):
        c = cases[int(s)]
        ka, va = c["k_anc"], c["v_anc"]
        if kv_for is not None:
            if c["anchor"] not in kv_cache:
                kv_cache[c["anchor"]] = kv_for(c["anchor"])
            ka, va = kv_cache[c["anchor"]]
        ref = oracle.suffix_attention(c["q_suf"] * q_scale, ka, va, c["k_suf"], c["v_suf"],
                                      scale)
        if results is not None:
            results[int(s)] = (c["rows"], ref)
        if with_head:
            oracle.restricted_head(h64[j:j + 1], g64, w64, 1e-6)
        tokens += c["rows"][1] - c["rows"][0]
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return tokens / dt, threads, f"{n} seeded suffixes ({tokens} tokens) of the {cfg.name} workload", dt


def fp8_oracle_kv(t_bf16, layout):
    """kv_for(anchor) for the FP8 workloads: the oracle's own E4M3 quantisation of the
    anchor's bf16 K/V (rows copied to the host), dequantised."""
    import oracle
    ao = layout.anchor_offsets

    def kv_for(a):
        lo, hi = int(ao[a]), int(ao[a + 1])
        pair = []
        for name in ("k_anc", "v_anc"):
            blk = t_bf16[name][lo:hi].to("cpu", torch.float32).numpy()
            codes, scales = oracle.quantize_kv_fp8(blk, np.array([0, hi - lo]))
            pair.append(oracle.dequantize_kv_fp8(codes, scales, np.array([0, hi - lo])))
        return tuple(pair)
    return kv_for


def sampled_parity(results, out, lse):
    """Errors of the timed call's output against the oracle on the sampled suffixes. A
    failure to compute them is reported in the line (as `error`), not hidden."""
    if not results:
        return {"error": "no sampled suffixes"}
    try:
        return _sampled_parity(results, out, lse)
    except Exception as e:  # noqa: BLE001 - reported, never fatal to the measurement
        return {"error": f"{type(e).__name__}: {e}"[:300]}


def _sampled_parity(results, out, lse):
    g_o, r_o, g_l, r_l = [], [], [], []
    for (r0, r1), (ro, rl) in results.values():
        if r1 == r0:
            continue
        g_o.append(out[r0:r1].to("cpu", torch.float64).numpy())
        g_l.append(lse[r0:r1].to("cpu", torch.float64).numpy())
        r_o.append(ro)
        r_l.append(rl)
    go, ro_, gl, rl_ = (np.concatenate(x) for x in (g_o, r_o, g_l, r_l))
    return {"suffixes": len(results), "max_abs": float(np.abs(go - ro_).max()),
            "rel_l2": float(np.linalg.norm(go - ro_) / max(np.linalg.norm(ro_), 1e-30)),
            "lse_abs": float(np.abs(gl - rl_).max()),
            "finite": bool(np.isfinite(go).all() and np.isfinite(gl).all())}


def attention_config(cfg, layout, world, scaling="weak"):
    """The `config` object of an attention workload's line (both arms)."""
    hcfg = workloads.HEAD_CONFIGS["join_last_token"]
    par = "1 GPU" if world == 1 else (
        f"anchors split over {world} ranks (LPT), " +
        ("one batch" if scaling == "strong" else f"{world} batches"))
    return {"workload": cfg.name, "anchors": cfg.num_anchors,
            "anchor_len": list(cfg.anchor_len), "suffixes_per_anchor": cfg.suffixes_per_anchor,
            "suffix_len": list(cfg.suffix_len), "q_heads": cfg.num_q_heads,
            "kv_heads": cfg.num_kv_heads, "head_dim": cfg.head_dim,
            "kv_anchor": "e4m3 + per-(anchor, KV head) fp32 scales" if cfg.kv_fp8 else "bf16",
            "suffix_tokens": layout.total_suffix_tokens, "head_hidden": hcfg.hidden,
            "head_rows": layout.num_suffixes, "l2": "inputs larger than L2 (no flush)",
            "parallelism": par}


def _attn_cfg(args, name=None):
    cfg = workloads.ATTN_CONFIGS[name or args.workload]
    if args.suffixes_per_anchor:
        cfg = dataclasses.replace(cfg, suffixes_per_anchor=args.suffixes_per_anchor)
    return cfg


def run_reference(args):
    """--impl reference: the float64 CPU oracle, as it stands, on the host cores."""
    world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    name = args.workload if args.workload in ATTN_WORKLOADS else "ragged"
    cfg = _attn_cfg(args, name)
    layout = workloads.make_layout(cfg)
    # a bounded per-step sample (about a second of float64 work): the same 10 seeded
    # suffixes every step (drawn from the parity sample, which holds one suffix per 8
    # anchors and the extreme lengths), generated on the host
    ids = workloads.sample_suffixes(layout, 12, cfg.seed + 200)
    ids = np.sort(np.random.default_rng(cfg.seed + 201).choice(ids, min(10, len(ids)),
                                                                replace=False))
    sub_anchor = sorted(set(int(layout.suffix_anchor[s]) for s in ids))
    lens_a = [int(layout.anchor_lens[a]) for a in sub_anchor]
    groups = [[s for s in ids if layout.suffix_anchor[s] == a] for a in sub_anchor]
    sub = workloads.layout_from_lengths(lens_a, [len(g) for g in groups],
                                        [int(layout.suffix_lens[s]) for g in groups for s in g])
    t = workloads.make_attention_inputs(cfg, sub, "cpu")
    import oracle
    f64 = lambda x: x.to(torch.float64).numpy()
    arr = {k: f64(t[k]) for k in ("q_suf", "k_anc", "v_anc", "k_suf", "v_suf")}
    hx = workloads.make_head_inputs(workloads.HEAD_CONFIGS["join_last_token"], "cpu",
                                    num_rows=sub.num_suffixes)
    hh = [f64(hx[k]) for k in ("h", "gamma", "w8")]
    ao = sub.anchor_offsets

    def step():
        k_anc, v_anc = arr["k_anc"], arr["v_anc"]
        if cfg.kv_fp8:  # the oracle quantises and dequantises the anchors itself
            k_anc, v_anc = (oracle.dequantize_kv_fp8(*oracle.quantize_kv_fp8(x, ao), ao)
                            for x in (k_anc, v_anc))
        oracle.cascade_attention(arr["q_suf"], k_anc, v_anc, arr["k_suf"], arr["v_suf"],
                                 sub.anchor_offsets, sub.anchor_suffix_ptr, sub.suffix_offsets)
        oracle.restricted_head(hh[0], hh[1], hh[2], 1e-6)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = sub.total_suffix_tokens / dt
    cores = len(os.sched_getaffinity(0))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "suffix tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "strong" if args.strong else "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        # our arm's workload; every step times a bounded sample of it (cpu_baseline.sample)
        "config": attention_config(cfg, layout, world, "strong" if args.strong else "weak"),
        "cpu_baseline": {"value": value, "unit": "suffix tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{sub.num_suffixes} seeded suffixes ({sub.total_suffix_tokens} tokens) "
                                   f"of the {cfg.name} workload with their anchors, every step"},
        "e2e": {"value": value, "unit": "suffix tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------- our arm

def _events(n):
    return [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(n)]


def redo_items(ws) -> int:
    """Work items the fast kernel handed to the exact kernel in the last call (the
    workspace's int32 at byte 4)."""
    return int(ws[4:8].view(torch.int32).item())


def compare_two_pass(q, desc, t, out, lse, k_scale, v_scale, fused_ms, steps, stream,
                     parity_refs=None):
    """The same batch through quail_cascade_attn_two_pass (anchor pass, suffix pass, LSE
    merge) with the merge in the suffix pass's epilogue and as its own kernel: mean call
    time of each (CUDA events) against the fused call, and parity of each on the sampled
    suffixes. Writes its results into out / lse (after the fused call's parity was taken)."""
    ws2 = torch.empty(q.cascade_two_pass_workspace_size(desc), dtype=torch.uint8,
                      device=out.device)
    res = {"fused_ms": round(fused_ms, 4)}
    for merge, key in ((True, "merge_in_suffix_pass"), (False, "merge_kernel")):
        run = lambda: q.cascade_attn_two_pass(
            desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
            t["anchor_offsets"], t["anchor_suffix_ptr"], t["suffix_offsets"], out, lse, ws2,
            k_scale, v_scale, merge_in_suffix_pass=merge, stream=stream)
        for _ in range(2):
            run()
        torch.cuda.synchronize()
        evs = _events(steps)
        for a, b in evs:
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
        if q.get_device_error() != q.QUAIL_OK:
            raise RuntimeError("device error in the two-pass run")
        entry = {"ms": round(statistics.mean(a.elapsed_time(b) for a, b in evs), 4)}
        entry["vs_fused"] = round(entry["ms"] / fused_ms, 4)
        if parity_refs:
            entry["parity"] = sampled_parity(parity_refs, out, lse)
        res[key] = entry
    best = min(("fused", fused_ms), ("two_pass_merge_in_suffix_pass",
                                     res["merge_in_suffix_pass"]["ms"]),
               ("two_pass_merge_kernel", res["merge_kernel"]["ms"]), key=lambda x: x[1])
    res["faster"] = best[0]
    res["launches"] = {"fused": "3 schedule + fast + exact",
                       "two_pass": "fill + 2 x (3 schedule + fast + exact) (+ merge kernel)"}
    res["workspace_bytes"] = int(ws2.numel())
    del ws2
    torch.cuda.empty_cache()
    return res


def measure_attention(q, cfg, layout, dev, args, *, steps, e2e=False, cpu_budget=15.0,
                      world=1, rank=0, scaling="weak", fp8_diagnostic=False, two_pass=False):
    """One attention workload: cascade attention over the whole batch then the restricted
    head on the last token of every suffix, `steps` times on resident inputs. Returns the
    measurement dict (the headline line's keys, or a sub-object)."""
    hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    t = workloads.make_attention_inputs(cfg, layout, dev)
    kv_fp8 = cfg.kv_fp8
    k_scale = v_scale = None
    t_bf16 = dict(t)  # the bf16 anchor K/V stay referenced for the oracle's own quantisation
    if kv_fp8:
        ka = torch.empty(t["k_anc"].shape, dtype=torch.uint8, device=dev)
        va = torch.empty_like(ka)
        k_scale = torch.empty(layout.num_anchors, hkv, dtype=torch.float32, device=dev)
        v_scale = torch.empty_like(k_scale)
        q.quantize_kv_fp8(t["k_anc"], t["anchor_offsets"], ka, k_scale)
        q.quantize_kv_fp8(t["v_anc"], t["anchor_offsets"], va, v_scale)
        t["k_anc"], t["v_anc"] = ka, va
    desc = q.make_desc(layout.num_anchors, layout.num_suffixes, layout.total_anchor_tokens,
                       layout.total_suffix_tokens, layout.max_anchor_len, layout.max_suffix_len,
                       hq, hkv, d, 0.0, kv_fp8)
    ws = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device=dev)
    out = torch.empty(layout.total_suffix_tokens, hq, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(layout.total_suffix_tokens, hq, dtype=torch.float32, device=dev)
    # restricted head on the last token of every suffix; hidden states of all suffix tokens
    hcfg = workloads.HEAD_CONFIGS["join_last_token"]
    hx = workloads.make_head_inputs(hcfg, dev, num_rows=layout.total_suffix_tokens)
    last = torch.from_numpy((layout.suffix_offsets[1:] - 1).astype(np.int32)).to(dev)
    # the end-to-end leg's pinned host inputs, made before anything else churns host memory
    e2e_host = e2e_host_inputs(t, hx["h"], last, k_scale, v_scale) if e2e else None
    S = layout.num_suffixes
    logits = torch.empty(S, 8, dtype=torch.float32, device=dev)
    am = torch.empty(S, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        q.cascade_attn(desc, t["q_suf"], t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
                       t["anchor_offsets"], t["anchor_suffix_ptr"], t["suffix_offsets"], out,
                       lse, ws, k_scale, v_scale, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        q.restricted_head(hx["h"], hx["gamma"], hx["w8"], logits, am, eps=hcfg.eps,
                          row_index=last, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if q.get_device_error() != q.QUAIL_OK:
        raise RuntimeError(f"device error during warm-up ({cfg.name})")

    evs = _events(steps)
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clk:
        e_start.record(stream)
        for i in range(steps):
            step(evs[i])
        e_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = max_over_ranks(world, e_start.elapsed_time(e_end))
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    if q.get_device_error() != q.QUAIL_OK:
        raise RuntimeError(f"device error during the timed region ({cfg.name})")
    redo = redo_items(ws)
    ms_per_step = elapsed_ms / steps
    tokens = sum_over_ranks(world, float(layout.total_suffix_tokens))
    value = tokens / (ms_per_step / 1e3)

    pk, src = peaks()
    flops = attention_flops(layout, hq, d)
    achieved_tflops = flops / (attn_ms / 1e3) / 1e12
    peak = pk["bf16_tflops"]
    abytes = attention_bytes(layout, hq, hkv, d, 1 if kv_fp8 else 2)
    traffic = traffic_from_profile(
        "cascade.cu", ("cascade_pair_" if pair_kernel(layout, hq, hkv, d) else "cascade_attn_") +
        f"{cfg.name}.md")
    roofline = {"bound": "tensor", "achieved": round(achieved_tflops, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved_tflops / peak, 4),
                "traffic": traffic, "peak_source": f"bf16_tflops (burst) of {src}",
                "frac_of_sustained": (round(achieved_tflops / pk["bf16_tflops_sustained"], 4)
                                      if "bf16_tflops_sustained" in pk else None),
                "kernel": (("cascade_pair_kernel (CTA pairs)" if pair_kernel(layout, hq, hkv, d)
                            else "cascade_attn_kernel") + " fast launch + the exact launch "
                           "(+ 3 schedule kernels" +
                           (" and the e4m3 -> bf16 anchor staging kernel" if kv_fp8 else "") +
                           "): one quail_cascade_attn call"),
                "kernel_ms": round(attn_ms, 4),
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": abytes,
                "hbm_frac_of_algorithmic_bytes": round(abytes / (attn_ms / 1e3) / 1e9 /
                                                       pk["hbm_gbs"], 4),
                "redo_items": redo, "work_items": work_items(layout, hkv, hq // hkv)}

    from prefill_only_cascade_gb300 import cost_model
    plan = cost_model.plan_report(layout.anchor_offsets, layout.anchor_suffix_ptr,
                                  layout.suffix_offsets, hq, hkv, d, cost_model.default_hardware(),
                                  1 if kv_fp8 else 2)
    model = {"sol_ms": round(plan["sol_seconds"] * 1e3, 4),
             "mma_floor_ms": round(plan["mma_floor_seconds"] * 1e3, 4),
             "model_ms": round(plan["model_seconds"] * 1e3, 4),
             "measured_ms": round(attn_ms, 4)}

    res = {"value": value, "unit": "suffix tokens/s", "steps": steps,
           "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
           "dtype": "bf16 (fp32 accumulate)" if not kv_fp8 else "bf16 Q / e4m3 anchor KV",
           "config": attention_config(cfg, layout, world, scaling),
           "roofline": roofline, "cost_model": model,
           # per step: segments, schedule, items, (FP8: anchor staging), fast + exact
           # cascade kernels, head
           "gpu_launches": (7 if kv_fp8 and layout.total_anchor_tokens > 0 else 6) * steps,
           "clocks": clk.summary()}

    if e2e:
        # right after the device-timed region, while the box is in the same state (after
        # seconds of host-only work the copies ran ~10 % slower)
        res["e2e"] = run_e2e_chunked(q, cfg, layout, t, hx["h"], last, k_scale, v_scale, dev,
                                     stream, world, steps=max(3, min(steps, 6)),
                                     host=e2e_host, head_weights=(hx["gamma"], hx["w8"]),
                                     check=(out, logits, am))
        del e2e_host
    parity_refs = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        def host_cases(ids):
            return workloads.gather_suffix_case(t_bf16, layout, ids)
        v, cores, sample, dt = cpu_oracle_sample(
            layout, cfg, host_cases, budget_s=cpu_budget,
            kv_for=fp8_oracle_kv(t_bf16, layout) if kv_fp8 else None, results=parity_refs)
        res["parity"] = sampled_parity(parity_refs, out, lse)
        res["cpu_baseline"] = {
            "value": v, "unit": "suffix tokens/s", "cores": cores, "kind": "oracle",
            "sample": sample + (" (the oracle quantises each sampled anchor itself)"
                                if kv_fp8 else ""), "seconds": round(dt, 2)}
        if fp8_diagnostic and kv_fp8:
            # reported only: the FP8 path against the oracle on the UNQUANTISED bf16 anchor
            # K/V (the error the e4m3 anchor KV itself adds)
            diag = {}
            cpu_oracle_sample(layout, cfg, host_cases, budget_s=min(cpu_budget, 6.0),
                              max_suffixes=64, results=diag, with_head=False)
            res["diagnostic_vs_unquantised"] = sampled_parity(diag, out, lse)
    if two_pass:
        res["fused_vs_two_pass"] = compare_two_pass(
            q, desc, t, out, lse, k_scale, v_scale, attn_ms, max(3, min(steps, 5)), stream,
            parity_refs)
    del t, t_bf16, ws, out, lse, hx
    torch.cuda.empty_cache()
    return res


def h2d_bandwidth(dev, nbytes=1 << 30, reps=5):
    """Host-to-device copy rate of this machine: one pinned 1 GiB buffer copied with one
    cudaMemcpyAsync (torch copy_), best of `reps` (CUDA events)."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = None
    for _ in range(reps + 1):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    del src, dst
    return nbytes / (best / 1e3) / 1e9


def _chunks(layout, n):
    """n contiguous anchor groups of about equal suffix tokens (each one cascade call)."""
    so, asp = layout.suffix_offsets.astype(np.int64), layout.anchor_suffix_ptr.astype(np.int64)
    tok = so[asp[1:]]  # suffix tokens up to the end of each anchor
    A = layout.num_anchors
    cuts = [0]
    for c in range(1, n):
        a = int(np.searchsorted(tok, tok[-1] * c / n, side="left")) + 1
        if cuts[-1] < a < A:
            cuts.append(a)
    cuts.append(A)
    return [(cuts[i], cuts[i + 1]) for i in range(len(cuts) - 1)]


def e2e_host_inputs(t, h_all, last, k_scale, v_scale):
    """The step's inputs in pinned host memory (queries, anchor and suffix K/V, the hidden
    states of the last tokens, FP8 scales), as a caller of the end-to-end path holds them.
    Made once, early in the process: pinned buffers made after much host allocation churn
    (a second or third 57 GB set in one process) fed the host-to-device copies at ~155
    instead of ~210 GB/s on GB300."""
    def pinned_like(x):
        return torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    names = ["q_suf", "k_anc", "v_anc", "k_suf", "v_suf"]
    host = {k: pinned_like(t[k]) for k in names}
    for k in names:
        host[k].copy_(t[k])
    h_last = h_all.index_select(0, last.long())
    host["h"] = pinned_like(h_last)
    host["h"].copy_(h_last)
    del h_last
    if k_scale is not None:
        host["k_scale"] = pinned_like(k_scale)
        host["v_scale"] = pinned_like(v_scale)
        host["k_scale"].copy_(k_scale)
        host["v_scale"].copy_(v_scale)
    return host


def run_e2e_chunked(q, cfg, layout, t, h_all, last, k_scale, v_scale, dev, stream, world,
                    steps, n_chunks=8, host=None, head_weights=None, check=None):
    """Same metric through the C ABI with host buffers. Every step copies all of its inputs
    from pinned host memory (queries, anchor and suffix K/V, offsets, the hidden states of
    the last tokens) and reads the step's result (logits and argmax) back. The batch goes
    in anchor groups, one quail_cascade_attn + quail_restricted_head call each, through two
    sets of device buffers: group i + 1 is copied on a copy stream while group i computes,
    so copies and kernels overlap inside the timed region."""
    hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    ao = layout.anchor_offsets.astype(np.int64)
    asp = layout.anchor_suffix_ptr.astype(np.int64)
    so = layout.suffix_offsets.astype(np.int64)
    chunks = _chunks(layout, min(n_chunks, layout.num_anchors))
    # host copies of every input (pinned), written from the device-resident tensors
    if host is None:
        host = e2e_host_inputs(t, h_all, last, k_scale, v_scale)
    host = dict(host)
    sc = None
    if "k_scale" in host:
        sc = {"k": host.pop("k_scale"), "v": host.pop("v_scale")}
    plan = []
    for a0, a1 in chunks:
        s0, s1 = int(asp[a0]), int(asp[a1])
        ar, sr = (int(ao[a0]), int(ao[a1])), (int(so[s0]), int(so[s1]))
        offs = {"anchor_offsets": ao[a0:a1 + 1] - ao[a0],
                "anchor_suffix_ptr": asp[a0:a1 + 1] - s0,
                "suffix_offsets": so[s0:s1 + 1] - sr[0]}
        offs = {k: torch.from_numpy(v.astype(np.int32)).pin_memory() for k, v in offs.items()}
        la = np.diff(offs["anchor_offsets"].numpy())
        ls = np.diff(offs["suffix_offsets"].numpy())
        desc = q.make_desc(a1 - a0, s1 - s0, ar[1] - ar[0], sr[1] - sr[0],
                           int(la.max()) if la.size else 0, int(ls.max()) if ls.size else 0,
                           hq, hkv, d, 0.0, cfg.kv_fp8)
        plan.append({"a": (a0, a1), "s": (s0, s1), "ar": ar, "sr": sr, "offs": offs,
                     "desc": desc, "ws": q.cascade_workspace_size(desc)})
    mx = lambda f: max(f(p) for p in plan)
    max_ta, max_ts = mx(lambda p: p["ar"][1] - p["ar"][0]), mx(lambda p: p["sr"][1] - p["sr"][0])
    max_a, max_s = mx(lambda p: p["a"][1] - p["a"][0]), mx(lambda p: p["s"][1] - p["s"][0])
    kv_dt = t["k_anc"].dtype

    def dev_set():
        return {"q_suf": torch.empty(max(max_ts, 1), hq, d, dtype=torch.bfloat16, device=dev),
                "k_suf": torch.empty(max(max_ts, 1), hkv, d, dtype=torch.bfloat16, device=dev),
                "v_suf": torch.empty(max(max_ts, 1), hkv, d, dtype=torch.bfloat16, device=dev),
                "k_anc": torch.empty(max(max_ta, 1), hkv, d, dtype=kv_dt, device=dev),
                "v_anc": torch.empty(max(max_ta, 1), hkv, d, dtype=kv_dt, device=dev),
                "h": torch.empty(max(max_s, 1), host["h"].shape[1], dtype=torch.bfloat16,
                                 device=dev),
                "anchor_offsets": torch.empty(max_a + 1, dtype=torch.int32, device=dev),
                "anchor_suffix_ptr": torch.empty(max_a + 1, dtype=torch.int32, device=dev),
                "suffix_offsets": torch.empty(max_s + 1, dtype=torch.int32, device=dev),
                "k_scale": torch.empty(max(max_a, 1), hkv, dtype=torch.float32, device=dev),
                "v_scale": torch.empty(max(max_a, 1), hkv, dtype=torch.float32, device=dev)}
    bufs = [dev_set(), dev_set()]
    out = torch.empty(max(max_ts, 1), hq, d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(mx(lambda p: p["ws"]), dtype=torch.uint8, device=dev)
    hcfg = workloads.HEAD_CONFIGS["join_last_token"]
    if head_weights is not None:  # the device-resident step's RMSNorm gain and W8
        gamma, w8 = head_weights
    else:
        gamma, w8 = (workloads.make_head_inputs(hcfg, dev, num_rows=1)[k] for k in ("gamma", "w8"))
    S = layout.num_suffixes
    logits = torch.empty(max(max_s, 1), 8, dtype=torch.float32, device=dev)
    am = torch.empty(max(max_s, 1), dtype=torch.int32, device=dev)
    logits_h = torch.empty(S, 8, dtype=torch.float32, pin_memory=True)
    am_h = torch.empty(S, dtype=torch.int32, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    h2d += sum(x.numel() * 4 for p in plan for x in p["offs"].values())
    if sc is not None:
        h2d += sum(x.numel() * 4 for x in sc.values())
    d2h = S * (8 * 4 + 4)
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        p, b = plan[i % len(plan)], bufs[i % 2]
        (a0, a1), (s0, s1), (r0, r1), (u0, u1) = p["a"], p["s"], p["ar"], p["sr"]
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(consumed[i % 2])  # group i - 2 has read this set
            for k in ("q_suf", "k_suf", "v_suf"):
                b[k][:u1 - u0].copy_(host[k][u0:u1], non_blocking=True)
            for k in ("k_anc", "v_anc"):
                b[k][:r1 - r0].copy_(host[k][r0:r1], non_blocking=True)
            b["h"][:s1 - s0].copy_(host["h"][s0:s1], non_blocking=True)
            for k, v in p["offs"].items():
                b[k][:v.numel()].copy_(v, non_blocking=True)
            if sc is not None:
                b["k_scale"][:a1 - a0].copy_(sc["k"][a0:a1], non_blocking=True)
                b["v_scale"][:a1 - a0].copy_(sc["v"][a0:a1], non_blocking=True)
            copied[i % 2].record(copy_stream)

    def compute(i):
        p, b = plan[i % len(plan)], bufs[i % 2]
        s0, s1 = p["s"]
        stream.wait_event(copied[i % 2])
        ks, vs = (b["k_scale"], b["v_scale"]) if sc is not None else (None, None)
        q.cascade_attn(p["desc"], b["q_suf"], b["k_anc"], b["v_anc"], b["k_suf"], b["v_suf"],
                       b["anchor_offsets"], b["anchor_suffix_ptr"], b["suffix_offsets"], out,
                       None, ws, ks, vs, stream=stream)
        q.restricted_head(b["h"], gamma, w8, logits, am, eps=1e-6, n_rows=s1 - s0,
                          stream=stream)
        consumed[i % 2].record(stream)
        logits_h[s0:s1].copy_(logits[:s1 - s0], non_blocking=True)
        am_h[s0:s1].copy_(am[:s1 - s0], non_blocking=True)

    def run(n_steps, step_ends=None):
        n = n_steps * len(plan)
        copy_stream.wait_stream(stream)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            if step_ends is not None and (i + 1) % len(plan) == 0:
                step_ends[i // len(plan)].record(stream)

    run(1)
    torch.cuda.synchronize()
    barrier(world)
    bw = h2d_bandwidth(dev)
    # the copy rate of the step's own pinned inputs, a group-sized slice at a time with
    # nothing else running (min / median / max over the slices): the 1 GiB probe above
    # stays at ~211 GB/s on every box, while on some boxes the leg's copies ran at half
    # that or less
    rates = []
    for k in ("q_suf", "k_suf", "v_suf"):
        for p_ in plan:
            u0, u1 = p_["sr"]
            if u1 <= u0:
                continue
            src, dstb = host[k][u0:u1], bufs[0][k][:u1 - u0]
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            dstb.copy_(src, non_blocking=True)
            eb.record(stream)
            torch.cuda.synchronize()
            rates.append(src.numel() * src.element_size() / (ea.elapsed_time(eb) / 1e3) / 1e9)
    set_rates = ({"min": round(min(rates), 1), "median": round(statistics.median(rates), 1),
                  "max": round(max(rates), 1), "slices": len(rates)} if rates else None)
    a = torch.cuda.Event(enable_timing=True)
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    a.record(stream)
    run(steps, ends)
    torch.cuda.synchronize()
    ms = max_over_ranks(world, a.elapsed_time(ends[-1])) / steps
    step_ms = [round(a.elapsed_time(ends[0]), 1)] + [
        round(ends[i - 1].elapsed_time(ends[i]), 1) for i in range(1, steps)]
    # the same copy probe right after the timed steps: a lower rate here than before them
    # means the host link was shared with other work during the leg
    bw_after = h2d_bandwidth(dev)
    if q.get_device_error() != q.QUAIL_OK:
        raise RuntimeError("device error during the end-to-end run")
    # the results against the device-resident step's: every suffix's logits and argmax
    # (read back each step), and the attention output of the last anchor group
    agree = None
    if check is not None:
        out_full, logits_full, am_full = check
        u0, u1 = plan[-1]["sr"]
        attn = ((out[:u1 - u0].float() - out_full[u0:u1].float()).abs().max().item()
                if u1 > u0 else 0.0)
        agree = {"head_logits_argmax_identical": bool(torch.equal(logits_h, logits_full.cpu()) and
                                                      torch.equal(am_h, am_full.cpu())),
                 "last_group_attention_max_abs_diff": attn}
    del bufs, out, host, ws
    torch.cuda.empty_cache()
    copy_ms = h2d / (bw * 1e9) * 1e3
    return {"value": sum_over_ranks(world, float(layout.total_suffix_tokens)) / (ms / 1e3),
            "unit": "suffix tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms, "steps": steps, "anchor_groups": len(plan),
            "overlap": "inputs of anchor group i + 1 copied on a second stream while group i "
                       "computes",
            "step_ms": step_ms,
            "vs_resident": agree,
            "host_set_h2d_gbs": set_rates,
            "roofline": {"bound": "host-to-device copy", "h2d_gbs_measured": round(bw, 1),
                         "h2d_gbs_after": round(bw_after, 1),
                         "copy_bound_ms": round(copy_ms, 3),
                         "frac": round(copy_ms / ms, 4),
                         "how": "one pinned 1 GiB host-to-device copy (cudaMemcpyAsync), "
                                "best of 5, same process, before the timed steps (and "
                                "after them: h2d_gbs_after)"}}


def measure_softmax_stress(q, args, dev, scales=(4.0, 8.0)):
    """The join with its queries multiplied by 4 and by 8 (exact in bf16): scores of
    standard deviation ~4 and ~8 instead of ~1. Per scale: the cascade call's time, the
    work items the fast kernel handed to the exact kernel, and parity on sampled
    suffixes against the oracle given the same scaled queries."""
    cfg = _attn_cfg(args, "join")
    layout = workloads.make_layout(cfg)
    hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    t = workloads.make_attention_inputs(cfg, layout, dev)
    desc = q.make_desc(layout.num_anchors, layout.num_suffixes, layout.total_anchor_tokens,
                       layout.total_suffix_tokens, layout.max_anchor_len, layout.max_suffix_len,
                       hq, hkv, d)
    ws = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device=dev)
    out = torch.empty(layout.total_suffix_tokens, hq, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(layout.total_suffix_tokens, hq, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    pk, src = peaks()
    flops = attention_flops(layout, hq, d)
    items = work_items(layout, hkv, hq // hkv)
    # Bound for these peaked rows: the bf16 bounds, plus one bf16 rounding (2^-9
    # relative) of the largest |V|: the output is close to one V row, and the fast
    # kernel's P of that row is 2^(s c - m_ref) rounded to bf16 whenever the row max lies
    # past the first key tile (the same derivation as the FP8 path's bound).
    vmax = float(max(t["v_anc"].abs().max(), t["v_suf"].abs().max()))
    bound = {"max_abs": 2e-2 + vmax * 2.0 ** -9, "rel_l2": 5e-3, "lse_abs": 1e-3}
    res = {}
    for s in (1.0,) + tuple(scales):
        qs = t["q_suf"] * s
        run = lambda: q.cascade_attn(desc, qs, t["k_anc"], t["v_anc"], t["k_suf"], t["v_suf"],
                                     t["anchor_offsets"], t["anchor_suffix_ptr"],
                                     t["suffix_offsets"], out, lse, ws, stream=stream)
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        evs = _events(10)
        for a, b in evs:
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
        if q.get_device_error() != q.QUAIL_OK:
            raise RuntimeError(f"device error in the softmax stress run (x{s})")
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
        entry = {"ms": round(ms, 4), "redo_items": redo_items(ws), "work_items": items,
                 "tflops": round(flops / (ms / 1e3) / 1e12, 2),
                 "frac": round(flops / (ms / 1e3) / 1e12 / pk["bf16_tflops"], 4)}
        if not args.no_cpu_baseline:
            refs = {}
            cpu_oracle_sample(layout, cfg, lambda ids: workloads.gather_suffix_case(t, layout, ids),
                              budget_s=3.0, max_suffixes=48, with_head=False, results=refs,
                              q_scale=s)
            par = sampled_parity(refs, out, lse)
            par["bound"] = bound
            par["within_bound"] = ("max_abs" in par and par["max_abs"] <= bound["max_abs"] and
                                   par["rel_l2"] <= bound["rel_l2"] and
                                   par["lse_abs"] <= bound["lse_abs"])
            entry["parity"] = par
        res[f"x{s:g}"] = entry
        del qs
    del t, ws, out, lse
    torch.cuda.empty_cache()
    return {"workload": "join, queries scaled", "peak_source": f"bf16_tflops (burst) of {src}",
            "by_query_scale": res}


def head_oracle_sample(h, gamma, w8, eps, logits, argmax, rows=65536):
    """The oracle's RMSNorm + 8-column head on the first `rows` rows (host cores, timed),
    and the kernel's output there against it: logits max |err|, argmax agreement where
    the oracle's top-2 margin exceeds 1e-2."""
    import oracle
    n = min(rows, h.shape[0])
    h64 = h[:n].to("cpu", torch.float64).numpy()
    g64, w64 = gamma.to("cpu", torch.float64).numpy(), w8.to("cpu", torch.float64).numpy()
    t0 = time.perf_counter()
    ref_logits, ref_am = oracle.restricted_head(h64, g64, w64, eps)
    dt = time.perf_counter() - t0
    lg = logits[:n].to("cpu", torch.float64).numpy()
    am = argmax[:n].cpu().numpy()
    sure = oracle.top2_margin(ref_logits) > 1e-2
    cpu = {"value": n / dt, "unit": "rows/s", "cores": len(os.sched_getaffinity(0)),
           "kind": "oracle", "sample": f"the first {n} rows", "seconds": round(dt, 2)}
    parity = {"rows": n, "logits_max_abs": float(np.abs(lg - ref_logits).max()),
              "argmax_checked": int(sure.sum()),
              "argmax_mismatches": int((am[sure] != ref_am[sure]).sum())}
    return cpu, parity


def quantize_oracle_sample(kv, anchor_offsets, codes, scale, anchors=8):
    """The oracle's E4M3 quantisation of the first `anchors` anchors (host cores, timed),
    and the kernel's codes and scales there against it, bit for bit."""
    import oracle
    hi = int(anchor_offsets[anchors])
    x = kv[:hi].to("cpu", torch.float32).numpy()
    t0 = time.perf_counter()
    ref_codes, ref_scale = oracle.quantize_kv_fp8(x, np.asarray(anchor_offsets[:anchors + 1]))
    dt = time.perf_counter() - t0
    got_codes = codes[:hi].cpu().numpy()
    got_scale = scale[:anchors].cpu().numpy()
    cpu = {"value": x.size / dt, "unit": "elements/s", "cores": len(os.sched_getaffinity(0)),
           "kind": "oracle", "sample": f"the first {anchors} anchor(s), {x.size} elements",
           "seconds": round(dt, 2)}
    parity = {"elements": int(x.size),
              "code_mismatches": int((got_codes != ref_codes).sum()),
              "scale_mismatches": int((got_scale != ref_scale).sum())}
    return cpu, parity


def measure_bandwidth_kernel(q, args, kind, steps):
    """Per-kernel measurement of the HBM-bound kernels:
    head      restricted head on 2,000,000 rows x 2,560 (bf16)
    quantize  E4M3 quantisation of the long-anchor workload's anchor K: the line is the
              given-scale quantiser (the max |x| of every (anchor, KV head) known, as the
              causal prefill emits it: one read and one write per element); `standalone`
              is quail_quantize_kv_fp8, which forms the max itself (one read, the slab held
              on chip across a cluster)
    Returns the kernel's CUDA-event time (L2 flushed between launches), its HBM roofline,
    the oracle baseline and parity."""
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    pk, src = peaks()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def timed(run):
        for _ in range(max(args.warmup, 3)):
            run()
        torch.cuda.synchronize()
        evs = _events(steps)
        with ClockSampler(0) as clk:
            for a, b in evs:
                flush.zero_()  # evict L2 (larger than L2) between timed launches
                a.record(stream)
                run()
                b.record(stream)
            torch.cuda.synchronize()
        if q.get_device_error() != q.QUAIL_OK:
            raise RuntimeError(f"device error during the timed region ({kind})")
        return statistics.median(a.elapsed_time(b) for a, b in evs), clk.summary()

    def roofline(algo_bytes, ms, kernel, traffic):
        gbs = algo_bytes / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / pk["hbm_gbs"], 4), "traffic": traffic,
                "peak_source": f"hbm_gbs of {src}", "kernel": kernel, "kernel_ms": round(ms, 4),
                "algorithmic_bytes_per_launch": algo_bytes}

    sub = {}
    if kind == "head":
        cfg = workloads.HEAD_CONFIGS["head"]
        n = args.head_rows or cfg.num_rows
        x = workloads.make_head_inputs(cfg, dev, num_rows=n)
        logits = torch.empty(n, 8, dtype=torch.float32, device=dev)
        am = torch.empty(n, dtype=torch.int32, device=dev)
        run = lambda: q.restricted_head(x["h"], x["gamma"], x["w8"], logits, am, eps=cfg.eps,
                                        stream=stream)
        algo_bytes = n * (cfg.hidden * 2 + 8 * 4 + 4) + cfg.hidden * 2 * 9
        units, unit = n, "rows/s"
        config = {"workload": "head", "rows": n, "hidden": cfg.hidden}
        ms, clocks = timed(run)
        roof = roofline(algo_bytes, ms, "restricted_head_kernel",
                        traffic_from_profile("head.cu", "restricted_head.md"))
    else:
        cfg = workloads.ATTN_CONFIGS["fp8_long"]
        lay = workloads.make_layout(cfg)
        g = torch.Generator(device=dev).manual_seed(4)
        kv = workloads._randn_bf16((lay.total_anchor_tokens, cfg.num_kv_heads, cfg.head_dim), g, dev)
        codes = torch.empty(kv.shape, dtype=torch.uint8, device=dev)
        scale = torch.empty(cfg.num_anchors, cfg.num_kv_heads, dtype=torch.float32, device=dev)
        ao = torch.from_numpy(lay.anchor_offsets.copy()).to(dev)
        # input of the given-scale call (in the pipeline the causal prefill's k_amax): max
        # |x| per (anchor, KV head), every anchor of this workload having the same length
        la = cfg.anchor_len[0]
        amax = kv.view(cfg.num_anchors, la, cfg.num_kv_heads, cfg.head_dim).abs().amax(
            dim=(1, 3)).float().contiguous()
        algo_bytes = kv.numel() * 3 + scale.numel() * 4
        units, unit = kv.numel(), "elements/s"
        config = {"workload": "quantize", "anchors": cfg.num_anchors,
                  "anchor_len": cfg.anchor_len[0], "kv_heads": cfg.num_kv_heads,
                  "head_dim": cfg.head_dim, "scales": "given (max |x| per anchor and KV head)"}
        codes_sa = torch.empty_like(codes)
        scale_sa = torch.empty_like(scale)
        ms_sa, clocks_sa = timed(lambda: q.quantize_kv_fp8(kv, ao, codes_sa, scale_sa,
                                                           stream=stream))
        sub["standalone"] = {
            "kernel_ms": round(ms_sa, 4),
            "roofline": roofline(algo_bytes, ms_sa, "kv_quantize_kernel (forms the max itself)",
                                 traffic_from_profile("quantize.cu", "quantize_fp8_long.md")),
            "clocks": clocks_sa}
        ms, clocks = timed(lambda: q.quantize_kv_fp8_with_scales(kv, ao, amax, codes, scale,
                                                                 stream=stream))
        roof = roofline(algo_bytes, ms, "kv_quantize_scaled_kernel (given scales)",
                        traffic_from_profile("quantize.cu", "quantize_scaled_fp8_long.md"))
        sub["standalone"]["same_codes_as_given_scale"] = bool(
            torch.equal(codes, codes_sa) and torch.equal(scale, scale_sa))
    del flush
    cpu = parity = None
    if not args.no_cpu_baseline:
        if kind == "head":
            cpu, parity = head_oracle_sample(x["h"], x["gamma"], x["w8"], cfg.eps, logits, am)
        else:
            cpu, parity = quantize_oracle_sample(kv, lay.anchor_offsets, codes, scale)
            sub["standalone"]["parity"] = quantize_oracle_sample(
                kv, lay.anchor_offsets, codes_sa, scale_sa, anchors=1)[1]
    config["l2"] = "flushed between launches"
    res = {"metric": f"{kind} kernel throughput", "value": units / (ms / 1e3), "unit": unit,
           "steps": steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
           "config": config, "roofline": roof,
           "cpu_baseline": cpu, "parity": parity, "gpu_launches": steps,
           "clocks": clocks}
    if sub:
        res["sub"] = sub
    if kind == "head":
        del x, logits, am
    else:
        del kv, codes, scale, codes_sa, scale_sa, amax
    torch.cuda.empty_cache()
    return res


def run_bandwidth_kernel(args):
    import prefill_only_cascade_gb300 as q
    torch.cuda.set_device(0)
    res = measure_bandwidth_kernel(q, args, args.workload, args.steps)
    line = {"metric": res.pop("metric"), **res, "n_gpus": 1, "higher_is_better": True,
            "data": "synthetic"}
    print(json.dumps(line))


def run_ours(args):
    import prefill_only_cascade_gb300 as q

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = _attn_cfg(args)
    scaling = "strong" if (args.strong and world > 1) else "weak"
    layout, shard_plan = rank_layout(cfg, world, rank, strong=args.strong)
    cfg_rank = dataclasses.replace(cfg, seed=cfg.seed + 7919 * rank) if rank else cfg
    head = measure_attention(q, cfg_rank, layout, dev, args, steps=args.steps,
                             e2e=not args.no_e2e, world=world, rank=rank, scaling=scaling,
                             two_pass=(world == 1 and not args.no_sub))
    line = {"metric": METRIC, "value": head.pop("value"), "unit": head.pop("unit"),
            "n_gpus": world, "steps": head.pop("steps"), "warmup": head.pop("warmup"),
            "ms_per_step": head.pop("ms_per_step"), "higher_is_better": True,
            "scaling": scaling, "vs_baseline": None, "dtype": head.pop("dtype"),
            "data": "synthetic (seeded N(0,1) bf16)", **head}
    line.setdefault("cpu_baseline", None)
    line.setdefault("parity", None)
    line.setdefault("e2e", None)
    if shard_plan is not None:
        line["shard_plan"] = shard_plan
    if rank == 0 and world == 1 and not args.no_sub and cfg.name == "ragged":
        sub = {}
        sub_steps = max(3, min(args.steps, 10))
        for name, budget in (("join", 8.0), ("fp8_long", 8.0)):
            c = _attn_cfg(args, name)
            sub[name] = measure_attention(q, c, workloads.make_layout(c), dev, args,
                                          steps=sub_steps, cpu_budget=budget,
                                          fp8_diagnostic=(name == "fp8_long"), two_pass=True)
        sub["head"] = measure_bandwidth_kernel(q, args, "head", sub_steps)
        sub["softmax_stress"] = measure_softmax_stress(q, args, dev)
        line["sub"] = sub
    if rank == 0:
        print(json.dumps(line))


def run_prefill(args):
    """Per-kernel line for quail_causal_prefill_attn (the anchors' own causal prefill; not
    the headline): 64 sequences x 4,096 tokens, 32/8 heads, d = 128. Inputs larger than L2."""
    import prefill_only_cascade_gb300 as q
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    pk, src = peaks()
    cfg = workloads.ATTN_CONFIGS["prefill"]
    if args.sequences:
        cfg = dataclasses.replace(cfg, num_anchors=args.sequences)
    lay = workloads.make_layout(cfg)
    t = workloads.make_attention_inputs(cfg, lay, dev)
    hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    T, S, L = lay.total_suffix_tokens, lay.num_suffixes, lay.max_suffix_len
    ws = torch.empty(q.causal_prefill_workspace_size(S, T, L, hq, hkv, d), dtype=torch.uint8,
                     device=dev)
    out = torch.empty(T, hq, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(T, hq, dtype=torch.float32, device=dev)
    run = lambda: q.causal_prefill_attn(t["q_suf"], t["k_suf"], t["v_suf"], t["suffix_offsets"],
                                        out, L, lse=lse, workspace=ws, stream=stream)
    for _ in range(max(args.warmup, 3)):
        run()
    torch.cuda.synchronize()
    if q.get_device_error() != q.QUAIL_OK:
        raise RuntimeError("device error during warm-up")
    evs = _events(args.steps)
    with ClockSampler(0) as clk:
        for a, b in evs:
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    flops = attention_flops(lay, hq, d)   # 4 d Hq sum over sequences of L (L + 1) / 2
    tflops = flops / (ms / 1e3) / 1e12
    line = {"metric": "causal prefill tokens/sec", "value": T / (ms / 1e3), "unit": "tokens/s",
            "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms,
            "higher_is_better": True, "dtype": "bf16 (fp32 accumulate)",
            "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": "prefill", "sequences": S, "sequence_len": L, "q_heads": hq,
                       "kv_heads": hkv, "head_dim": d, "l2": "inputs larger than L2 (no flush)"},
            "roofline": {"bound": "tensor", "achieved": round(tflops, 2),
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(tflops / pk["bf16_tflops"], 4),
                         "traffic": traffic_from_profile(
                             "cascade.cu", "cascade_pair_prefill.md" if pair_kernel(lay, hq, hkv, d)
                             else "cascade_attn_prefill.md"),
                         "peak_source": f"bf16_tflops (burst) of {src}",
                         "kernel": (("cascade_pair_kernel (CTA pairs)" if pair_kernel(lay, hq, hkv, d) else "cascade_attn_kernel") + " with anchors of length 0, one call"),
                         "algorithmic_flops_per_launch": flops},
            "gpu_launches": 6 * args.steps, "clocks": clk.summary()}
    if not args.no_cpu_baseline:
        # the oracle on one seeded sequence at least (each is 4,096 tokens of causal
        # attention: ~20 s of float64 work on the host cores)
        parity_refs = {}
        v, cores, sample, dt = cpu_oracle_sample(
            lay, cfg, lambda ids: workloads.gather_suffix_case(t, lay, ids), budget_s=15.0,
            max_suffixes=4, with_head=False, results=parity_refs)
        line["parity"] = sampled_parity(parity_refs, out, lse)
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample, "seconds": round(dt, 2)}
    from prefill_only_cascade_gb300 import cost_model
    plan = cost_model.plan_report(lay.anchor_offsets, lay.anchor_suffix_ptr, lay.suffix_offsets,
                                  hq, hkv, d, cost_model.default_hardware())
    line["cost_model"] = {"sol_ms": round(plan["sol_seconds"] * 1e3, 4),
                          "mma_floor_ms": round(plan["mma_floor_seconds"] * 1e3, 4),
                          "model_ms": round(plan["model_seconds"] * 1e3, 4),
                          "measured_ms": round(ms, 4)}
    line["fused_quantise"] = prefill_quantise_pair(q, t, lay, out, lse, ws, ms, args, stream, pk,
                                                   src)
    print(json.dumps(line))


def prefill_quantise_pair(q, t, lay, out, lse, ws, prefill_ms, args, stream, pk, src):
    """The anchors' prefill followed by their FP8 quantisation, two ways: (a) the prefill
    emits the K/V amax per (sequence, KV head) from the tiles it loads, then
    quail_quantize_kv_fp8_with_scales reads K and V once; (b) the plain prefill, then the
    standalone quail_quantize_kv_fp8 (which finds the amax itself). Times (CUDA events,
    median; the quantise calls with L2 flushed before each), HBM fractions of the quantise
    calls (3 algorithmic bytes per element) and a bit-for-bit check that (a) and (b) give
    the same codes and scales."""
    T, hkv, d = t["k_suf"].shape
    S = lay.num_suffixes
    L = lay.max_suffix_len
    k_amax = torch.empty(S, hkv, dtype=torch.float32, device=out.device)
    v_amax = torch.empty_like(k_amax)
    codes = {n: torch.empty(t[n].shape, dtype=torch.uint8, device=out.device)
             for n in ("k_suf", "v_suf")}
    scale = {n: torch.empty(S, hkv, dtype=torch.float32, device=out.device)
             for n in ("k_suf", "v_suf")}
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=out.device)

    def timed(fn, n, flush_l2):
        evs = _events(n)
        for a, b in evs:
            if flush_l2:
                flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    pre_amax = lambda: q.causal_prefill_attn(t["q_suf"], t["k_suf"], t["v_suf"],
                                             t["suffix_offsets"], out, L, lse=lse, workspace=ws,
                                             k_amax=k_amax, v_amax=v_amax, stream=stream)
    pre_amax()
    torch.cuda.synchronize()
    steps = max(3, min(args.steps, 10))
    amax_ms = timed(pre_amax, steps, False)
    scaled = {n: (lambda n=n: q.quantize_kv_fp8_with_scales(
        t[n], t["suffix_offsets"], k_amax if n == "k_suf" else v_amax, codes[n], scale[n],
        stream=stream)) for n in codes}
    plain = {n: (lambda n=n: q.quantize_kv_fp8(t[n], t["suffix_offsets"], codes[n], scale[n],
                                               stream=stream)) for n in codes}
    for fn in list(scaled.values()) + list(plain.values()):
        fn()
    torch.cuda.synchronize()
    ref = {n: (codes[n].clone(), scale[n].clone()) for n in codes}   # from the plain call
    scaled_ms = {n: timed(scaled[n], steps, True) for n in codes}
    same = all(torch.equal(codes[n], ref[n][0]) and torch.equal(scale[n], ref[n][1])
               for n in codes)
    plain_ms = {n: timed(plain[n], steps, True) for n in codes}
    if q.get_device_error() != q.QUAIL_OK:
        raise RuntimeError("device error in the prefill + quantise measurement")
    del flush
    algo = T * hkv * d * 3 + S * hkv * 4
    frac = lambda ms_: round(algo / (ms_ / 1e3) / 1e9 / pk["hbm_gbs"], 4)
    return {
        "prefill_ms": round(prefill_ms, 4), "prefill_with_amax_ms": round(amax_ms, 4),
        "quantise_with_scales_ms": {n: round(v, 4) for n, v in scaled_ms.items()},
        "quantise_with_scales_hbm_frac": {n: frac(v) for n, v in scaled_ms.items()},
        "standalone_quantise_ms": {n: round(v, 4) for n, v in plain_ms.items()},
        "standalone_quantise_hbm_frac": {n: frac(v) for n, v in plain_ms.items()},
        "pair_ms": {"amax_then_scaled": round(amax_ms + sum(scaled_ms.values()), 4),
                    "plain_then_standalone": round(prefill_ms + sum(plain_ms.values()), 4)},
        "codes_and_scales_identical": bool(same),
        "algorithmic_bytes_per_quantise": algo, "peak_source": f"hbm_gbs of {src}"}


def run_kvplan(args):
    """Query-aware anchor-KV cache plan (host code, no GPU): regret tokens of a general
    server's LRU against furthest-next-use on seeded synthetic join plans, and the
    planner's throughput. One JSON line; value = furthest-next-use regret on the zipf plan."""
    import prefill_only_cascade_gb300 as q
    res = {}
    for name, cfg in workloads.KV_PLAN_CONFIGS.items():
        acc, size, cap = workloads.make_kv_plan(cfg)
        row = {"accesses": int(acc.size), "anchors": int(size.size), "capacity_tokens": cap}
        for pol, label in ((q.KV_LRU, "lru"), (q.KV_FURTHEST_NEXT_USE, "furthest_next_use")):
            t0 = time.perf_counter()
            for _ in range(max(args.steps, 1)):
                _, st = q.kv_plan(acc, size, cap, pol)
            dt = (time.perf_counter() - t0) / max(args.steps, 1)
            row[label] = {"regret_tokens": st["regret_tokens"], "hits": st["hits"],
                          "accesses_per_s": acc.size / dt}
            row["compulsory_tokens"] = st["compulsory_tokens"]
        res[name] = row
    z = res["zipf"]
    line = {"metric": "KV regret tokens (query-aware anchor cache, zipf plan)",
            "value": z["furthest_next_use"]["regret_tokens"], "unit": "tokens",
            "higher_is_better": False, "n_gpus": 0, "steps": max(args.steps, 1),
            "data": "synthetic seeded join plans", "config": {"workload": "kvplan"},
            "plans": res}
    print(json.dumps(line))


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.workload in ("head", "quantize"):
        run_bandwidth_kernel(args)
    elif args.workload == "prefill":
        run_prefill(args)
    elif args.workload == "kvplan":
        run_kvplan(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
