"""Benchmark of the prefill-only AI.IF / AI_JOIN hot path on GB300.

One step = one pass of the whole path over one batch: the cascade attention over every
suffix token of the workload, then the restricted head (RMSNorm + 8 columns + argmax) on
the last token of every suffix. Default workload: the Qwen3-4B-shaped join (8 anchors of
1,024 tokens, 4,144 suffixes each, suffix length U[8, 24], 32 query / 8 KV heads,
d = 128; hidden size 2,560 for the head). Inputs are synthetic and seeded and already
resident in HBM; they are larger than L2, so L2 is not flushed between steps.

Prints ONE JSON line (metric: suffix tokens per second). `--impl reference` times the
float64 CPU oracle on a bounded sample of the same workload instead.
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


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="join",
                    choices=["join", "ragged", "fp8_long", "head", "quantize", "prefill",
                             "kvplan"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--head-rows", type=int, default=None,
                    help="fewer rows for --workload head (profiling only)")
    ap.add_argument("--suffixes-per-anchor", type=int, default=None,
                    help="smaller case of the same workload (profiling only)")
    return ap.parse_args()


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


def traffic_from_profile(kernel_file: str, profile_md: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the current
    kernel source (the summary records the source's sha256)."""
    path = os.path.join(ROOT, "profiles", profile_md)
    src = os.path.join(ROOT, "prefill_only_cascade_gb300", "csrc", kernel_file)
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    vals = {}
    for line in open(path):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != sha:
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


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


def rank_workload(cfg, rank: int):
    """Weak scaling: every rank gets its own batch of the same shape (independent anchors
    with their suffixes; nothing is exchanged between ranks), drawn with a rank-specific
    seed."""
    import dataclasses
    return dataclasses.replace(cfg, seed=cfg.seed + 7919 * rank) if rank else cfg


# ---------------------------------------------------------------------------- oracle timing

def cpu_oracle_sample(layout, cfg, t_host_fn, budget_s=15.0, max_suffixes=1024, kv_for=None,
                      with_head=True, results=None):
    """Time the float64 oracle (attention of each suffix + its head row) on host cores over a
    seeded sample of suffixes until `budget_s` is spent. kv_for(anchor) -> (k, v) float64
    replaces the anchor K/V (FP8: the oracle quantises and dequantises the anchor itself,
    once per anchor, inside the timed loop). With a dict `results`, each sampled suffix's
    oracle (out, lse) is stored under its id. Returns tokens/s and details."""
    import oracle
    try:
        from threadpoolctl import threadpool_info
        threads = max([i.get("num_threads", 1) for i in threadpool_info()] or [1])
    except Exception:  # threadpoolctl is not installed everywhere
        threads = len(os.sched_getaffinity(0))
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
        ref = oracle.suffix_attention(c["q_suf"], ka, va, c["k_suf"], c["v_suf"], scale)
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
    """Errors of the timed call's output against the oracle on the sampled suffixes."""
    if not results:
        return None
    try:
        return _sampled_parity(results, out, lse)
    except Exception as e:  # a reporting aid: never fail the measurement over it
        print(f"parity figures unavailable: {e}", file=sys.stderr)
        return None


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
            "lse_abs": float(np.abs(gl - rl_).max())}


def attention_config(cfg, layout, world):
    """The `config` object of an attention workload's line (both arms)."""
    hcfg = workloads.HEAD_CONFIGS["join_last_token"]
    return {"workload": cfg.name, "anchors": cfg.num_anchors,
            "anchor_len": list(cfg.anchor_len), "suffixes_per_anchor": cfg.suffixes_per_anchor,
            "suffix_len": list(cfg.suffix_len), "q_heads": cfg.num_q_heads,
            "kv_heads": cfg.num_kv_heads, "head_dim": cfg.head_dim,
            "suffix_tokens": layout.total_suffix_tokens, "head_hidden": hcfg.hidden,
            "head_rows": layout.num_suffixes, "l2": "inputs larger than L2 (no flush)",
            "parallelism": f"replicas x{world}"}


def run_reference(args):
    """--impl reference: the float64 CPU oracle, as it stands, on the host cores."""
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return
    cfg = workloads.ATTN_CONFIGS[args.workload]
    if args.suffixes_per_anchor:
        cfg = dataclasses.replace(cfg, suffixes_per_anchor=args.suffixes_per_anchor)
    layout = workloads.make_layout(cfg)
    # a bounded per-step sample: the same seeded suffixes every step, generated on the host
    ids = workloads.sample_suffixes(layout, 48, cfg.seed + 200)
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

    def step():
        oracle.cascade_attention(arr["q_suf"], arr["k_anc"], arr["v_anc"], arr["k_suf"],
                                 arr["v_suf"], sub.anchor_offsets, sub.anchor_suffix_ptr,
                                 sub.suffix_offsets)
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
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        # our arm's workload; every step times a bounded sample of it (cpu_baseline.sample)
        "config": attention_config(cfg, layout, world),
        "cpu_baseline": {"value": value, "unit": "suffix tokens/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"{sub.num_suffixes} seeded suffixes ({sub.total_suffix_tokens} tokens) "
                                   f"of the {cfg.name} workload with their anchors, every step"},
        "e2e": {"value": value, "unit": "suffix tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---------------------------------------------------------------------------- our arm

def run_ours(args):
    import dataclasses

    import prefill_only_cascade_gb300 as q

    world, rank, local = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workloads.ATTN_CONFIGS[args.workload]
    if args.suffixes_per_anchor:
        cfg = dataclasses.replace(cfg, suffixes_per_anchor=args.suffixes_per_anchor)
    cfg = rank_workload(cfg, rank)
    layout = workloads.make_layout(cfg)
    hq, hkv, d = cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
    t = workloads.make_attention_inputs(cfg, layout, dev)
    kv_fp8 = cfg.kv_fp8
    k_scale = v_scale = None
    t_bf16 = dict(t)  # the bf16 anchor K/V stay referenced for the oracle's own quantisation
    if kv_fp8:
        ka = torch.empty(t["k_anc"].shape, dtype=torch.uint8, device=dev)
        va = torch.empty_like(ka)
        k_scale = torch.empty(cfg.num_anchors, hkv, dtype=torch.float32, device=dev)
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
        raise RuntimeError("device error during warm-up")

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        time.sleep(0.3)  # let the sampler start
        e_start.record(stream)
        for i in range(args.steps):
            step(evs[i])
        e_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = max_over_ranks(world, e_start.elapsed_time(e_end))
    attn_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    if q.get_device_error() != q.QUAIL_OK:
        raise RuntimeError("device error during the timed region")
    ms_per_step = elapsed_ms / args.steps
    tokens = sum_over_ranks(world, float(layout.total_suffix_tokens))
    value = tokens / (ms_per_step / 1e3)

    pk, src = peaks()
    flops = attention_flops(layout, hq, d)
    achieved_tflops = flops / (attn_ms / 1e3) / 1e12
    peak = pk["bf16_tflops"]
    traffic = traffic_from_profile("cascade.cu", f"cascade_attn_{cfg.name}.md")
    roofline = {"bound": "tensor", "achieved": round(achieved_tflops, 2), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved_tflops / peak, 4),
                "traffic": traffic, "peak_source": f"bf16_tflops (burst) of {src}",
                "frac_of_sustained": (round(achieved_tflops / pk["bf16_tflops_sustained"], 4)
                                      if "bf16_tflops_sustained" in pk else None),
                "kernel": "cascade_attn_kernel, fast + exact launches (+ its 3 schedule "
                          "kernels" + (" and the e4m3 -> bf16 anchor staging kernel"
                                       if kv_fp8 else "") + "): one quail_cascade_attn call",
                "kernel_ms": round(attn_ms, 4),
                "algorithmic_flops_per_launch": flops,
                "algorithmic_bytes_per_launch": attention_bytes(
                    layout, hq, hkv, d, 1 if kv_fp8 else 2),
                "hbm_frac_of_algorithmic_bytes": round(
                    attention_bytes(layout, hq, hkv, d, 1 if kv_fp8 else 2) /
                    (attn_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}

    from prefill_only_cascade_gb300 import cost_model
    plan = cost_model.plan_report(layout.anchor_offsets, layout.anchor_suffix_ptr,
                                  layout.suffix_offsets, hq, hkv, d, cost_model.default_hardware(),
                                  1 if kv_fp8 else 2)
    model = {"sol_ms": round(plan["sol_seconds"] * 1e3, 4),
             "mma_floor_ms": round(plan["mma_floor_seconds"] * 1e3, 4),
             "model_ms": round(plan["model_seconds"] * 1e3, 4),
             "measured_ms": round(attn_ms, 4)}

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, q, desc, layout, t, hx, last, k_scale, v_scale, dev, stream, world)

    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        def host_cases(ids):
            return workloads.gather_suffix_case(t_bf16, layout, ids)
        parity_refs = {}
        v, cores, sample, dt = cpu_oracle_sample(
            layout, cfg, host_cases, kv_for=fp8_oracle_kv(t_bf16, layout) if kv_fp8 else None,
            results=parity_refs)
        parity = sampled_parity(parity_refs, out, lse)
        cpu = {"value": v, "unit": "suffix tokens/s", "cores": cores, "kind": "oracle",
               "sample": sample + (" (the oracle quantises each sampled anchor itself)"
                                   if kv_fp8 else ""), "seconds": round(dt, 2)}

    line = {
        "metric": METRIC, "value": value, "unit": "suffix tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (fp32 accumulate)" if not kv_fp8 else "bf16 Q / e4m3 anchor KV",
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": attention_config(cfg, layout, world),
        "roofline": roofline, "cost_model": model, "cpu_baseline": cpu, "e2e": e2e,
        # the timed call's output against the oracle on the CPU baseline's sampled suffixes
        "parity": parity,
        # per step: segments, schedule, items, (FP8: anchor staging), fast + exact cascade
        # kernels, head
        "gpu_launches": (7 if kv_fp8 and layout.total_anchor_tokens > 0 else 6) * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0:
        print(json.dumps(line))


def run_e2e(args, q, desc, layout, t, hx, last, k_scale, v_scale, dev, stream, world):
    """Same metric through the C ABI with host buffers: every step copies its inputs from
    pinned host memory and reads the step's result (logits and argmax) back. Two sets of
    device input buffers: the copies of step i + 1 run on a copy stream while step i
    computes (copy engines and SMs overlap; every step's copies are inside the timed
    region)."""
    names = ["q_suf", "k_anc", "v_anc", "k_suf", "v_suf", "anchor_offsets",
             "anchor_suffix_ptr", "suffix_offsets"]
    host = {k: t[k].cpu().pin_memory() for k in names}
    host["h"] = hx["h"].index_select(0, last.long()).cpu().pin_memory()
    bufs = [{k: torch.empty(v.shape, dtype=v.dtype, device=dev) for k, v in host.items()}
            for _ in range(2)]
    S = layout.num_suffixes
    logits = torch.empty(S, 8, dtype=torch.float32, device=dev)
    am = torch.empty(S, dtype=torch.int32, device=dev)
    logits_h = torch.empty(S, 8, dtype=torch.float32).pin_memory()
    am_h = torch.empty(S, dtype=torch.int32).pin_memory()
    out = torch.empty(layout.total_suffix_tokens, desc.num_q_heads, desc.head_dim,
                      dtype=torch.bfloat16, device=dev)
    ws = torch.empty(q.cascade_workspace_size(desc), dtype=torch.uint8, device=dev)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = logits_h.numel() * 4 + am_h.numel() * 4
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]

    def copy_in(i):
        b = bufs[i % 2]
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(consumed[i % 2])  # step i - 2 has read this set
            for k, v in host.items():
                b[k].copy_(v, non_blocking=True)
            copied[i % 2].record(copy_stream)

    def compute(i):
        b = bufs[i % 2]
        stream.wait_event(copied[i % 2])
        q.cascade_attn(desc, b["q_suf"], b["k_anc"], b["v_anc"], b["k_suf"], b["v_suf"],
                       b["anchor_offsets"], b["anchor_suffix_ptr"], b["suffix_offsets"], out,
                       None, ws, k_scale, v_scale, stream=stream)
        q.restricted_head(b["h"], hx["gamma"], hx["w8"], logits, am, eps=1e-6, stream=stream)
        consumed[i % 2].record(stream)
        logits_h.copy_(logits, non_blocking=True)
        am_h.copy_(am, non_blocking=True)

    def run(n):
        copy_stream.wait_stream(stream)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)

    steps = max(3, min(args.steps, 10))
    run(2)
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    run(steps)
    b.record(stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(world, a.elapsed_time(b)) / steps
    del bufs, out
    torch.cuda.empty_cache()
    return {"value": sum_over_ranks(world, float(layout.total_suffix_tokens)) / (ms / 1e3),
            "unit": "suffix tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": ms, "steps": steps,
            "overlap": "inputs of step i + 1 copied on a second stream during step i"}


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


def run_bandwidth_kernel(args):
    """Per-kernel measurement of the HBM-bound kernels (not the headline step):
    --workload head      restricted head on 2,000,000 rows x 2,560 (bf16)
    --workload quantize  E4M3 quantisation of the long-anchor workload's anchor K
    Prints one JSON line with the kernel's CUDA-event time and its HBM roofline."""
    import prefill_only_cascade_gb300 as q
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    pk, src = peaks()
    if args.workload == "head":
        cfg = workloads.HEAD_CONFIGS["head"]
        n = args.head_rows or cfg.num_rows
        x = workloads.make_head_inputs(cfg, dev, num_rows=n)
        logits = torch.empty(n, 8, dtype=torch.float32, device=dev)
        am = torch.empty(n, dtype=torch.int32, device=dev)
        run = lambda: q.restricted_head(x["h"], x["gamma"], x["w8"], logits, am, eps=cfg.eps,
                                        stream=stream)
        algo_bytes = n * (cfg.hidden * 2 + 8 * 4 + 4) + cfg.hidden * 2 * 9
        units, unit = n, "rows/s"
        kernel = "restricted_head_kernel"
    else:
        cfg = workloads.ATTN_CONFIGS["fp8_long"]
        lay = workloads.make_layout(cfg)
        g = torch.Generator(device=dev).manual_seed(4)
        kv = workloads._randn_bf16((lay.total_anchor_tokens, cfg.num_kv_heads, cfg.head_dim), g, dev)
        codes = torch.empty(kv.shape, dtype=torch.uint8, device=dev)
        scale = torch.empty(cfg.num_anchors, cfg.num_kv_heads, dtype=torch.float32, device=dev)
        ao = torch.from_numpy(lay.anchor_offsets.copy()).to(dev)
        run = lambda: q.quantize_kv_fp8(kv, ao, codes, scale, stream=stream)
        algo_bytes = kv.numel() * 3 + scale.numel() * 4
        units, unit = kv.numel(), "elements/s"
        kernel = "kv_quantize_cluster_kernel"
    for _ in range(max(args.warmup, 3)):
        run()
    torch.cuda.synchronize()
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        time.sleep(0.3)
        for a, b in evs:
            flush.zero_()  # evict L2 (larger than L2) between timed launches
            a.record(stream)
            run()
            b.record(stream)
        torch.cuda.synchronize()
    ms = statistics.median(a.elapsed_time(b) for a, b in evs)
    gbs = algo_bytes / (ms / 1e3) / 1e9
    cpu = parity = None
    if not args.no_cpu_baseline:
        if args.workload == "head":
            cpu, parity = head_oracle_sample(x["h"], x["gamma"], x["w8"], cfg.eps, logits, am)
        else:
            cpu, parity = quantize_oracle_sample(kv, lay.anchor_offsets, codes, scale)
    line = {"metric": f"{args.workload} kernel throughput", "value": units / (ms / 1e3),
            "unit": unit, "n_gpus": 1, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": ms, "higher_is_better": True, "data": "synthetic",
            "config": {"workload": args.workload, "l2": "flushed between launches"},
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4), "traffic": None,
                         "peak_source": f"hbm_gbs of {src}", "kernel": kernel,
                         "algorithmic_bytes_per_launch": algo_bytes},
            "cpu_baseline": cpu, "parity": parity, "clocks": clk.summary()}
    print(json.dumps(line))


def run_prefill(args):
    """Per-kernel line for quail_causal_prefill_attn (the anchors' own causal prefill; not
    the headline): 64 sequences x 4,096 tokens, 32/8 heads, d = 128. Inputs larger than L2."""
    import prefill_only_cascade_gb300 as q
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    pk, src = peaks()
    cfg = workloads.ATTN_CONFIGS["prefill"]
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
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    with ClockSampler(0) as clk:
        time.sleep(0.3)
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
                         "traffic": traffic_from_profile("cascade.cu", "cascade_attn_prefill.md"),
                         "peak_source": f"bf16_tflops (burst) of {src}",
                         "kernel": "cascade_attn_kernel (anchors of length 0), one call",
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
    print(json.dumps(line))


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
