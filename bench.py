#!/usr/bin/env python3
"""Benchmark of the MIS prefill hot path on one GB300 (or N replicas).

One step = the whole hot path over one batch of synthetic requests:
layout packing, mask-aware tile planning (host) and its upload (step i+1's
plan travels on a copy stream during step i, which ends only once it has
landed), MIS attention
(one layer's worth: Q/K/V -> O), delimiter-row gather, LM-head contraction
with fused full-vocabulary logsumexp, and the label read-out. The metric is
scored items per second; attention is also reported as useful (unmasked)
TFLOP/s against the measured dense BF16 peak.

  python bench.py [--gpus N --steps K --warmup W] [--workload NAME]
  python bench.py --impl reference      # the fp64 CPU oracle on the host cores
  python bench.py --sweep               # request-size sweep N = 1..200 vs eq. 5's R(N)

Prints one JSON line (rank 0). Under torchrun every rank runs its own copy of
the workload (requests are independent: no exchange), the timed region is
bracketed by a barrier and a device synchronisation, and the slowest rank's
time is reported.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MIS scored items/s; masked-attention useful TFLOP/s vs GB300 BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Evict L2 between timed steps: write a buffer larger than L2, then read a
    second one, so L2 holds only clean lines of neither input nor output (a
    write alone would leave dirty lines whose write-back the next step pays)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.fill_(1)
        self.r.sum()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_sha(name: str) -> str:
    with open(os.path.join(ROOT, "ranking_prefill_gb300", "csrc", name), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel_file: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it describes
    the current kernel source on this workload; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_file)
    if not e or e.get("source_sha") != kernel_source_sha(kernel_file) or e.get("workload") != workload:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while it runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1])); mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workload

def make_workload(name: str):
    from ranking_prefill_gb300 import lib, synth
    w = synth.WORKLOADS[name]
    shapes = synth.draw_shapes(w)
    size = lib.mis_setwise_layout_size if w.layout == "setwise" else lib.mis_layout_size
    T, M = size(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
    vals = synth.draw_values(w.seed, T, w.hq, w.hkv, w.head_dim, w.d_model, w.vocab)
    return w, shapes, vals, T, M


def oracle_sizes(w, shapes):
    """(T, M) of a workload from the oracle's own layout."""
    import oracle as O
    if w.layout == "setwise":
        sl = O.setwise_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
        return int(sl.causal.cu_seqlens[-1]), len(sl.marker_positions)
    lay = O.build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
    return int(lay.cu_seqlens[-1]), len(lay.delim_positions)


def make_workload_oracle(name: str):
    """make_workload for the reference arm: the sizes come from the oracle's
    own layout, so that arm runs without the CUDA library."""
    from ranking_prefill_gb300 import synth
    w = synth.WORKLOADS[name]
    shapes = synth.draw_shapes(w)
    T, M = oracle_sizes(w, shapes)
    vals = synth.draw_values(w.seed, T, w.hq, w.hkv, w.head_dim, w.d_model, w.vocab)
    return w, shapes, vals, T, M


class HostLayout:
    """The attention descriptor arrays and readout rows of one batch: MIS
    requests (items isolated, read at their trailing DELIMs) or setwise
    prompts (plain causal, read at their markers)."""

    def __init__(self, w, shapes, with_positions=False):
        from ranking_prefill_gb300 import lib
        if w.layout == "setwise":
            l = lib.mis_build_setwise_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens,
                                             with_positions=with_positions)
            self.item_ptr = self.item_offsets = None
            self.readout = l.marker_positions
        else:
            l = lib.mis_build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens,
                                     with_positions=with_positions)
            self.item_ptr, self.item_offsets = l.item_ptr, l.item_offsets
            self.readout = l.delim_positions
        self.cu_seqlens, self.prefix_len = l.cu_seqlens, l.prefix_len
        self.position_ids = l.position_ids
        self.T, self.M = l.T, len(self.readout)

    def plan_args(self):
        return self.cu_seqlens, self.prefix_len, self.item_ptr, self.item_offsets


def max_over_ranks(value: float, dist, device=None) -> float:
    """The slowest rank's value (all ranks get it); identity without a group."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def useful_flops(pairs: int, hq: int, D: int) -> float:
    return 4.0 * hq * D * pairs


L2_NOTE = "evicted between timed steps (256 MB write, then 256 MB read; untimed)"


def workload_config(w, shapes, T: int, M: int, K: int, world: int) -> dict:
    """The `config` object of the JSON line; both arms print the same one."""
    return {"workload": w.name, "requests": int(len(shapes.prefix_tokens)), "tokens": int(T),
            "items": int(M), "hq": w.hq, "hkv": w.hkv, "head_dim": w.head_dim,
            "d_model": w.d_model, "vocab": w.vocab, "labels": int(K), "l2": L2_NOTE,
            "parallelism": f"replicas x{world}"}


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, dist):
    import torch
    from ranking_prefill_gb300 import lib

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib.load()
    result = measure(args, args.workload, rank, world, dist, dev, local, full=True)
    # further workloads, timed the same way (throughput, per-call split and
    # roofline only; no end-to-end leg, comparators or CPU baseline)
    others = {}
    for name in [x for x in args.extra_workloads.split(",") if x not in ("", "none", args.workload)]:
        r = measure(args, name, rank, world, dist, dev, local, full=False)
        others[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "roofline", "attention",
                                          "scoring", "clocks")}
        others[name]["config"] = r["config"]
    if others:
        result["other_workloads"] = others
    return result


def measure(args, name, rank, world, dist, dev, local, full):
    """The timed steps of one workload; with `full`, also the end-to-end leg,
    the GPU comparators and the CPU oracle baseline."""
    import torch
    from ranking_prefill_gb300 import lib

    w, shapes, vals, T, M = make_workload(name)
    labels = [int(x) for x in shapes.label_sets[0]]
    K = len(labels)
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream

    # inputs resident in HBM
    q, k, v = (vals[n].to(dev) for n in ("q", "k", "v"))
    hidden, w_lm = vals["hidden"].to(dev), vals["w_lm"].to(dev)
    o = torch.empty_like(q)
    out = torch.empty(M, K, dtype=torch.float32, device=dev)
    lay0 = HostLayout(w, shapes)
    plan0 = lib.Plan(*lay0.plan_args(), w.hq, w.hkv, w.head_dim)
    # two plan workspaces, each followed by its batch's readout rows, uploaded
    # together: the plan of step i+1 travels on a copy stream while step i
    # computes, as in a serving loop (with --rope the position ids come from
    # the plan itself)
    wsz = plan0.workspace_size()
    n_extra = M
    ws_plans = [torch.zeros(wsz + 4 * n_extra, dtype=torch.uint8, device=dev) for _ in range(2)]
    delim_devs = [wp[wsz:wsz + 4 * M].view(torch.int32) for wp in ws_plans]
    kr = torch.empty_like(k) if args.rope else k
    ws_score = torch.zeros(lib.mis_label_scores_workspace_size(M, w.d_model, w.vocab, K),
                           dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    plan0.create(ws_plans[0], sp)
    stats = plan0.stats()
    plan0.destroy()
    planner = lib.Planner()
    copy_stream = torch.cuda.Stream(dev)
    uploaded = [torch.cuda.Event(), torch.cuda.Event()]
    used = [None, None]            # the step that last read each plan workspace
    plans = {}
    ev = lambda: torch.cuda.Event(enable_timing=True)

    host_s = []                    # host time of each step's layout + plan + upload call

    def enqueue_plan(i, after=None):
        """a1 + a2 of step i on the host (layout, plan), then one asynchronous
        upload of the plan and the readout rows into workspace i % 2 on the
        copy stream; `after`: an event of the step during which it travels."""
        h0 = time.perf_counter()
        s = i % 2
        lay = HostLayout(w, shapes)
        extra = lay.readout
        with torch.cuda.stream(copy_stream):
            if after is not None:
                copy_stream.wait_event(after)
            if used[s] is not None:
                copy_stream.wait_event(used[s])
            plans[i] = planner.plan(*lay.plan_args(), w.hq, w.hkv, w.head_dim, ws_plans[s],
                                    stream=copy_stream.cuda_stream, extra=extra)
            uploaded[s].record(copy_stream)
        host_s.append(time.perf_counter() - h0)

    def step(i, t):
        """Step i between the events t["st"] (recorded by the caller) and
        t["s1"]. Its plan arrived during step i-1; the plan of step i+1 is
        uploaded during this one, and the step ends only once that upload has
        landed, so every copy lies inside a timed step."""
        s = i % 2
        plan = plans.pop(i)
        stream.wait_event(uploaded[s])
        if "a0" in t:
            t["a0"].record(stream)
        # (with --rope) rotary embedding at the reused position ids, which
        # both kernels derive from the plan: K in its own pass, Q inside the
        # attention kernel as each tile loads
        if args.rope:
            lib.mis_rope_k_plan(plan, k, kr, 1.0e6, stream=sp)
            if "r1" in t:
                t["r1"].record(stream)
            # a3: MIS attention, Q rotated on load
            lib.mis_attention_fwd_plan_rope(plan, q, kr, v, o, None, 1.0e6, sp)
        else:
            # a3: MIS attention
            lib.mis_attention_fwd_plan(plan, q, kr, v, o, None, sp)
        if "a1" in t:
            t["a1"].record(stream)
        # a4-a6: gather + LM head + full-vocab LSE + label read-out
        lib.mis_label_scores(hidden, w_lm, delim_devs[s], labels, out, None, ws_score, stream=sp)
        done = torch.cuda.Event()
        done.record(stream)
        used[s] = done
        if "s1" in t and "a0" in t:
            t["s0"].record(stream)             # end of this step's kernels
        enqueue_plan(i + 1, after=t["st"])
        stream.wait_event(uploaded[(i + 1) % 2])
        t["s1"].record(stream)
        plan.destroy()

    with torch.cuda.stream(stream):
        n = 0
        enqueue_plan(0)
        for _ in range(args.warmup):
            flush()
            t = {"st": ev(), "s1": ev()}
            t["st"].record(stream)
            step(n, t)
            n += 1
        torch.cuda.synchronize()
        if any(lib.mis_get_device_status(wp, sp) for wp in ws_plans) or \
                lib.mis_get_device_status(ws_score, sp):
            raise RuntimeError("device status not ok after warm-up")

        recs, split_recs = [], []
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        with ClockSampler(local) as clk:
            # throughput: events around whole steps only. An event between two
            # calls would wait for the first call's kernels to finish, so the
            # next kernel's launch could no longer overlap their tail.
            for _ in range(args.steps):
                flush()                              # L2 eviction between timed steps (untimed)
                t = {"st": ev(), "s1": ev()}
                t["st"].record(stream)
                step(n, t)
                n += 1
                recs.append(t)
            torch.cuda.synchronize()
            if dist is not None:
                dist.barrier()
            # per-call split (attention, scoring, RoPE): as many steps again,
            # with events between the calls
            for _ in range(args.steps):
                flush()
                t = {"st": ev(), "a0": ev(), "r1": ev(), "a1": ev(), "s0": ev(), "s1": ev()}
                t["st"].record(stream)
                step(n, t)
                n += 1
                split_recs.append(t)
            torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
    for pl in plans.values():
        pl.destroy()
    step_ms = [r["st"].elapsed_time(r["s1"]) for r in recs]
    attn_ms = [r["r1" if args.rope else "a0"].elapsed_time(r["a1"]) for r in split_recs]
    rope_ms = [r["a0"].elapsed_time(r["r1"]) for r in split_recs] if args.rope else []
    score_ms = [r["a1"].elapsed_time(r["s0"]) for r in split_recs]
    split_ms = [r["st"].elapsed_time(r["s1"]) for r in split_recs]
    total_ms = float(sum(step_ms))
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    items_per_s = world * M * args.steps / (total_ms / 1e3)

    # correctness guard: the timed outputs are finite and the device status clean
    torch.cuda.synchronize()
    assert all(lib.mis_get_device_status(wp, sp) == 0 for wp in ws_plans)
    assert lib.mis_get_device_status(ws_score, sp) == 0
    assert bool(torch.isfinite(out).all())

    peaks, peak_src = load_peaks()
    t_attn = statistics.mean(attn_ms) / 1e3
    t_score = statistics.mean(score_ms) / 1e3
    pairs = stats["visible_pairs"]
    attn_flops = useful_flops(pairs, w.hq, w.head_dim)
    attn_tflops = attn_flops / t_attn / 1e12
    score_bytes = w.vocab * w.d_model * 2 + M * w.d_model * 2 + M * K * 4
    score_flops = 2.0 * M * w.d_model * w.vocab
    attn_bytes = T * (2 * w.hq + 2 * w.hkv) * w.head_dim * 2
    score_gbs = score_bytes / t_score / 1e9
    score_tflops = score_flops / t_score / 1e12

    # dominant kernel: the longer of the two, against its own bound
    if t_score >= t_attn:
        bound_hbm = score_bytes / (peaks["hbm_gbs"] * 1e9) >= score_flops / (peaks["bf16_tflops"] * 1e12)
        if bound_hbm:
            roof = {"kernel": "mis_label_scores (gather + tcgen05 LM head with fused LSE + combine)",
                    "bound": "hbm", "achieved": round(score_gbs, 1), "peak": peaks["hbm_gbs"],
                    "unit": "GB/s", "traffic": ncu_traffic("mis_score.cu", w.name),
                    "algorithmic_bytes_per_launch": score_bytes}
        else:
            roof = {"kernel": "mis_label_scores", "bound": "tensor", "achieved": round(score_tflops, 1),
                    "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "traffic": ncu_traffic("mis_score.cu", w.name),
                    "algorithmic_flops_per_launch": score_flops}
    else:
        roof = {"kernel": "mis_attention_fwd", "bound": "tensor", "achieved": round(attn_tflops, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "traffic": ncu_traffic("mis_attn.cu", w.name),
                "algorithmic_flops_per_launch": attn_flops}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["peak_source"] = peak_src

    result = {
        "metric": METRIC, "value": round(items_per_s, 1), "unit": "items/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the pages' workloads, random-init LM head)",
        "config": workload_config(w, shapes, T, M, K, world),
        "plan_upload": "host layout and plan every step; the upload of step i+1's plan and "
                       "readout rows overlaps step i, which ends only once it has landed",
        "roofline": roof,
        "attention": {"ms": round(t_attn * 1e3, 4), "useful_tflops": round(attn_tflops, 1),
                      "frac_of_bf16_peak": round(attn_tflops / peaks["bf16_tflops"], 4),
                      "visible_pairs": pairs, "tiles": stats["n_tiles"],
                      "causal_tiles": stats["n_causal_tiles"],
                      "hbm_gbs_qkvo": round(attn_bytes / t_attn / 1e9, 1)},
        "scoring": {"ms": round(t_score * 1e3, 4), "w_lm_stream_gbs": round(score_gbs, 1),
                    "tflops": round(score_tflops, 1)},
        "gpu_launches": (5 if args.rope else 4) * args.steps,
        "clocks": clk.summary(),
        "host_plan_ms": round(1e3 * statistics.median(host_s[-args.steps:]), 4),
        "host_plan_note": "host time of a step's layout + plan + upload call, including any "
                          "wait for a free pinned staging buffer while the GPU is behind",
        "per_call_split": {"steps": args.steps, "ms_per_step": round(statistics.mean(split_ms), 4),
                           "note": "attention, scoring and roofline times from as many further "
                                   "steps with CUDA events between the calls; value and "
                                   "ms_per_step from steps timed at their ends only"},
    }
    if args.rope:
        t_rope = statistics.mean(rope_ms) / 1e3
        rope_bytes = T * w.hkv * w.head_dim * 2 * 2
        result["rope"] = {"ms": round(t_rope * 1e3, 4), "bytes": rope_bytes,
                          "hbm_gbs": round(rope_bytes / t_rope / 1e9, 1),
                          "frac_of_hbm_peak": round(rope_bytes / t_rope / 1e9 / peaks["hbm_gbs"], 4),
                          "q": "rotated on load inside the attention kernel (ms above: the K pass)",
                          "note": "rotary embedding of Q and K at the reused position ids, "
                                  "inside the timed step before the attention"}
        result["config"]["rope"] = "base 1e6, rotate-half, reused position ids"
    if full and not args.no_e2e:
        result["e2e"] = run_e2e(args, w, shapes, vals, labels, dev, stream, dist, world)
    if full and not args.no_comparators:
        result["comparators"] = run_comparators(w, shapes, vals, labels, dev, stream, q, k, v,
                                                hidden, w_lm, t_attn, t_score, M, pairs)
    if full and rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, shapes, vals, labels, args.cpu_budget_s)
    del q, k, v, o, hidden, w_lm, ws_plans, ws_score, flush
    torch.cuda.empty_cache()
    return result


def run_e2e(args, w, shapes, vals, labels, dev, stream, dist, world):
    """Same metric through the C ABI from pinned host buffers: every step
    copies Q, K, V, hidden and the readout rows to the device and reads the
    label log-probs back. W_lm (a weight) stays resident. As in a serving
    loop, the inputs of step i+1 are copied on a second stream into the other
    of two device buffer sets while step i computes; every copy of every
    timed step is inside the timed region."""
    import torch
    from ranking_prefill_gb300 import lib
    sp = stream.cuda_stream
    # the step's inputs packed in one pinned block (one copy per step), each
    # at a 256-byte-aligned offset; the device buffer sets hold matching views
    names = ("q", "k", "v", "hidden")
    offs, total = {}, 0
    for n in names:
        offs[n] = total
        total += (vals[n].numel() * vals[n].element_size() + 255) // 256 * 256
    host_all = torch.empty(total, dtype=torch.uint8).pin_memory()

    def views(buf):
        return {n: buf[offs[n]:offs[n] + vals[n].numel() * vals[n].element_size()]
                .view(vals[n].dtype).view(vals[n].shape) for n in names}
    host = views(host_all)
    for n in names:
        host[n].copy_(vals[n])
    dev_all = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
    sets = [views(b) for b in dev_all]
    copy_stream = torch.cuda.Stream(dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    used = [None, None]          # step that last read each buffer set is done
    w_lm = vals["w_lm"].to(dev)
    T = host["q"].shape[0]
    lay = HostLayout(w, shapes)
    M, K = lay.M, len(labels)
    o = torch.empty_like(sets[0]["q"])
    out_dev = torch.empty(M, K, dtype=torch.float32, device=dev)
    out_host = torch.empty(M, K, dtype=torch.float32).pin_memory()
    planner = lib.Planner()
    plan0 = lib.Plan(*lay.plan_args(), w.hq, w.hkv, w.head_dim)
    wsz = plan0.workspace_size()
    # one plan workspace (plan + readout rows) per buffer set: the plan of step
    # i+1 is uploaded while step i may still read its own
    ws_plans = [torch.zeros(wsz + 4 * M, dtype=torch.uint8, device=dev) for _ in range(2)]
    delims = [wp[wsz:wsz + 4 * M].view(torch.int32) for wp in ws_plans]
    ws_score = torch.zeros(lib.mis_label_scores_workspace_size(M, w.d_model, w.vocab, K),
                           dtype=torch.uint8, device=dev)
    h2d = total + M * 4
    d2h = M * K * 4

    def step(i):
        s = i % 2
        dbuf = sets[s]
        l = HostLayout(w, shapes)
        # inputs, then the plan (with the readout rows), on the copy stream:
        # the copy engine serves them in that order, so this step's small plan
        # upload never queues behind the next step's inputs
        with torch.cuda.stream(copy_stream):
            if used[s] is not None:
                copy_stream.wait_event(used[s])
            dev_all[s].copy_(host_all, non_blocking=True)
            plan = planner.plan(*l.plan_args(), w.hq, w.hkv, w.head_dim, ws_plans[s],
                                stream=copy_stream.cuda_stream, extra=l.readout)
            copied[s].record(copy_stream)
        stream.wait_event(copied[s])
        lib.mis_attention_fwd_plan(plan, dbuf["q"], dbuf["k"], dbuf["v"], o, None, sp)
        lib.mis_label_scores(dbuf["hidden"], w_lm, delims[s], labels, out_dev, None, ws_score, stream=sp)
        ev = torch.cuda.Event()
        ev.record(stream)
        used[s] = ev
        out_host.copy_(out_dev, non_blocking=True)
        plan.destroy()

    steps = max(3, min(args.steps, 50))
    with torch.cuda.stream(stream):
        for i in range(3):
            step(i)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copy_stream.wait_stream(stream)               # the first copies start after `a`
        for i in range(steps):
            step(3 + i)
        b.record(stream)                              # after the last step's read-back
        torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    ms = max_over_ranks(ms, dist, dev)
    assert bool(torch.isfinite(out_host).all())
    for wsp in ws_plans + [ws_score]:
        assert lib.mis_get_device_status(wsp, sp) == 0
    return {"value": round(world * M * steps / (ms / 1e3), 1), "unit": "items/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": steps,
            "ms_per_step": round(ms / steps, 4),
            "overlap": "inputs of step i+1 copied on a second stream while step i computes"}


def _median_time(fn, stream, flush, reps=5):
    import torch
    ts = []
    for _ in range(reps + 2):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / 1e3)
    return statistics.median(ts[2:])


def run_comparators(w, shapes, vals, labels, dev, stream, q, k, v, hidden, w_lm, t_attn, t_score,
                    M, pairs):
    """Dense causal attention over the same cu_seqlens, and single-item scoring
    (every item as its own [prefix; item] sequence) on the GPU."""
    import torch
    from ranking_prefill_gb300 import lib
    sp = stream.cuda_stream
    flush = L2Flush(dev)
    if w.layout == "setwise":
        return {"mis_same_candidates": _mis_same_candidates(w, shapes, labels, dev, stream, w_lm,
                                                            t_attn, t_score, M, flush)}
    lay = lib.mis_build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
    res = {}
    with torch.cuda.stream(stream):
        # dense causal, same total length
        lens = np.diff(lay.cu_seqlens)
        cp = lib.Plan(lay.cu_seqlens, lens, None, None, w.hq, w.hkv, w.head_dim)
        ws = torch.zeros(cp.workspace_size(), dtype=torch.uint8, device=dev)
        cp.create(ws, sp)
        o = torch.empty_like(q)
        t_c = _median_time(lambda: lib.mis_attention_fwd_plan(cp, q, k, v, o, None, sp), stream, flush)
        cpairs = cp.stats()["visible_pairs"]
        res["dense_causal"] = {"ms": round(t_c * 1e3, 4),
                               "useful_tflops": round(useful_flops(cpairs, w.hq, w.head_dim) / t_c / 1e12, 1),
                               "mis_attention_speedup": round(t_c / t_attn, 2)}
        # single-item scoring: M sequences [Q_b; I_i], packed varlen, causal
        seqs, last = [], []
        for b in range(lay.B):
            s0, S = int(lay.cu_seqlens[b]), int(lay.prefix_len[b])
            for i in range(int(lay.item_ptr[b]), int(lay.item_ptr[b + 1])):
                a = int(lay.item_offsets[i])
                e = int(lay.item_offsets[i + 1]) if i + 1 < int(lay.item_ptr[b + 1]) else int(lay.cu_seqlens[b + 1])
                seqs.append(np.concatenate([np.arange(s0, s0 + S), np.arange(a, e)]))
        sis_tokens = int(sum(len(s) for s in seqs))
        budget = 3_000_000          # tokens per chunk (bounded device memory)
        t_sis, n_chunks, i0 = 0.0, 0, 0
        while i0 < len(seqs):
            i1, tok = i0, 0
            while i1 < len(seqs) and (tok + len(seqs[i1]) <= budget or i1 == i0):
                tok += len(seqs[i1]); i1 += 1
            idx = torch.as_tensor(np.concatenate(seqs[i0:i1]), device=dev, dtype=torch.long)
            qs, ks_, vs = q.index_select(0, idx), k.index_select(0, idx), v.index_select(0, idx)
            hs = hidden.index_select(0, idx)          # gathers are untimed
            sl = np.array([len(s) for s in seqs[i0:i1]])
            cu = np.concatenate([[0], np.cumsum(sl)]).astype(np.int32)
            sp_plan = lib.Plan(cu, sl, None, None, w.hq, w.hkv, w.head_dim)
            ws2 = torch.zeros(sp_plan.workspace_size(), dtype=torch.uint8, device=dev)
            sp_plan.create(ws2, sp)
            os_ = torch.empty_like(qs)
            rd = torch.as_tensor(cu[1:] - 1, device=dev, dtype=torch.int32)
            out = torch.empty(i1 - i0, len(labels), dtype=torch.float32, device=dev)
            wss = torch.zeros(lib.mis_label_scores_workspace_size(i1 - i0, w.d_model, w.vocab, len(labels)),
                              dtype=torch.uint8, device=dev)
            def run():
                lib.mis_attention_fwd_plan(sp_plan, qs, ks_, vs, os_, None, sp)
                lib.mis_label_scores(hs, w_lm, rd, labels, out, None, wss, stream=sp)
            t_sis += _median_time(run, stream, flush, reps=3)
            n_chunks += 1
            i0 = i1
            del qs, ks_, vs, hs, os_
        res["single_item_scoring_gpu"] = {
            "items_per_s": round(M / t_sis, 1), "ms": round(t_sis * 1e3, 4), "tokens": sis_tokens,
            "chunks": n_chunks, "note": "each item packed as its own causal [prefix; item] sequence, "
            "batched varlen through the same kernels; row gathers untimed",
            "mis_speedup_kernels_only": round(t_sis / (t_attn + t_score), 2)}
        res["prefix_cache"] = _prefix_cache(w, lay, labels, dev, stream, flush, q, k, v, hidden,
                                            w_lm, t_attn, t_score, M)
    return res


def _prefix_cache(w, lay, labels, dev, stream, flush, q, k, v, hidden, w_lm, t_attn, t_score, M):
    """The same requests with their prefixes in a K/V cache (the in-batch
    prefix cache of "Scaling LLM-Based Ranking Systems with Prefill-Only
    Optimization", Components table, and the knock-knock second request of
    "Turbocharging LinkedIn's recommendation systems with SGLang"). Times the prefix prefill
    (causal attention over each prefix: the first request, which fills the
    cache), the item request (MIS among the items over the cached prefix,
    then scoring) and single-item scoring with the prefix cache (one request
    per item over the same cached rows). Row gathers are untimed."""
    import torch
    from ranking_prefill_gb300 import lib
    sp = stream.cuda_stream
    B = lay.B
    S = lay.prefix_len.astype(np.int64)
    cu = lay.cu_seqlens.astype(np.int64)
    cum_s = np.concatenate([[0], np.cumsum(S)])
    pre_rows = np.concatenate([np.arange(cu[b], cu[b] + S[b]) for b in range(B)])
    item_rows = np.concatenate([np.arange(cu[b] + S[b], cu[b + 1]) for b in range(B)])
    ip = lay.item_ptr.astype(np.int64)
    req_of_item = np.repeat(np.arange(B), np.diff(ip))
    # the item sequence: each request's item sets without its prefix
    cu_i = (cu - cum_s).astype(np.int32)
    io_i = (lay.item_offsets - cum_s[req_of_item + 1]).astype(np.int32)
    rd_i = (lay.delim_positions - cum_s[req_of_item + 1]).astype(np.int32)
    take = lambda t, rows: t.index_select(0, torch.as_tensor(rows, device=dev, dtype=torch.long))
    kc, vc, qp = take(k, pre_rows), take(v, pre_rows), take(q, pre_rows)
    qi, ki, vi, hi = take(q, item_rows), take(k, item_rows), take(v, item_rows), take(hidden, item_rows)
    cache_T = int(cum_s[-1])
    out = torch.empty(M, len(labels), dtype=torch.float32, device=dev)
    res = {}
    with torch.cuda.stream(stream):
        # first request: causal prefill of the prefixes (fills the cache)
        cpl = lib.Plan(cum_s.astype(np.int32), S.astype(np.int32), None, None, w.hq, w.hkv, w.head_dim)
        wsp = torch.zeros(cpl.workspace_size(), dtype=torch.uint8, device=dev)
        cpl.create(wsp, sp)
        op = torch.empty_like(qp)
        t_pre = _median_time(lambda: lib.mis_attention_fwd_plan(cpl, qp, kc, vc, op, None, sp), stream, flush)
        # second request: the items over the cached prefix, then scoring
        rd = torch.as_tensor(rd_i, device=dev)
        wss = torch.zeros(lib.mis_label_scores_workspace_size(M, w.d_model, w.vocab, len(labels)),
                          dtype=torch.uint8, device=dev)
        t_sc = _median_time(lambda: lib.mis_label_scores(hi, w_lm, rd, labels, out, None, wss, stream=sp),
                            stream, flush)
        oi = torch.empty_like(qi)

        def cached_time(cu_, ip_, io_, cs_, cl_):
            pl = lib.CachedPlan(cu_, ip_, io_, cs_, cl_, cache_T, w.hq, w.hkv, w.head_dim)
            wsc = torch.zeros(pl.workspace_size(), dtype=torch.uint8, device=dev)
            pl.create(wsc, sp)
            t = _median_time(lambda: lib.mis_attention_fwd_cached(pl, qi, ki, vi, kc, vc, oi, None, sp),
                             stream, flush)
            torch.cuda.synchronize()
            assert lib.mis_get_device_status(wsc, sp) == 0
            return t, pl.stats()
        t_mis, st_mis = cached_time(cu_i, lay.item_ptr, io_i, cum_s[:-1].astype(np.int32), S.astype(np.int32))
        # single-item scoring with the prefix cache: one request per item
        ends_i = np.concatenate([io_i[1:], [cu_i[-1]]]).astype(np.int64)
        ends_i[ip[1:][np.diff(ip) > 0] - 1] = cu_i[1:][np.diff(ip) > 0]
        cu_s = np.concatenate([[0], np.cumsum(ends_i - io_i)]).astype(np.int32)
        t_sis, _ = cached_time(cu_s, np.arange(M + 1, dtype=np.int32), cu_s[:-1],
                               cum_s[req_of_item].astype(np.int32), S[req_of_item].astype(np.int32))
    res = {"prefix_prefill_ms": round(t_pre * 1e3, 4),
           "item_request": {"attention_ms": round(t_mis * 1e3, 4), "scoring_ms": round(t_sc * 1e3, 4),
                            "items_per_s": round(M / (t_mis + t_sc), 1),
                            "useful_tflops": round(useful_flops(st_mis["visible_pairs"], w.hq, w.head_dim)
                                                   / t_mis / 1e12, 1),
                            "vs_full_mis_step": round((t_attn + t_score) / (t_mis + t_sc), 3)},
           "single_item_scoring_with_prefix_cache": {
               "attention_ms": round(t_sis * 1e3, 4), "items_per_s": round(M / (t_sis + t_sc), 1),
               "mis_item_request_speedup": round((t_sis + t_sc) / (t_mis + t_sc), 3)},
           "knock_knock_total_ms": round((t_pre + t_mis + t_sc) * 1e3, 4),
           "note": "prefix K/V gathered into a cache; item rows as their own sequence; gathers untimed"}
    return res


def _mis_same_candidates(w, shapes, labels, dev, stream, w_lm, t_attn, t_score, M, flush):
    """The same requests as MIS (items isolated, read at their DELIMs) through
    the same kernels, against the setwise run (one causal sequence per
    request, read at its markers). Inputs N(0, 1) drawn on the device."""
    import torch
    from ranking_prefill_gb300 import lib
    sp = stream.cuda_stream
    lay = lib.mis_build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens,
                               with_positions=False)
    g = torch.Generator(device=dev).manual_seed(w.seed)
    rnd = lambda *shape: torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
    q, k, v = rnd(lay.T, w.hq, w.head_dim), rnd(lay.T, w.hkv, w.head_dim), rnd(lay.T, w.hkv, w.head_dim)
    hidden = rnd(lay.T, w.d_model)
    plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, w.hq, w.hkv,
                    w.head_dim)
    ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    delim = torch.as_tensor(lay.delim_positions, device=dev)
    out = torch.empty(lay.M, len(labels), dtype=torch.float32, device=dev)
    wss = torch.zeros(lib.mis_label_scores_workspace_size(lay.M, w.d_model, w.vocab, len(labels)),
                      dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        plan.create(ws, sp)
        ta = _median_time(lambda: lib.mis_attention_fwd_plan(plan, q, k, v, o, None, sp), stream, flush)
        ts = _median_time(lambda: lib.mis_label_scores(hidden, w_lm, delim, labels, out, None, wss,
                                                       stream=sp), stream, flush)
    return {"items_per_s": round(lay.M / (ta + ts), 1), "attention_ms": round(ta * 1e3, 4),
            "scoring_ms": round(ts * 1e3, 4), "tokens": lay.T,
            "setwise_vs_mis_kernel_time": round((t_attn + t_score) / (ta + ts), 3),
            "note": "same candidate lengths packed as MIS requests; MIS isolates items, setwise "
                    "markers see every candidate"}


# ------------------------------------------------------- request-size sweep

def run_sweep(args):
    """Request-size sweep ("From Generation to Scoring", Section 6.4, RQ3): the
    same members and candidates scored as requests of N items for N = 1..200.
    Each request re-prefills its member's query. Reports per N the kernel time
    per label (attention + scoring, L2 evicted between repetitions), the
    speedup over N = 1, and eq. 5's prefill-token ratio R(N) computed from the
    raw token counts (delimiters omitted, as in eq. 5)."""
    import torch
    from ranking_prefill_gb300 import lib, synth
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS["qwen3-0.6b-layer"]           # heads, head dim, model and vocabulary sizes
    pool = synth.sweep_pool(args.sweep_members, w.vocab)
    labels = [int(x) for x in pool.labels]
    stream = torch.cuda.Stream(dev)
    sp = stream.cuda_stream
    flush = L2Flush(dev)
    g = torch.Generator(device=dev).manual_seed(6)
    w_lm = (torch.randn(w.vocab, w.d_model, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    rows = []
    for n in synth.SWEEP_N:
        shapes = synth.sweep_shapes(pool, n)
        lay = lib.mis_build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens,
                                   with_positions=False)
        T, M = lay.T, lay.M
        rnd = lambda *shape: torch.randn(*shape, generator=g, device=dev).to(torch.bfloat16)
        q, k, v = rnd(T, w.hq, w.head_dim), rnd(T, w.hkv, w.head_dim), rnd(T, w.hkv, w.head_dim)
        hidden = rnd(T, w.d_model)
        o = torch.empty_like(q)
        plan = lib.Plan(lay.cu_seqlens, lay.prefix_len, lay.item_ptr, lay.item_offsets, w.hq,
                        w.hkv, w.head_dim)
        ws = torch.zeros(plan.workspace_size(), dtype=torch.uint8, device=dev)
        delim = torch.as_tensor(lay.delim_positions, device=dev)
        out = torch.empty(M, len(labels), dtype=torch.float32, device=dev)
        wss = torch.zeros(lib.mis_label_scores_workspace_size(M, w.d_model, w.vocab, len(labels)),
                          dtype=torch.uint8, device=dev)
        with torch.cuda.stream(stream):
            plan.create(ws, sp)
            ta = _median_time(lambda: lib.mis_attention_fwd_plan(plan, q, k, v, o, None, sp),
                              stream, flush, reps=5)
            ts = _median_time(lambda: lib.mis_label_scores(hidden, w_lm, delim, labels, out, None,
                                                           wss, stream=sp), stream, flush, reps=5)
        torch.cuda.synchronize()
        assert lib.mis_get_device_status(ws) == 0 and lib.mis_get_device_status(wss) == 0
        raw = int(shapes.prefix_tokens.sum()) + int(shapes.item_lens.sum())
        rows.append({"N": n, "requests": int(len(shapes.prefix_tokens)), "tokens": T,
                     "raw_tokens": raw, "pairs": plan.stats()["visible_pairs"],
                     "attention_ms": round(ta * 1e3, 4), "scoring_ms": round(ts * 1e3, 4),
                     "labels_per_s": round(M / (ta + ts), 1)})
        del q, k, v, hidden, o, ws, out, wss, plan
        torch.cuda.empty_cache()
    b = rows[0]
    for r in rows:
        r["speedup_vs_n1"] = round(r["labels_per_s"] / b["labels_per_s"], 3)
        r["attention_speedup_vs_n1"] = round(b["attention_ms"] / r["attention_ms"], 3)
        r["R_eq5"] = round(b["raw_tokens"] / r["raw_tokens"], 3)
        r["pairs_ratio_vs_n1"] = round(b["pairs"] / r["pairs"], 3)
    return {"sweep": "request size", "members": args.sweep_members,
            "candidates_per_member": synth.SWEEP_CANDIDATES, "labels": M,
            "model": {"hq": w.hq, "hkv": w.hkv, "head_dim": w.head_dim, "d_model": w.d_model,
                      "vocab": w.vocab},
            "query_tokens": [int(x) for x in pool.query_tokens], "rows": rows}


# ---------------------------------------------------------------- CPU oracle

def _as_f64(vals):
    """The oracle's inputs as float64 arrays (converted once per run)."""
    import torch
    return {n: (t.to(torch.float64).numpy() if isinstance(t, torch.Tensor) else t)
            for n, t in vals.items() if n in ("q", "k", "v", "hidden", "w_lm")}


def _oracle_sample(w, shapes, vals, labels, budget_s, seed=0, rates=None):
    """Time the oracle on a seeded sample of rows and items sized from a small
    timed pilot, so the whole run stays near `budget_s`; returns an estimate
    of the full workload's oracle time and the sample description."""
    import oracle as O
    import torch
    if w.layout == "setwise":
        sl = O.setwise_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
        lay, readout = sl.causal, sl.marker_positions
    else:
        lay = O.build_layout(shapes.prefix_tokens, shapes.n_items, shapes.item_lens)
        readout = lay.delim_positions
    n_read = len(readout)
    t_call = time.perf_counter()
    x = _as_f64(vals)
    q, k, v, hidden, W = x["q"], x["k"], x["v"], x["hidden"], x["w_lm"]
    rng = np.random.default_rng(seed)

    def timed(fn):
        t0 = time.perf_counter()
        fn()
        return time.perf_counter() - t0

    # attention: cost per row from a 32-row pilot, then as many rows as fit
    # (`rates`, when given, carries the measured per-row cost from one call
    # to the next, so repeated samples skip the pilot)
    if rates is not None and "per_row" in rates:
        per_row = rates["per_row"]
    else:
        pilot = np.sort(rng.choice(lay.T, size=min(32, lay.T), replace=False))
        per_row = timed(lambda: O.attention(q, k, v, lay, rows=pilot)) / len(pilot)
    n_rows = int(min(lay.T, max(min(32, lay.T), 0.7 * budget_s / max(per_row, 1e-9))))
    rows = None if n_rows >= lay.T else np.sort(rng.choice(lay.T, size=n_rows, replace=False))
    t_attn = timed(lambda: O.attention(q, k, v, lay, rows=rows))
    frac_r = 1.0 if rows is None else n_rows / lay.T
    if rates is not None:
        rates["per_row"] = t_attn / n_rows
    # scoring: the oracle makes one W_lm pass per block of 64 items, so the
    # pilot is one full block (all items when fewer), which amortises that
    # pass as the full run does; more items only when the budget allows
    base = min(n_read, 64)
    pilot_i = np.sort(rng.choice(n_read, size=base, replace=False))
    t_pilot = timed(lambda: O.label_scores(hidden, W, readout, labels, items=pilot_i))
    per_item = t_pilot / base
    n_items = int(min(n_read, max(base, 0.3 * budget_s / max(per_item, 1e-9))))
    if n_items == base:
        items, t_score = (None if base == n_read else pilot_i), t_pilot
    else:
        items = None if n_items >= n_read else np.sort(rng.choice(n_read, size=n_items, replace=False))
        t_score = timed(lambda: O.label_scores(hidden, W, readout, labels, items=items))
    frac_i = 1.0 if items is None else n_items / n_read
    t_full = t_attn / frac_r + t_score / frac_i
    if rows is None and items is None:
        sample = f"oracle on the whole workload ({lay.T} rows x {w.hq} heads, {n_read} items)"
    else:
        sample = (f"oracle on {'all' if rows is None else n_rows} of {lay.T} rows x {w.hq} heads and "
                  f"{'all' if items is None else n_items} of {n_read} items; full-workload time "
                  f"extrapolated by rows and items")
    # wall time of this call: the pilots and the timed parts
    return t_full, n_read, sample, time.perf_counter() - t_call


def cpu_baseline(w, shapes, vals, labels, budget_s):
    t_full, M, sample, spent = _oracle_sample(w, shapes, vals, labels, budget_s)
    return {"value": round(M / t_full, 3), "unit": "items/s", "cores": os.cpu_count(),
            "kind": "oracle", "sample": sample, "seconds": round(spent, 2)}


def run_reference(args, rank, world):
    """The fp64 CPU oracle as the reference arm. Each step runs the oracle on
    the whole workload when that fits the step's budget (at least 2 s, more
    when --cpu-budget-s spread over the steps allows), else on a seeded
    sample of rows and items; `value` is the whole workload's items over its
    full oracle time (measured, or extrapolated from the sample by rows and
    items), `ms_per_step` the wall time each executed step actually took."""
    if rank != 0:
        return None
    w, shapes, vals, T, M = make_workload_oracle(args.workload)
    labels = [int(x) for x in shapes.label_sets[0]]
    budget = max(2.0, args.cpu_budget_s / max(1, args.steps + args.warmup))
    vals = _as_f64(vals)
    rates = {}
    for _ in range(args.warmup):
        _oracle_sample(w, shapes, vals, labels, budget, rates=rates)
    tot_est, spent, sample = 0.0, 0.0, ""
    for s in range(args.steps):
        t_full, M, sample, sp = _oracle_sample(w, shapes, vals, labels, budget, seed=s, rates=rates)
        tot_est += t_full
        spent += sp
    v = M * args.steps / tot_est
    return {"metric": METRIC, "value": round(v, 3), "unit": "items/s", "impl": "reference",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * spent / args.steps, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, shapes, T, M, len(labels), world),
            "cpu_baseline": {"value": round(v, 3), "unit": "items/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample,
                             "full_workload_s_estimate": round(tot_est / args.steps, 3),
                             "note": "ms_per_step: wall time of each executed step; value: the "
                                     "workload's items over its full oracle time"},
            "e2e": {"value": round(v, 3), "unit": "items/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="varlen-16",
                    help="the headline workload (default: varlen-16, the largest configuration "
                         "that fits one GPU)")
    ap.add_argument("--extra-workloads", default="qwen3-0.6b-layer",
                    help="comma-separated workloads also timed (throughput and roofline only); "
                         "'none' for none")
    ap.add_argument("--sweep", action="store_true",
                    help="request-size sweep N = 1..200 (prints its own JSON table)")
    ap.add_argument("--sweep-members", type=int, default=16)
    ap.add_argument("--rope", action="store_true",
                    help="rotate Q and K at the reused position ids inside the timed step")
    ap.add_argument("--cpu-budget-s", type=float, default=20.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-comparators", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.rope:
        args.no_e2e = True        # the end-to-end leg times the default path only
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    dist = None
    if world > 1 and args.impl == "ours":
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        tdist.init_process_group("nccl")
        dist = tdist
    if args.sweep:
        res = run_sweep(args) if rank == 0 else None
    elif args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, dist)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
