#!/usr/bin/env python3
"""Benchmark of the MoE-layer forward on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload mixtral]
                    [--impl ours|reference]

One step is one moe_forward (router -> dispatch -> expert grouped GEMMs ->
combine -> statistics) over the whole synthetic batch of the workload.  The
default workload is the Mixtral-8x7B-shaped layer (16384 tokens, d_model
4096, 8 experts, top-2, SwiGLU d_ff 14336, bf16, residual).  Inputs are
resident in HBM before the timed region; the 2.82 GB of expert weights and
the 134 MB activation exceed the 126 MB L2, so every step reads from HBM
without an explicit flush.

Prints one JSON line (rank 0).  With --gpus N > 1 (under torchrun) every rank
runs an independent replica of the workload (weak scaling, no collective on
the data path); the time is the maximum over ranks.

--routing expert_choice | hash runs the same layer under expert-choice
routing (every expert takes C = ceil(T/E * k) tokens, the compute of top-k)
or under hash routing of Zipf-distributed token ids; the default, top-k, is
the headline.

--train times a training step instead: the forward keeping its activations
plus moe_backward (aux_coef 0.01, z_coef 0.001), with the backward's stage
times and the TFLOP/s of its four GEMMs.

--impl reference times the plain CPU oracle on this machine's host cores on
a bounded sample of the same workload (full routing of every token plus the
experts of a sample of tokens, extrapolated to the whole batch).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_mixture_experts_60_b300 import workloads as wl  # noqa: E402

METRIC = "MoE-layer fwd tokens/s on 1 B300; expert GEMM TFLOP/s and % of bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
# nominal B300 figures (dense bf16 tensor rate, HBM3e bandwidth), reported
# next to the fractions of the measured peaks
SPEC_PEAKS = {"bf16_tflops": 2250.0, "hbm_gbs": 8000.0}
# a timed region shorter than this runs at the burst clocks: the tensor-core
# kernels inside it are compared with the burst bf16 figure, longer regions
# with the sustained one (measured under the power cap)
BURST_REGION_S = 1.0
GEMM_SRC = os.path.join(ROOT, "sparse_mixture_experts_60_b300", "csrc", "gemm_sm103.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
ACT_NAME = {wl.GELU: "gelu", wl.RELU: "relu", wl.SWIGLU: "swiglu"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def config_of(w, routing="topk", gemm_pair="auto"):
    extra = {} if gemm_pair == "auto" else {"gemm_kernel": "cta_pair" if gemm_pair == "1" else "one_cta"}
    return {**extra, "workload": w.name, "routing": routing, "tokens": w.T, "batch": w.batch, "seq": w.seq, "d_model": w.d,
            "experts": w.E, "top_k": w.k, "d_ff": w.F, "activation": ACT_NAME[w.activation],
            "score": "sigmoid" if w.score_fn == wl.SIGMOID else "softmax",
            "shared_experts": w.num_shared, "residual": bool(w.residual),
            "capacity": "dropping" if w.drop_tokens else "none",
            "l2": "no flush: expert weights (%.2f GB) and x (%.0f MB) exceed L2 and are read every step"
                  % (weight_bytes(w) / 1e9, w.T * w.d * w.elem_bytes / 1e6)}


def weight_bytes(w):
    mats = (3 if w.gated else 2) * w.E * w.F * w.d + w.E * w.d
    if w.num_shared:
        mats += (3 if w.gated else 2) * w.F * w.d
    return mats * w.elem_bytes


def gemm_flops(w, kept_rows):
    """Algorithmic FLOPs (2 per multiply-add) of the two expert GEMMs."""
    n1 = (2 if w.gated else 1) * w.F
    f1 = 2.0 * kept_rows * w.d * n1
    f2 = 2.0 * kept_rows * w.F * w.d
    if w.num_shared:
        f1 += 2.0 * w.T * w.d * n1
        f2 += 2.0 * w.T * w.F * w.d
    return f1, f2


def hbm_bytes(w, kept_rows, routing="topk"):
    """Algorithmic bytes of the HBM-bound stages (route, dispatch, combine):
    every tensor the stage must read or write, once, at its storage type
    (expert outputs y and the shared expert's z in the layer dtype)."""
    eb = w.elem_bytes
    T, d, E, S = w.T, w.d, w.E, w.T * w.k
    if routing == "hash":
        # hash routing: token ids in, expert ids and gates out
        route = T * 4 + S * 8
        permute = T * d * eb + kept_rows * d * eb + S * 4 * 3 + T * w.k * 4
        combine = kept_rows * d * eb + T * d * eb + (T * d * eb if w.residual else 0) + \
            (T * d * eb if w.num_shared else 0) + S * 8
        return route, permute, combine
    if routing == "expert_choice":
        R = kept_rows
        # logits GEMM (x, w_r in; logits out), selection (logits in; tok_row,
        # row_token out), gates (logits, tok_row in; tok_gate out)
        route = T * d * eb + E * d * eb + T * E * 4 + T * E * 4 + T * E * 4 + R * 4 + 3 * T * E * 4
        permute = 2 * R * d * eb + R * 4                       # row gather: read and write each chosen row
        combine = R * d * eb + T * d * eb + (T * d * eb if w.residual else 0) + \
            (T * d * eb if w.num_shared else 0) + T * E * 8
        return route, permute, combine
    route = T * d * eb + E * d * eb + T * E * 4 + S * 8 + T * 4
    permute = T * d * eb + kept_rows * d * eb + S * 4 * 3 + T * w.k * 4
    combine = kept_rows * d * eb + T * d * eb + (T * d * eb if w.residual else 0) + \
        (T * d * eb if w.num_shared else 0) + S * 8
    return route, permute, combine


def tensor_peak(pk, region_s):
    """The bf16 tensor peak a kernel inside a timed region of region_s
    seconds is compared with: burst below BURST_REGION_S, else sustained."""
    if region_s < BURST_REGION_S:
        return float(pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])), "bf16_tflops (burst)"
    return float(pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])), \
        "bf16_tflops_sustained"


def forward_roofline(w, kept_rows, active_experts, stage_ms, clocks, region_s, routing="topk"):
    """Roofline of the first routed expert GEMM, the expert GEMMs together,
    and the HBM-bound stages, from the mean stage times (ms: route, permute,
    ffn1, ffn2, shared, combine, stats).

    The first GEMM's algorithmic FLOPs are 2 kept_rows d nF; its algorithmic
    bytes are W1 (+ W3) of the experts that hold at least one kept row (an
    expert with no rows loads no weight tile), x_perm read once and H
    written once.  It is classed by whichever of the two takes longer at
    the measured peaks."""
    pk, pk_kind = peaks()
    peak, peak_name = tensor_peak(pk, region_s)
    hbm_peak = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    f1, f2 = gemm_flops(w, kept_rows)
    ffn1_ms, ffn2_ms = float(stage_ms[2]), float(stage_ms[3])
    n1 = (2 if w.gated else 1) * w.F
    f1r = 2.0 * kept_rows * w.d * n1
    b1r = float(active_experts * n1 * w.d * w.elem_bytes + kept_rows * w.d * w.elem_bytes +
                kept_rows * w.F * w.elem_bytes)
    kname = ("grouped_gemm_kernel (expert W1/W3 + SwiGLU)" if w.gated
             else "grouped_gemm_kernel (expert W1 + activation)")
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    clock_ratio = (smax / sm) if sm and smax else None
    if b1r / (hbm_peak * 1e9) > f1r / (peak * 1e12):
        gbs = b1r / (ffn1_ms * 1e-3) / 1e9
        roof = {"kernel": kname, "bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                "frac": gbs / hbm_peak, "peak_kind": f"hbm_gbs of {pk_kind}",
                "frac_of_spec": gbs / SPEC_PEAKS["hbm_gbs"], "spec_peak": SPEC_PEAKS["hbm_gbs"],
                "traffic": traffic_for_gemm(w, routing), "bytes_per_launch": b1r, "ms_per_launch": ffn1_ms,
                "active_experts": int(active_experts)}
    else:
        achieved = f1r / (ffn1_ms * 1e-3) / 1e12
        roof = {"kernel": kname, "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_kind": f"{peak_name} of {pk_kind}",
                "frac_of_sustained": achieved / float(pk.get("bf16_tflops_sustained",
                                                            FALLBACK_PEAKS["bf16_tflops_sustained"])),
                "frac_of_spec": achieved / SPEC_PEAKS["bf16_tflops"], "spec_peak": SPEC_PEAKS["bf16_tflops"],
                "frac_at_sm_max_clock": (achieved / peak / clock_ratio) if clock_ratio else None,
                "traffic": traffic_for_gemm(w, routing), "flops_per_launch": f1r, "ms_per_launch": ffn1_ms}
    gemm_ms = ffn1_ms + ffn2_ms + float(stage_ms[4])
    gemm_tf = (f1 + f2) / (gemm_ms * 1e-3) / 1e12
    expert_gemm = {"tflops": gemm_tf, "frac_of_peak": gemm_tf / peak, "peak_kind": peak_name,
                   "ffn1_tflops": f1r / (ffn1_ms * 1e-3) / 1e12,
                   "ffn2_tflops": 2.0 * kept_rows * w.F * w.d / (ffn2_ms * 1e-3) / 1e12,
                   "ms": gemm_ms, "kept_rows": int(kept_rows), "active_experts": int(active_experts)}
    expert_gemm["ffn1_frac"] = expert_gemm["ffn1_tflops"] / peak
    expert_gemm["ffn2_frac"] = expert_gemm["ffn2_tflops"] / peak
    rb, pb, cb = hbm_bytes(w, kept_rows, routing)
    hbm_ms = float(stage_ms[0] + stage_ms[1] + stage_ms[5])
    gbs = (rb + pb + cb) / (hbm_ms * 1e-3) / 1e9
    hbm = {"gbs": gbs, "peak_gbs": hbm_peak, "frac": gbs / hbm_peak, "frac_of_spec": gbs / SPEC_PEAKS["hbm_gbs"],
           "ms": hbm_ms, "bytes": rb + pb + cb}
    for name, b, i in (("route", rb, 0), ("permute", pb, 1), ("combine", cb, 5)):
        g = b / (float(stage_ms[i]) * 1e-3) / 1e9
        hbm[f"{name}_gbs"] = g
        hbm[f"{name}_frac"] = g / hbm_peak
    return roof, expert_gemm, hbm


def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time: every rank contributes its elapsed ms."""
    if dist is None:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Tokens per second over all ranks (weak scaling: every rank runs a replica)."""
    return tokens_per_rank * world / (ms_per_step * 1e-3)


def launches_per_step(w, routing="topk"):
    S = w.T * w.k
    if routing == "expert_choice":
        n = 1 + (1 if w.router_bias else 0)   # logits GEMM (+ bias)
        n += 3                                # selection, gates, row gather
        n += 2 + (2 if w.num_shared else 0)   # expert GEMMs (+ shared expert)
        return n + 1                          # combine
    if routing == "hash":
        n = 1                                 # hash routing
    else:
        n = 1 if w.E <= 32 else 2             # fused router (GEMM epilogue / CUDA-core kernel), else logits + routing
    nchunk = -(-S // 2048)                    # the two-launch dispatch's largest chunk
    if S == 0:
        n += 1
    elif S <= 2048 and w.E <= 256:
        n += 2                                # one-CTA dispatch, row copy
    elif nchunk * w.E <= 8192:
        n += 2                                # chunk ranks, row copy with the chunk bases
    else:
        n += 4                                # histogram, scan, rank, row copy
    n += 2 + (2 if w.num_shared else 0)       # expert GEMMs (+ shared expert)
    n += 2                                    # combine, statistics
    return n


def traffic_for_gemm(w, routing):
    """dram bytes per launch of the first expert GEMM from the committed ncu
    summary: only for the workload it was captured on, and only while the
    kernel source is unchanged."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as f:
        t = json.load(f)
    key = t.get("key", {})
    if key.get("workload") != w.name or key.get("tokens") != w.T or key.get("routing") != routing:
        return None
    sha = hashlib.sha256(open(GEMM_SRC, "rb").read()).hexdigest()
    if t.get("source_sha256") != sha:
        return None
    return t.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid):
        self.uuid = uuid
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", self.uuid], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons, pw = [], 0.0, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
                pw.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        busy = [s for s, p in zip(sm, pw) if p > 0.5 * max(pw)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw)}


def upload(inp, torch):
    out = {}
    for k, a in inp.items():
        if a.dtype == np.uint16:
            out[k] = torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return out


# ---------------------------------------------------------------------- CPU oracle
def oracle_sample(w, inp, budget_s, n_first=None):
    """Oracle time for the whole layer from a bounded sample: every token is
    routed and dispatched, the experts run for a sample of tokens, and the
    expert time is scaled to all tokens.  Returns (seconds for the layer,
    sample description, threads)."""
    from oracle import oracle as orc
    cores = orc.num_threads()
    t0 = time.perf_counter()
    lg = orc.router_logits(w, inp)
    r = orc.route(w, lg, inp.get("sel_bias"))
    dsp = orc.dispatch(w, r["idx"])
    orc.stats(w, dsp["counts"], dsp["kept"], r["prob_sum"], r["lse"])
    t_route = time.perf_counter() - t0
    n = n_first or max(1, cores)
    spent, done = 0.0, 0
    g = np.random.default_rng(7)
    while True:
        toks = np.sort(g.choice(w.T, size=min(n, w.T), replace=False))
        t1 = time.perf_counter()
        orc.forward_tokens(w, inp, r["idx"], r["gate"], dsp["inv"], toks)
        spent += time.perf_counter() - t1
        done += len(toks)
        if spent >= budget_s or done >= w.T:
            break
        per = spent / done
        n = int(max(1, min(w.T - done, (budget_s - spent) / per)))
    total = t_route + spent * w.T / done
    desc = (f"routing+dispatch of all {w.T} tokens ({t_route:.2f} s) + experts of {done} sampled tokens "
            f"({spent:.2f} s) scaled to {w.T}")
    return total, desc, cores


def run_reference(args, w, rank, world):
    if rank != 0:
        return 0
    inp = wl.make_inputs(w)
    per_step = max(1.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        oracle_sample(w, inp, per_step * 0.5)
    times, desc, cores = [], "", 1
    for _ in range(args.steps):
        t, desc, cores = oracle_sample(w, inp, per_step * 0.5)
        times.append(t)
    ms = 1e3 * statistics.mean(times)
    value = w.T / (ms / 1e3)          # one host process: the oracle is not replicated
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------- the other workloads
EXTRA = ("quickstart_bf16", "capacity_e128", "deepseek_v3", "tiny_fp32")


def device_expert_weights(w, torch, seed):
    """Expert weights of a workload drawn on the device (N(0, 0.02), the
    workload's distribution; biases N(0, 0.02)), one matrix at a time: the
    timing of the other workloads does not depend on the exact values, and
    the 22.6 GB of the DeepSeek-V3 experts would take a minute on the host."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    dt = torch.bfloat16 if w.dtype == wl.BF16 else torch.float32

    def stack(n, rows, cols):
        out = torch.empty(n, rows, cols, dtype=dt, device="cuda")
        for e in range(n):
            out[e].copy_(torch.randn(rows, cols, generator=g, device="cuda") * 0.02)
        return out

    wts = {"w1": stack(w.E, w.F, w.d), "w2": stack(w.E, w.d, w.F)}
    if w.gated:
        wts["w3"] = stack(w.E, w.F, w.d)
    if w.expert_bias:
        wts["b1"] = (torch.randn(w.E, w.F, generator=g, device="cuda") * 0.02).to(dt)
        wts["b2"] = (torch.randn(w.E, w.d, generator=g, device="cuda") * 0.02).to(dt)
    if w.num_shared:
        wts["shared_w1"] = stack(1, w.F, w.d)[0]
        wts["shared_w2"] = stack(1, w.d, w.F)[0]
        if w.gated:
            wts["shared_w3"] = stack(1, w.F, w.d)[0]
    return wts


def time_extra(name, steps, warmup, torch, moe):
    """Device-timed forward of another workload at its full size (the
    router inputs and x from the seeded generators, so its routing is the
    workload's; expert weights drawn on the device).  Returns the summary
    kept in the headline line's "workloads" key."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, with_weights=False) if w.name != "tiny_fp32" else wl.make_inputs(w)
    dev = upload(inp, torch)
    wts = {k: dev[k] for k in ("w_router", "b_router", "w1", "b1", "w3", "w2", "b2", "shared_w1", "shared_w3",
                               "shared_w2") if k in dev}
    if "w1" not in wts:
        wts.update(device_expert_weights(w, torch, 1000 + w.index))
    layer = moe.MoELayer(moe.config_for(w), wts, dev.get("sel_bias"))
    x = dev["x"]
    out = torch.empty(w.T, w.d, dtype=layer.out_dtype(), device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        layer.forward(x, out)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_STAGE_EVENTS)] for _ in range(steps)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(steps):
        layer.forward(x, out, stage_events=[e.cuda_event for e in evs[i]])
    t1.record(stream)
    torch.cuda.synchronize()
    if moe.moe_check_device_error():
        raise RuntimeError(f"device error flag after timing {name}")
    ms = t0.elapsed_time(t1) / steps
    stage_ms = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(7)] for i in range(steps)]).mean(0)
    res = {"tokens_per_s": w.T / (ms * 1e-3), "ms_per_step": ms, "steps": steps, "tokens": w.T,
           "dtype": "bf16" if w.dtype == wl.BF16 else "f32",
           "stage_ms": dict(zip(["route", "permute", "ffn1", "ffn2", "shared", "combine", "stats"],
                                stage_ms.tolist())),
           "weights": "router and x seeded as the workload; expert weights N(0, 0.02) drawn on the device"
                      if w.name != "tiny_fp32" else "all seeded as the workload"}
    if ms < 1.0:
        # a layer whose step is launch-bound, replayed from a CUDA graph
        # (MoELayer.graphed): one host launch per step instead of one per
        # kernel (the GEMM-bound layers gain nothing measurable)
        g = layer.graphed(x, out)
        for _ in range(2):
            g.replay()
        t0.record(stream)
        for _ in range(steps):
            g.replay()
        t1.record(stream)
        torch.cuda.synchronize()
        res["ms_per_step_graph"] = t0.elapsed_time(t1) / steps
        res["tokens_per_s_graph"] = w.T / (res["ms_per_step_graph"] * 1e-3)
        del g
        if moe.moe_check_device_error():
            raise RuntimeError(f"device error flag after the graph replays of {name}")
    if w.name == "tiny_fp32":
        res["latency_us"] = ms * 1e3
        res["latency_us_graph"] = res["ms_per_step_graph"] * 1e3
        res["note"] = "latency only: the layer (70 KB) stays in L2"
    else:
        kept = int(layer.stats()["total_kept"])
        active = int((layer.io["kept"] > 0).sum().item())
        roof, eg, hbm = forward_roofline(w, kept, active, stage_ms, {}, ms * steps * 1e-3)
        res["roofline"] = {k: roof[k] for k in ("kernel", "bound", "achieved", "peak", "unit", "frac",
                                                "frac_of_spec", "peak_kind")}
        res["expert_gemm"] = {k: eg[k] for k in ("tflops", "frac_of_peak", "ffn1_tflops", "ffn2_tflops",
                                                 "kept_rows", "active_experts")}
        res["hbm_stages"] = {k: hbm[k] for k in ("gbs", "frac", "route_frac", "permute_frac", "combine_frac")}
    del layer, wts, dev
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------- GPU path
def run_e2e(args, layer, x, out, ms, stream, barrier, dist, torch):
    """End to end through MoELayer.run_host_batches: two pinned input and
    output batches, used round-robin; every step uploads its whole x and
    downloads its whole output, overlapped with the neighbouring steps'
    compute.  Returns (ms per step, steps)."""
    x_hosts = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for _ in range(2)]
    for h in x_hosts:
        h.copy_(x)
    out_hosts = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    # enough steps that the pipeline's fill (the first upload) and drain
    # (the last download) weigh little against the steady state
    n_e2e = max(args.steps, min(50, max(3, int(2000.0 / max(ms, 1e-3)))))
    layer.run_host_batches(x_hosts, out_hosts, 3)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    layer.run_host_batches(x_hosts, out_hosts, n_e2e)
    e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / n_e2e, dist, "cuda")
    return e2e_ms, n_e2e


def run_ours(args, w, rank, world, local):
    import torch
    import sparse_mixture_experts_60_b300 as moe
    from sparse_mixture_experts_60_b300 import build as mbuild

    mbuild.build()
    torch.cuda.set_device(local)
    if args.gemm_pair != "auto":
        moe.moe_set_option(moe.MOE_OPT_GEMM_PAIR, int(args.gemm_pair))
    if args.gemm_band != -1:
        moe.moe_set_option(moe.MOE_OPT_GEMM_BAND, args.gemm_band)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    inp = wl.make_inputs(w)
    dev = upload(inp, torch)
    cfg = moe.config_for(w)
    wts = {k: dev[k] for k in ("w_router", "b_router", "w1", "b1", "w3", "w2", "b2", "shared_w1",
                               "shared_w3", "shared_w2") if k in dev}
    if args.routing == "expert_choice":
        layer = moe.ExpertChoiceLayer(cfg, wts)
        fwd = layer.forward
    elif args.routing == "hash":
        layer = moe.MoELayer(cfg, wts, dev.get("sel_bias"))
        token_ids = torch.from_numpy(wl.make_token_ids(w)).cuda()

        def fwd(xx, oo, stream=None, stage_events=None):
            return layer.forward_hashed(xx, token_ids, oo, stream, stage_events)
    else:
        layer = moe.MoELayer(cfg, wts, dev.get("sel_bias"))
        fwd = layer.forward
    x = dev["x"]
    out = torch.empty(w.T, w.d, dtype=layer.out_dtype(), device="cuda")
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    def new_events(n):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(moe.MOE_STAGE_EVENTS)] for _ in range(n)]
        for row in evs:
            for e in row:
                e.record(stream)      # creates the underlying cudaEvent_t
        torch.cuda.synchronize()
        return evs, [[e.cuda_event for e in row] for row in evs]

    for _ in range(max(3, args.warmup)):
        fwd(x, out)
    torch.cuda.synchronize()
    code = moe.moe_check_device_error()
    if code:
        raise RuntimeError(f"device error flag {code} after warm-up")

    uuid = str(torch.cuda.get_device_properties(local).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid

    def timed():
        evs, handles = new_events(args.steps)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier()
        with ClockSampler(uuid) as cs:
            t0.record(stream)
            for i in range(args.steps):
                if args.routing == "hash":
                    # the hash routing runs before moe_forward_from_routing:
                    # the route stage starts before it
                    evs[i][0].record(stream)
                    fwd(x, out, stage_events=[0] + list(handles[i][1:]))
                else:
                    fwd(x, out, stage_events=handles[i])
            t1.record(stream)
            barrier()
        return t0.elapsed_time(t1), evs, cs.summary()

    total_ms, evs, clocks = timed()
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(clocks["reasons"]):
        total_ms, evs, clocks = timed()          # re-measure once
        clocks["remeasured"] = True
    stage = np.array([[evs[i][j].elapsed_time(evs[i][j + 1]) for j in range(7)] for i in range(args.steps)])
    stage_ms = stage.mean(axis=0)               # route, permute, ffn1, ffn2, shared, combine, stats
    total_ms = max_over_ranks(total_ms, dist, "cuda")
    ms = total_ms / args.steps
    if args.routing == "expert_choice":
        stats = None
        kept = w.E * layer.capacity
        active = w.E if layer.capacity > 0 else 0
    else:
        stats = layer.stats()
        kept = int(stats["total_kept"])
        active = int((layer.io["kept"] > 0).sum().item())
    code = moe.moe_check_device_error()
    if code:
        raise RuntimeError(f"device error flag {code} after the timed region")

    # ----------------------------------------------------------- end to end from host buffers
    # (right after the timed region, before the other workloads heat the GPU)
    e2e_ms = None
    if not (args.no_e2e or args.routing == "hash"):
        e2e_ms = run_e2e(args, layer, x, out, ms, stream, barrier, dist, torch)
    # ----------------------------------------------------------- the other workloads (headline run only)
    extra = None
    if rank == 0 and args.extra_steps > 0 and w.name == "mixtral" and args.routing == "topk" and not args.train:
        extra = {}
        with ClockSampler(uuid) as cs:
            for name in EXTRA:
                extra[name] = time_extra(name, args.extra_steps, 3, torch, moe)
        extra["clocks"] = cs.summary()
    return finish(args, w, rank, world, dist, inp, x, out, ms, stage_ms, stats, kept, clocks, e2e_ms, active,
                  extra)


# ---------------------------------------------------------------------- training step
BWD_STAGES = ["gate_router", "dh_gemm", "dx_gemm", "shared", "dx_assemble", "dw2_gemm", "dw13_gemm",
              "bias_router_shared"]


def bwd_launches(w):
    """Kernels moe_backward launches (the order of its implementation)."""
    gated = w.activation == wl.SWIGLU
    wide = w.E >= 64 and w.E % 64 == 0
    n = 2 + (1 if wide else 0)                       # combine, router (+ dx router GEMM)
    n += 2                                           # dh, dx GEMMs (weights read in place)
    if w.num_shared:
        n += 2
    n += 1                                           # dx assembly
    n += 2 + (1 if gated else 0)                     # dW2, dW1 (+ dW3), activations read in place
    if w.expert_bias and not gated:
        n += 2                                       # db1, db2
    n += 8 if wide else 2                            # router weights (wide: offsets x2, 4 packs, GEMM, db)
    if w.num_shared:
        n += 1 + 2 + (1 if gated else 0)             # token range, shared dW2, dW1 (+ dW3)
    return n


def train_line(args, w, world, ms, fst, bst, kept, clocks):
    """The training step's JSON line from its timings: ms per step, the
    forward's 7 and the backward's 8 mean stage times (ms), the kept rows."""
    pk, pk_kind = peaks()
    peak, peak_name = tensor_peak(pk, ms * args.steps * 1e-3)
    nF = 2 * w.F if w.activation == wl.SWIGLU else w.F
    R = kept
    f1, f2 = gemm_flops(w, kept)                  # forward expert GEMMs
    flops = {"dh_gemm": 2.0 * R * w.d * w.F, "dx_gemm": 2.0 * R * nF * w.d, "dw2_gemm": 2.0 * R * w.d * w.F,
             "dw13_gemm": 2.0 * R * nF * w.d}
    bms = dict(zip(BWD_STAGES, bst.tolist()))
    gemm_tf = {k: flops[k] / (bms[k] * 1e-3) / 1e12 for k in flops}
    top = max(flops, key=lambda k: bms[k])
    # algorithmic HBM bytes of the weight-gradient GEMMs: the fp32 gradient
    # written once, each bf16 operand read once per launch (dW1 and dW3 are
    # two launches over x_perm); at large E and few rows per expert these
    # GEMMs are bound by the gradient writes, not by the tensor cores
    hbm_peak = float(pk.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    n13 = 2 if w.activation == wl.SWIGLU else 1
    wbytes = {"dw2_gemm": 4.0 * w.E * w.d * w.F + 2.0 * R * (w.d + w.F),
              "dw13_gemm": 4.0 * w.E * nF * w.d + 2.0 * R * (nF + n13 * w.d)}
    gemm_roof = {}
    for k in flops:
        t_tc = flops[k] / (peak * 1e12)
        t_hbm = wbytes.get(k, 0.0) / (hbm_peak * 1e9)
        ms_k = bms[k] * 1e-3
        gemm_roof[k] = ({"bound": "hbm", "frac": t_hbm / ms_k, "gbs": wbytes[k] / ms_k / 1e9} if t_hbm > t_tc
                        else {"bound": "tensor", "frac": t_tc / ms_k, "tflops": gemm_tf[k]})
    if gemm_roof[top]["bound"] == "hbm":
        roofline = {"kernel": f"grouped_gemm ({top}, backward)", "bound": "hbm", "achieved": gemm_roof[top]["gbs"],
                    "peak": hbm_peak, "unit": "GB/s", "frac": gemm_roof[top]["frac"],
                    "peak_kind": f"hbm_gbs of {pk_kind}", "traffic": None, "bytes_per_step": wbytes[top],
                    "ms_per_step": bms[top]}
    else:
        roofline = {"kernel": f"grouped_gemm ({top}, backward)", "bound": "tensor", "achieved": gemm_tf[top],
                    "peak": peak, "unit": "TFLOP/s", "frac": gemm_tf[top] / peak,
                    "peak_kind": f"{peak_name} of {pk_kind}", "traffic": None,
                    "frac_of_spec": gemm_tf[top] / SPEC_PEAKS["bf16_tflops"],
                    "flops_per_step": flops[top], "ms_per_step": bms[top]}
    train_flops = f1 + f2 + sum(flops.values())
    gemm_ms = float(fst[2] + fst[3]) + sum(bms[k] for k in flops)
    line = {
        "metric": "MoE-layer training step (forward + backward) tokens/s on 1 B300", "value":
        whole_job_value(w.T, world, ms), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic", "config": dict(config_of(w), mode="train", aux_coef=0.01, z_coef=0.001),
        "roofline": roofline,
        "expert_gemm": {"tflops": train_flops / (gemm_ms * 1e-3) / 1e12,
                        "frac_of_peak": train_flops / (gemm_ms * 1e-3) / 1e12 / peak, "peak_kind": peak_name,
                        "ms": gemm_ms,
                        "backward_gemm_tflops": gemm_tf, "backward_gemm_roofline": gemm_roof},
        "stage_ms": {"forward": dict(zip(["route", "permute", "ffn1", "ffn2", "shared", "combine", "stats"],
                                         fst.tolist())), "backward": bms},
        "clocks": clocks, "e2e": None,
        "gpu_launches": (launches_per_step(w) + bwd_launches(w)) * args.steps,
    }
    return line


def run_train(args, w, rank, world, local):
    """One step = the training forward (activations kept) + moe_backward
    with aux_coef 0.01, z_coef 0.001."""
    import torch
    import sparse_mixture_experts_60_b300 as moe
    from sparse_mixture_experts_60_b300 import build as mbuild

    mbuild.build()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    inp = wl.make_inputs(w)
    dev = upload(inp, torch)
    cfg = moe.config_for(w)
    wts = {k: dev[k] for k in ("w_router", "b_router", "w1", "b1", "w3", "w2", "b2", "shared_w1",
                               "shared_w3", "shared_w2") if k in dev}
    layer = moe.TrainingLayer(cfg, wts, dev.get("sel_bias"))
    x = dev["x"]
    out = torch.empty(w.T, w.d, dtype=layer.out_dtype(), device="cuda")
    g = torch.Generator(device="cuda").manual_seed(11)
    dout = torch.randn(w.T, w.d, device="cuda", generator=g).to(torch.bfloat16)
    grads = layer.new_grads()
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    def events(n, m):
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(m)] for _ in range(n)]
        for row in evs:
            for e in row:
                e.record(stream)
        torch.cuda.synchronize()
        return evs, [[e.cuda_event for e in row] for row in evs]

    for _ in range(max(3, args.warmup)):
        layer.forward(x, out)
        layer.backward(dout, 0.01, 0.001, grads)
    torch.cuda.synchronize()
    if moe.moe_check_device_error():
        raise RuntimeError("device error flag after warm-up")
    uuid = str(torch.cuda.get_device_properties(local).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid

    def timed():
        fe, fh = events(args.steps, moe.MOE_STAGE_EVENTS)
        be, bh = events(args.steps, moe.MOE_BWD_STAGE_EVENTS)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        barrier()
        with ClockSampler(uuid) as cs:
            t0.record(stream)
            for i in range(args.steps):
                layer.forward(x, out, stage_events=fh[i])
                layer.backward(dout, 0.01, 0.001, grads, stage_events=bh[i])
            t1.record(stream)
            barrier()
        return t0.elapsed_time(t1), fe, be, cs.summary()

    total_ms, fe, be, clocks = timed()
    if {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"} & set(clocks["reasons"]):
        total_ms, fe, be, clocks = timed()
        clocks["remeasured"] = True
    fst = np.array([[fe[i][j].elapsed_time(fe[i][j + 1]) for j in range(7)] for i in range(args.steps)]).mean(0)
    bst = np.array([[be[i][j].elapsed_time(be[i][j + 1]) for j in range(8)] for i in range(args.steps)]).mean(0)
    total_ms = max_over_ranks(total_ms, dist, "cuda")
    ms = total_ms / args.steps
    kept = int(layer.stats()["total_kept"])
    if moe.moe_check_device_error():
        raise RuntimeError("device error flag after the timed region")
    if rank != 0:
        dist.destroy_process_group()
        return 0
    line = train_line(args, w, world, ms, fst, bst, kept, clocks)
    print(json.dumps(line, default=float), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def finish(args, w, rank, world, dist, inp, x, out, ms, stage_ms, stats, kept, clocks, e2e_ms, active=None,
           extra=None):
    if rank != 0:
        dist.destroy_process_group()
        return 0
    active = w.E if active is None else active
    roofline, expert_gemm, hbm = forward_roofline(w, kept, active, stage_ms, clocks, ms * args.steps * 1e-3,
                                                  args.routing)
    line = {
        "metric": METRIC, "value": whole_job_value(w.T, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w.dtype == wl.BF16 else "f32",
        "data": "synthetic", "config": config_of(w, args.routing, getattr(args, "gemm_pair", "auto")),
        "roofline": roofline,
        "expert_gemm": expert_gemm,
        "hbm_stages": hbm,
        "stage_ms": {"route": stage_ms[0], "permute": stage_ms[1], "ffn1": stage_ms[2], "ffn2": stage_ms[3],
                     "shared": stage_ms[4], "combine": stage_ms[5], "stats": stage_ms[6]},
        "clocks": clocks,
        "e2e": None if e2e_ms is None else {
            "value": whole_job_value(w.T, world, e2e_ms[0]), "unit": "tokens/s",
            "h2d_bytes_per_step": int(x.numel() * x.element_size()),
            "d2h_bytes_per_step": int(out.numel() * out.element_size()), "ms_per_step": e2e_ms[0],
            "steps": e2e_ms[1]},
        "gpu_launches": launches_per_step(w, args.routing) * args.steps,
    }
    if extra:
        line["workloads"] = extra
    if world == 1 and not args.no_cpu_baseline and args.routing == "topk":
        t, desc, cores = oracle_sample(w, inp, args.cpu_seconds)
        line["cpu_baseline"] = {"value": w.T / t, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": desc}
    print(json.dumps(line, default=float), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_dense_reference(args, w):
    """The dense bf16 GEMMs of the same sizes as the workload's two expert
    GEMMs, by the vendor library (torch.matmul): kept rows x d x nF and kept
    rows x F x d with every row routed (T k rows), timed as a burst (10 calls)
    and in a loop of about a second under the power cap, with the clocks
    sampled.  A yardstick for the grouped expert GEMMs, not part of the
    layer."""
    import torch
    torch.cuda.set_device(0)
    uuid = str(torch.cuda.get_device_properties(0).uuid)
    uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    rows = w.T * w.k
    n1 = (2 if w.gated else 1) * w.F
    out = {"metric": "dense bf16 GEMM of the expert GEMM sizes (torch.matmul)", "impl": "dense_gemm_reference",
           "config": {"workload": w.name, "rows": rows, "d_model": w.d, "d_ff": w.F}, "gemms": {}}
    g = torch.Generator(device="cuda").manual_seed(11)
    for name, (M, K, N) in (("ffn1", (rows, w.d, n1)), ("ffn2", (rows, w.F, w.d))):
        a = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
        b = (torch.randn(K, N, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
        c = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
        for _ in range(3):
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        flops = 2.0 * M * N * K
        res = {"M": M, "K": K, "N": N}
        for label, n in (("burst", 10), ("loop", None)):
            if n is None:   # about one second of back-to-back calls
                n = max(10, int(1.0 / max(res["burst"]["ms"] * 1e-3, 1e-6)))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with ClockSampler(uuid) as cs:
                e0.record()
                for _ in range(n):
                    torch.matmul(a, b, out=c)
                e1.record()
                torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / n
            res[label] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "calls": n, "clocks": cs.summary()}
        out["gemms"][name] = res
        del a, b, c
        torch.cuda.empty_cache()
    print(json.dumps(out))
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=150)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="mixtral", choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--tokens", type=int, default=None,
                    help="override the token count (profiling of a smaller case; not a headline)")
    ap.add_argument("--experts", type=int, default=None,
                    help="override the routed expert count (profiling of another shape; not a headline)")
    ap.add_argument("--top-k", type=int, default=None,
                    help="override top_k (profiling of another shape; not a headline)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--gemm-pair", default="auto", choices=["auto", "0", "1"],
                    help="expert GEMM kernel: chosen by shape (auto), one-CTA (0) or CTA-pair (1) tiles")
    ap.add_argument("--gemm-band", type=int, default=-1,
                    help="expert GEMM raster band in M tiles: -1 chosen by shape, 0 whole experts, n > 0 n tiles")
    ap.add_argument("--extra-steps", type=int, default=20,
                    help="timed steps of each of the other workloads added to the headline (Mixtral) line; 0: none")
    ap.add_argument("--train", action="store_true",
                    help="time the training step (forward keeping activations + backward) instead")
    ap.add_argument("--routing", default="topk", choices=["topk", "expert_choice", "hash"],
                    help="token-choice top-k (the headline), expert-choice or hash routing")
    ap.add_argument("--dense-gemm-reference", action="store_true",
                    help="time the vendor library's dense bf16 GEMMs of the expert GEMM sizes instead")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus and world > 1:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    w = wl.WORKLOADS[args.workload]
    if args.tokens is not None:
        w = w.scaled(args.tokens)
    if args.experts is not None or args.top_k is not None:
        w = w.with_(E=args.experts or w.E, k=args.top_k or w.k, name=f"{w.name}_E{args.experts or w.E}"
                    f"_k{args.top_k or w.k}")
    if args.routing == "expert_choice":
        w = dataclasses.replace(w, capacity_factor=float(w.k))
    if args.dense_gemm_reference:
        return run_dense_reference(args, w)
    if args.impl == "reference":
        if args.routing != "topk":
            ap.error("--impl reference times the top-k layer only")
        return run_reference(args, w, rank, world)
    if args.train:
        if args.routing != "topk" or w.dtype != wl.BF16:
            ap.error("--train times the top-k layer of a bf16 workload")
        return run_train(args, w, rank, world, local)
    return run_ours(args, w, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
