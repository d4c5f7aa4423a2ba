"""The benchmark's JSON lines built on CPU from stage times measured on a
B300, checking the contract keys and the roofline classification.  The
first routed expert GEMM of the Mixtral shape is tensor-bound.  Those of
the DeepSeek-V3 and E = 128 capacity shapes are bound by streaming their
weights from HBM.  The DeepSeek-V3 weight-gradient GEMMs are bound by
their fp32 gradient writes."""
import argparse
import json
import os
import sys

import numpy as np
import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from sparse_mixture_experts_60_b300 import workloads as wl  # noqa: E402

CLOCKS = {"sm_mhz": 1275.0, "sm_max_mhz": 2032.0, "reasons": ["sw_power_cap"], "samples": 10}
PEAKS = {"hbm_gbs": 6486.5, "bf16_tflops": 1805.2, "bf16_tflops_sustained": 1405.8}


@pytest.fixture(autouse=True)
def fixed_peaks(monkeypatch):
    """The lines are checked against fixed peaks, not this machine's file."""
    monkeypatch.setattr(bench, "peaks", lambda: (dict(PEAKS), "measured"))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "e2e", "gpu_launches"}

# measured on one B300 (ms): route, permute, ffn1, ffn2, shared, combine, stats; kept rows; experts
# holding kept rows; bound of the first expert GEMM
FORWARD = {
    "mixtral": (9.3748, [0.04629, 0.09512, 5.88898, 3.16829, 0.00143, 0.15551, 0.01289], 32768, 8, "tensor"),
    "deepseek_v3": (4.8929, [0.15674, 0.14200, 2.53212, 1.45942, 0.36588, 0.20369, 0.02652], 32768, 256, "hbm"),
    "capacity_e128": (0.38982, [0.03563, 0.01909, 0.14534, 0.14765, 0.00156, 0.02042, 0.01446], 2879, 61, "hbm"),
}


def expected_frac(w, ms_ffn1, kept, active, steps, ms_step):
    """First routed expert GEMM: FLOPs 2 kept d nF against the burst (timed
    region under 1 s) or sustained bf16 peak, or bytes (W1 (+ W3) of the
    experts with kept rows, x_perm read, H written) against the copy peak."""
    nF = 2 * w.F if w.gated else w.F
    flops = 2.0 * kept * w.d * nF
    nbytes = (active * nF * w.d + kept * w.d + kept * w.F) * w.elem_bytes
    tpk = PEAKS["bf16_tflops"] if steps * ms_step < 1000.0 else PEAKS["bf16_tflops_sustained"]
    t_tc, t_hbm = flops / (tpk * 1e12), nbytes / (PEAKS["hbm_gbs"] * 1e9)
    return max(t_tc, t_hbm) / (ms_ffn1 * 1e-3), "tensor" if t_tc >= t_hbm else "hbm"
# forward stages as above; backward: gate_router, dh, dx, shared, dx_assemble, dW2, dW1|dW3, bias/router/shared
TRAIN = {
    "mixtral": (29.966, [0.04647, 0.09398, 6.02053, 3.14277, 0.00140, 0.15314, 0.01104],
                [0.18328, 3.36744, 5.82591, 0.00199, 0.33901, 3.53388, 7.02107, 0.19902], "tensor",
                2.0 * 32768 * 28672 * 4096 / 7.02107e-3 / 1e12 / PEAKS["bf16_tflops"]),
    "deepseek_v3": (20.036, [0.12149, 0.12313, 2.30103, 1.28188, 0.31187, 0.19892, 0.02132],
                    [0.34430, 1.18386, 2.33069, 0.31982, 0.22989, 3.57827, 7.15927, 0.50534], "hbm",
                    (4.0 * 256 * 4096 * 7168 + 2.0 * 32768 * (4096 + 2 * 7168)) / 7.15927e-3 / 1e9
                    / PEAKS["hbm_gbs"]),
}


def _args(steps=150, warmup=5, routing="topk"):
    return argparse.Namespace(steps=steps, warmup=warmup, routing=routing, no_cpu_baseline=True, cpu_seconds=1.0)


@pytest.mark.parametrize("steps", [20, 150])
@pytest.mark.parametrize("name", list(FORWARD))
def test_forward_line(name, steps, capsys):
    ms, stages, kept, active, bound = FORWARD[name]
    w = wl.WORKLOADS[name]
    frac, bound2 = expected_frac(w, stages[2], kept, active, steps, ms)
    assert bound2 == bound
    x = torch.empty(w.T, w.d, dtype=torch.bfloat16)
    bench.finish(_args(steps=steps), w, 0, 1, None, None, x, x, ms, stages, None, kept, CLOCKS, (ms * 1.01, 50),
                 active)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert KEYS <= set(line)
    assert line["n_gpus"] == 1 and line["scaling"] == "weak" and line["higher_is_better"] is True
    assert line["value"] == pytest.approx(w.T / (ms * 1e-3))
    assert line["config"]["workload"] == name and line["config"]["tokens"] == w.T
    r = line["roofline"]
    assert {"bound", "achieved", "peak", "unit", "frac", "traffic"} <= set(r)
    assert r["bound"] == bound and r["frac"] == pytest.approx(frac, rel=2e-3)
    assert r["achieved"] == pytest.approx(r["frac"] * r["peak"])
    assert r["unit"] == ("TFLOP/s" if bound == "tensor" else "GB/s")
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == e2e["d2h_bytes_per_step"] == w.T * w.d * 2
    assert e2e["steps"] == 50 and e2e["value"] == pytest.approx(w.T / (ms * 1.01e-3))
    assert line["gpu_launches"] == bench.launches_per_step(w) * steps
    if bound == "tensor":
        assert r["peak"] == (PEAKS["bf16_tflops"] if steps * ms < 1000.0 else PEAKS["bf16_tflops_sustained"])
        assert r["frac_of_spec"] == pytest.approx(r["achieved"] / 2250.0)
    else:
        assert r["active_experts"] == active
    # HBM stages: y and the output at the layer dtype (2 bytes)
    h = line["hbm_stages"]
    assert h["frac"] == pytest.approx(h["gbs"] / PEAKS["hbm_gbs"])
    assert h["combine_gbs"] == pytest.approx(
        (kept * w.d * 2 + w.T * w.d * 2 * (1 + int(w.residual) + int(w.num_shared > 0)) + w.T * w.k * 8)
        / (stages[5] * 1e-3) / 1e9)
    if name != "mixtral":
        assert r["traffic"] is None                          # captured on the Mixtral forward only
    else:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            assert r["traffic"] in (None, json.load(f)["dram_bytes_per_launch"])


@pytest.mark.parametrize("name", list(TRAIN))
def test_train_line(name):
    ms, fst, bst, bound, frac = TRAIN[name]
    w = wl.WORKLOADS[name]
    line = bench.train_line(_args(steps=30, warmup=5), w, 1, ms, np.array(fst), np.array(bst), w.T * w.k, CLOCKS)
    json.dumps(line, default=float)
    assert KEYS <= set(line)
    r = line["roofline"]
    assert r["bound"] == bound and r["frac"] == pytest.approx(frac, rel=2e-3)
    roof = line["expert_gemm"]["backward_gemm_roofline"]
    assert {k: v["bound"] for k, v in roof.items()} == (
        {"dh_gemm": "tensor", "dx_gemm": "tensor", "dw2_gemm": "tensor", "dw13_gemm": "tensor"} if name == "mixtral"
        else {"dh_gemm": "tensor", "dx_gemm": "tensor", "dw2_gemm": "hbm", "dw13_gemm": "hbm"})
    assert line["gpu_launches"] == (bench.launches_per_step(w) + bench.bwd_launches(w)) * 30


def test_launch_counts_follow_the_forward_sequence():
    """Kernels of one moe_forward per workload, counted from its launch
    sequence: router (one fused GEMM with the routing epilogue for bf16
    E <= 32 or the fp32 CUDA-core router; logits GEMM + routing kernel for
    wider routers), dispatch (one CTA for <= 8192 slots, else two launches
    while a table of chunks (512 to 2048 slots) x experts fits in 8192
    entries, else four), the two expert GEMMs (+ two for the shared expert), combine,
    statistics."""
    expect = {"tiny_fp32": 1 + 2 + 2 + 2, "quickstart_bf16": 1 + 2 + 2 + 2, "capacity_e128": 2 + 2 + 2 + 2,
              "mixtral": 1 + 2 + 2 + 2, "deepseek_v3": 2 + 2 + 4 + 2}
    for name, n in expect.items():
        assert bench.launches_per_step(wl.WORKLOADS[name]) == n, name
    big = wl.WORKLOADS["mixtral"].with_(T=150000, E=64)          # 147 2048-slot chunks x 64: four launches
    assert bench.launches_per_step(big) == 2 + 4 + 2 + 2                 # router of 64 experts: two launches
