"""Backward parity on the GPU: a training forward (moe_forward keeping the
activations) then moe_backward, against the oracle's backward fed the
GPU's own fp32 logits (so the routing is the same, bit for bit) and the same
bf16 dout.  Every gradient meets the bf16 bar: max |gpu - ref| <= 2e-2 of
the reference's RMS."""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl
from tests.gpu_util import dev, float_check, host, weights

pytestmark = pytest.mark.gpu

GRADS = [("dx", "dx"), ("dw_router", "dw_router"), ("db_router", "db_router"), ("dw1", "dw1"), ("db1", "db1"),
         ("dw3", "dw3"), ("dw2", "dw2"), ("db2", "db2"), ("shared_dw1", "dsw1"), ("shared_dw3", "dsw3"),
         ("shared_dw2", "dsw2"), ("dw1_rows", "dw1_rows"), ("dw3_rows", "dw3_rows"), ("dw2_cols", "dw2_cols"),
         ("db1_units", "db1_units")]


def run_backward(w, inp, aux, z, seed=5, units=None):
    """GPU and oracle gradients.  With ``units`` (u = expert * F + f) the
    expert weight gradients are compared on those rows only."""
    layer = moe.TrainingLayer(moe.config_for(w), weights(inp), dev(inp["sel_bias"]) if "sel_bias" in inp else None)
    x = dev(inp["x"])
    layer.forward(x)
    g = np.random.default_rng(seed)
    dout_h = wl.bf16_round(g.standard_normal((w.T, w.d)).astype(np.float32))
    grads = layer.backward(dev(dout_h), aux, z)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    if units is None:
        got = {k: host(v) for k, v in grads.items()}
    else:
        got = {k: host(grads[k]) for k in ("dx", "dw_router", "db_router", "db2") if k in grads}
        r1, r3, c2, b1 = [], [], [], []
        for u in units:
            e, f = divmod(int(u), w.F)
            if e < w.E:
                r1.append(grads["dw1"][e, f])
                c2.append(grads["dw2"][e, :, f])
                if "dw3" in grads:
                    r3.append(grads["dw3"][e, f])
                if "db1" in grads:
                    b1.append(grads["db1"][e, f])
            else:
                r1.append(grads["shared_dw1"][f])
                c2.append(grads["shared_dw2"][:, f])
                if "shared_dw3" in grads:
                    r3.append(grads["shared_dw3"][f])
        got["dw1_rows"] = host(torch.stack(r1))
        got["dw2_cols"] = host(torch.stack(c2))
        if r3:
            got["dw3_rows"] = host(torch.stack(r3))
        if b1 and len(b1) == len(units):
            got["db1_units"] = host(torch.stack(b1))
    lg = host(layer.io["logits"])
    r = orc.route(w, lg, inp.get("sel_bias"))
    dsp = orc.dispatch(w, r["idx"])
    np.testing.assert_array_equal(host(layer.io["topk_idx"]).reshape(w.T, w.k), r["idx"])
    np.testing.assert_array_equal(host(layer.io["inv"]).reshape(-1)[:w.T * w.k], dsp["inv"])
    fwd = dict(logits=lg, idx=r["idx"], gate=r["gate"], inv=dsp["inv"], counts=dsp["counts"])
    ref = orc.backward(w, inp, fwd, wl.bf16_to_f32(dout_h).astype(np.float64), aux, z, units=units)
    ref["inv"] = dsp["inv"]
    ref["idx"] = r["idx"]
    return got, ref


def check_grads(w, got, ref, tag):
    n = 0
    for gk, rk in GRADS:
        if gk not in got or ref.get(rk) is None:
            continue
        a, b = got[gk], ref[rk]
        if gk == "dx":
            a = a[:w.T]
        float_check(a.reshape(b.shape), b, w, f"{tag} {gk}")
        n += 1
    assert n >= 5


CASES = {
    # name: Workload kwargs, aux, z
    "gelu_bias_softmax": (dict(T=300, d=256, E=8, k=2, F=512, activation=wl.GELU, score_fn=wl.SOFTMAX,
                               router_bias=True, expert_bias=True), 0.01, 0.001),
    "swiglu_residual": (dict(T=500, d=256, E=8, k=2, F=384, activation=wl.SWIGLU, score_fn=wl.SOFTMAX,
                             router_bias=False, expert_bias=False, residual=True), 0.02, 0.0),
    "sigmoid_shared": (dict(T=200, d=192, E=16, k=4, F=256, activation=wl.SWIGLU, score_fn=wl.SIGMOID,
                            router_bias=True, expert_bias=False, residual=True, num_shared=1), 0.01, 0.001),
    "dropping_top2": (dict(T=400, d=128, E=8, k=2, F=256, activation=wl.SWIGLU, score_fn=wl.SOFTMAX,
                           router_bias=True, expert_bias=False, drop_tokens=True, capacity_factor=0.5,
                           min_capacity=4), 0.05, 0.01),
    "switch_relu_raw": (dict(T=333, d=128, E=4, k=1, F=256, activation=wl.RELU, score_fn=wl.SOFTMAX,
                             router_bias=True, expert_bias=True, renormalize=False), 0.1, 0.01),
    # skewed router: empty experts, experts with a few rows and with more than
    # 64 (partial K blocks everywhere in the weight-gradient GEMMs)
    "skewed_segments": (dict(T=210, d=128, E=16, k=2, F=128, activation=wl.SWIGLU, score_fn=wl.SOFTMAX,
                             router_bias=True, expert_bias=False, residual=True), 0.02, 0.01),
}


@pytest.mark.parametrize("case", list(CASES))
def test_backward_parity(case):
    kw, aux, z = CASES[case]
    w = wl.Workload(f"bwd_{case}", 90 + len(case), dtype=wl.BF16, **kw)
    inp = wl.make_inputs(w)
    if case == "skewed_segments":
        # two popular experts, a middle group, rare ones and four never chosen
        inp["b_router"] = np.array([0.5, 0.4, 0, 0, 0, 0, -0.15, -0.25, -0.35, -0.45, -0.55, -0.65, -40, -40, -40, -40],
                                   np.float32)
    got, ref = run_backward(w, inp, aux, z)
    if w.drop_tokens:
        assert (ref["inv"] < 0).any()               # slots were dropped
    if case == "skewed_segments":
        counts = np.bincount(ref["idx"].reshape(-1), minlength=w.E)
        assert (counts == 0).any() and ((counts > 0) & (counts < 8)).any() and (counts > 64).any(), counts
    check_grads(w, got, ref, case)


@pytest.mark.parametrize("name,T", [("quickstart_bf16", 256), ("capacity_e128", 512), ("mixtral", 128),
                                    ("deepseek_v3", 64)])
def test_backward_parity_workload_shapes(name, T):
    """The benchmark workloads' layer shapes (d, F, E, k, activation,
    scoring, shared expert) at a few hundred tokens; expert weight
    gradients on 48 sampled rows (every expert's first row, the shared
    expert's rows included)."""
    w = wl.WORKLOADS[name].scaled(T)
    inp = wl.make_inputs(w)
    g = np.random.default_rng(T)
    n_exp = w.E + w.num_shared
    units = np.unique(np.concatenate([np.arange(min(n_exp, 16)) * w.F,
                                      g.choice(n_exp * w.F, size=32, replace=False)])).astype(np.int64)
    got, ref = run_backward(w, inp, 0.01, 0.001, units=units)
    check_grads(w, got, ref, name)


def test_backward_empty_batch():
    w = wl.WORKLOADS["quickstart_bf16"].scaled(0)
    inp = wl.make_inputs(w)
    layer = moe.TrainingLayer(moe.config_for(w), weights(inp))
    layer.forward(dev(inp["x"]))
    grads = layer.backward(torch.empty(0, w.d, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    for k, v in grads.items():
        if k != "dx":
            assert torch.count_nonzero(v).item() == 0, k


def test_backward_deterministic():
    w = wl.Workload("bwd_det", 99, T=300, d=128, E=8, k=2, F=256, activation=wl.SWIGLU, score_fn=wl.SOFTMAX,
                    dtype=wl.BF16, router_bias=True, expert_bias=False)
    inp = wl.make_inputs(w)
    a, _ = run_backward(w, inp, 0.01, 0.001)
    b, _ = run_backward(w, inp, 0.01, 0.001)
    for k in a:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
