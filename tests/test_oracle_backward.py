"""Pins of the oracle's backward: central finite differences of the
oracle's own forward loss (an independent route to every gradient), and the
E = 1 dense special case against torch autograd in fp64."""
import numpy as np
import pytest
import torch

from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl


def _inputs(w, seed, scale_router=1.0):
    """fp32 tensors at scales that put the activations in their non-linear
    range and keep the routing decisions far from ties."""
    g = np.random.default_rng(seed)
    f = lambda *s, sd=1.0: (g.standard_normal(s) * sd).astype(np.float32)
    inp = dict(x=f(w.T, w.d), w_router=f(w.E, w.d, sd=scale_router),
               w1=f(w.E, w.F, w.d, sd=0.4), w2=f(w.E, w.d, w.F, sd=0.4))
    if w.router_bias:
        inp["b_router"] = f(w.E, sd=0.5)
    if w.activation == wl.SWIGLU:
        inp["w3"] = f(w.E, w.F, w.d, sd=0.4)
    elif w.expert_bias:
        inp["b1"] = f(w.E, w.F, sd=0.3)
        inp["b2"] = f(w.E, w.d, sd=0.3)
    if w.score_fn == wl.SIGMOID:
        inp["sel_bias"] = f(w.E, sd=0.3)
    if w.num_shared:
        inp["shared_w1"] = f(w.num_shared, w.F, w.d, sd=0.4)
        inp["shared_w2"] = f(w.num_shared, w.d, w.F, sd=0.4)
        if w.activation == wl.SWIGLU:
            inp["shared_w3"] = f(w.num_shared, w.F, w.d, sd=0.4)
    return inp


GRAD_OF = {"x": "dx", "w_router": "dw_router", "b_router": "db_router", "w1": "dw1", "b1": "db1", "w3": "dw3",
           "w2": "dw2", "b2": "db2", "shared_w1": "dsw1", "shared_w3": "dsw3", "shared_w2": "dsw2"}

CASES = {
    # name: (score, activation, renorm, k, router_bias, expert_bias, shared, residual, drop, aux, z)
    "softmax_gelu_bias": (wl.SOFTMAX, wl.GELU, True, 2, True, True, 0, False, False, 0.3, 0.2),
    "switch_raw_relu": (wl.SOFTMAX, wl.RELU, False, 1, True, True, 0, True, False, 0.5, 0.1),
    "softmax_raw_top2": (wl.SOFTMAX, wl.GELU, False, 2, False, False, 0, False, False, 0.0, 0.3),
    "sigmoid_swiglu_shared": (wl.SIGMOID, wl.SWIGLU, True, 2, False, False, 1, True, False, 0.2, 0.2),
    "sigmoid_raw": (wl.SIGMOID, wl.RELU, False, 2, True, True, 0, False, False, 0.1, 0.0),
    "dropping": (wl.SOFTMAX, wl.SWIGLU, True, 2, True, False, 0, True, True, 0.4, 0.1),
}


@pytest.mark.parametrize("case", list(CASES))
def test_backward_matches_finite_differences(case):
    score, act, renorm, k, rb, eb, shared, resid, drop, aux, z = CASES[case]
    w = wl.Workload(case, 80, T=7, d=8, E=4, k=k, F=6, activation=act, score_fn=score, dtype=wl.F32,
                    router_bias=rb, expert_bias=eb, renormalize=renorm, num_shared=shared, residual=resid,
                    drop_tokens=drop, capacity_factor=0.75, min_capacity=2)
    inp = _inputs(w, seed=len(case))
    g = np.random.default_rng(7)
    dout = g.standard_normal((w.T, w.d))
    base = orc.layer(w, inp)
    if drop:
        assert (base["inv"] < 0).any()          # the case really drops slots
    grads = orc.backward(w, inp, base, dout, aux, z)
    eps = 1e-3
    checked = picked = 0
    for name, gname in GRAD_OF.items():
        if name not in inp:
            continue
        arr = inp[name]
        flat = arr.reshape(-1)
        picks = g.choice(flat.size, size=min(flat.size, 24), replace=False)
        picked += len(picks)
        for i in picks:
            old = flat[i]
            vals = []
            for sgn in (1, -1):
                flat[i] = old + sgn * np.float32(eps)
                r = orc.layer(w, inp)
                same = np.array_equal(r["idx"], base["idx"]) and np.array_equal(r["inv"], base["inv"])
                vals.append((orc.loss(w, inp, dout, aux, z), same, float(flat[i])))
            flat[i] = old
            if not (vals[0][1] and vals[1][1]):
                continue                             # a routing decision flipped: not differentiable here
            fd = (vals[0][0] - vals[1][0]) / (vals[0][2] - vals[1][2])
            an = grads[gname].reshape(-1)[i]
            assert abs(fd - an) <= 2e-3 * max(1.0, abs(an)), (name, int(i), fd, an)
            checked += 1
    assert checked >= 0.8 * picked            # few coordinates sit next to a routing decision


@pytest.mark.parametrize("act", [wl.GELU, wl.SWIGLU, wl.RELU])
def test_backward_dense_special_case_matches_autograd(act):
    """E = 1, k = 1 with renormalisation: gate 1, no router gradient from
    the gate, and the layer is a dense FFN whose gradients torch autograd
    computes in fp64."""
    w = wl.Workload("dense", 81, T=9, d=12, E=1, k=1, F=10, activation=act, score_fn=wl.SOFTMAX, dtype=wl.F32,
                    router_bias=True, expert_bias=act != wl.SWIGLU, residual=True)
    inp = _inputs(w, seed=3 + act)
    dout = np.random.default_rng(1).standard_normal((w.T, w.d))
    base = orc.layer(w, inp)
    gr = orc.backward(w, inp, base, dout, 0.0, 0.0)
    t = {k: torch.tensor(v.astype(np.float64), requires_grad=True) for k, v in inp.items()}
    a = t["x"] @ t["w1"][0].T
    if act == wl.SWIGLU:
        h = torch.nn.functional.silu(a) * (t["x"] @ t["w3"][0].T)
    else:
        a = a + t["b1"][0]
        h = torch.nn.functional.gelu(a) if act == wl.GELU else torch.relu(a)
    y = h @ t["w2"][0].T
    if act != wl.SWIGLU:
        y = y + t["b2"][0]
    out = y + t["x"]
    (out * torch.tensor(dout)).sum().backward()
    np.testing.assert_allclose(gr["dx"], t["x"].grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gr["dw1"][0], t["w1"].grad[0].numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(gr["dw2"][0], t["w2"].grad[0].numpy(), rtol=1e-10, atol=1e-12)
    if act == wl.SWIGLU:
        np.testing.assert_allclose(gr["dw3"][0], t["w3"].grad[0].numpy(), rtol=1e-10, atol=1e-12)
    else:
        np.testing.assert_allclose(gr["db1"][0], t["b1"].grad[0].numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(gr["db2"][0], t["b2"].grad[0].numpy(), rtol=1e-10, atol=1e-12)
    # one expert, gate identically 1: no gradient reaches the router
    assert np.all(gr["dlogits"] == 0.0) and np.all(gr["dw_router"] == 0.0)


def test_backward_dgate_is_output_projection():
    """dgate[t, j] = <dout_t, y_{t,j}>: with dout = e_n the gate gradient is
    coordinate n of the expert output, checked against the forward's own
    expert evaluation."""
    w = wl.Workload("dg", 82, T=5, d=6, E=3, k=2, F=4, activation=wl.GELU, score_fn=wl.SOFTMAX, dtype=wl.F32,
                    router_bias=False, expert_bias=True)
    inp = _inputs(w, seed=11)
    base = orc.layer(w, inp)
    dout = np.zeros((w.T, w.d))
    dout[:, 2] = 1.0
    gr = orc.backward(w, inp, base, dout)
    for t in range(w.T):
        for j in range(w.k):
            y = orc.expert_row(w, inp, int(base["idx"][t, j]), inp["x"][t].astype(np.float64))
            assert abs(gr["dgate"][t, j] - y[2]) < 1e-12


def test_backward_units_equal_full_arrays():
    """The per-unit weight gradients equal the rows / columns of the full
    arrays (shared expert included)."""
    w = wl.Workload("units", 83, T=9, d=8, E=3, k=2, F=5, activation=wl.SWIGLU, score_fn=wl.SIGMOID, dtype=wl.F32,
                    router_bias=True, expert_bias=False, num_shared=1, residual=True)
    inp = _inputs(w, seed=21)
    base = orc.layer(w, inp)
    dout = np.random.default_rng(2).standard_normal((w.T, w.d))
    full = orc.backward(w, inp, base, dout, 0.1, 0.1)
    units = np.array([0, 4, 7, 14, 15, 19], np.int64)       # 15.. are the shared expert's rows
    part = orc.backward(w, inp, base, dout, 0.1, 0.1, units=units)
    for i, u in enumerate(units):
        e, f = divmod(int(u), w.F)
        W1 = full["dw1"][e] if e < w.E else full["dsw1"][e - w.E]
        W3 = full["dw3"][e] if e < w.E else full["dsw3"][e - w.E]
        W2 = full["dw2"][e] if e < w.E else full["dsw2"][e - w.E]
        np.testing.assert_allclose(part["dw1_rows"][i], W1[f], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(part["dw3_rows"][i], W3[f], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(part["dw2_cols"][i], W2[:, f], rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(part["dx"], full["dx"])
