"""Pins of the oracle's backward: central finite differences of the
oracle's own forward loss (an independent route to every gradient), and the
E = 1 dense special case against torch autograd in fp64."""
import math

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


# ------------------------------------------------------------ bf16 rounding points, worked by hand
def _bf16(v: float) -> float:
    """Nearest bf16 value of an fp64 number (ties to even), by rounding the
    fp64 bit pattern to 7 fraction bits (finite normal values)."""
    import struct
    b = struct.unpack("<Q", struct.pack("<d", float(v)))[0]
    drop = 52 - 7
    rem = b & ((1 << drop) - 1)
    b >>= drop
    half = 1 << (drop - 1)
    if rem > half or (rem == half and (b & 1)):
        b += 1
    return struct.unpack("<d", struct.pack("<Q", b << drop))[0]


def _bf16_array(shape, g, scale):
    return np.vectorize(_bf16)(g.standard_normal(shape) * scale).astype(np.float32)


@pytest.mark.parametrize("act", [wl.SWIGLU, wl.GELU])
def test_backward_bf16_rounding_points_worked_by_hand(act):
    """Three tokens, two experts, top-1 with the raw softmax gate, eight
    hidden units, residual, bf16 storage.  Every gradient is worked out here
    from the chain rule of the "MoE Training: Mixture of Experts" objective
    (loss = <dout, out>; L = main + coef * aux with coef 0), with the bf16
    rounding at each point where a bf16 layer stores a value: the forward's
    H, the stored pre-activations the activation derivative reads,
    dy = gate * dout, and da (the expert output y is kept in fp32).  Each rounding changes some
    of its values here (checked), and with 24 rounded pre-activations per
    point a change that large moves some rounded da, so moving or dropping
    any one rounding in the oracle changes a gradient far beyond the 1e-12
    tolerance."""
    T, d, F, E = 3, 8, 8, 2
    w = wl.Workload("bf16_pin", 84, T=T, d=d, E=E, k=1, F=F, activation=act, score_fn=wl.SOFTMAX, dtype=wl.BF16,
                    router_bias=False, expert_bias=act != wl.SWIGLU, renormalize=False, residual=True)
    g = np.random.default_rng(40 + act)
    x = _bf16_array((T, d), g, 1.0)
    wr = _bf16_array((E, d), g, 0.7)
    w1 = _bf16_array((E, F, d), g, 0.6)
    w2 = _bf16_array((E, d, F), g, 0.6)
    dout = _bf16_array((T, d), g, 1.0)
    inp = {"x": wl.bf16_round(x), "w_router": wl.bf16_round(wr), "w1": wl.bf16_round(w1), "w2": wl.bf16_round(w2)}
    if act == wl.SWIGLU:
        w3 = _bf16_array((E, F, d), g, 0.6)
        inp["w3"] = wl.bf16_round(w3)
    else:
        b1 = _bf16_array((E, F), g, 0.3)
        b2 = _bf16_array((E, d), g, 0.3)
        inp["b1"], inp["b2"] = wl.bf16_round(b1), wl.bf16_round(b2)
    base = orc.layer(w, inp)
    gr = orc.backward(w, inp, base, dout.astype(np.float64), 0.0, 0.0)

    bfv = np.vectorize(_bf16)
    f64 = lambda a: np.asarray(a, np.float64)
    silu = lambda v: v / (1.0 + np.exp(-v))
    erf = np.vectorize(math.erf)
    gelu = lambda v: 0.5 * v * (1.0 + erf(v / math.sqrt(2.0)))
    dgelu = lambda v: 0.5 * (1.0 + erf(v / math.sqrt(2.0))) + v * np.exp(-0.5 * v * v) / math.sqrt(2 * math.pi)
    Wr = f64(wr)
    dx = np.zeros((T, d))
    dW1, dW3, dW2 = np.zeros((E, F, d)), np.zeros((E, F, d)), np.zeros((E, d, F))
    db1, db2, dWr = np.zeros((E, F)), np.zeros((E, d)), np.zeros((E, d))
    points = {k: [] for k in ("h", "dy", "a1", "a3", "da1", "da3")}
    for t in range(T):
        X, D = f64(x[t]), f64(dout[t])
        lg = f64(base["logits"][t])                      # fp32 router logits of the forward
        e = int(base["idx"][t, 0])
        assert e == int(np.argmax(lg))
        p = np.exp(lg - lg.max())
        p /= p.sum()
        gate = p[e]                                      # raw softmax gate (top-1, no renormalisation)
        W1, W2 = f64(w1[e]), f64(w2[e])
        a1 = W1 @ X
        if act == wl.SWIGLU:
            a3 = f64(w3[e]) @ X
            hv = silu(a1) * a3
        else:
            a1 = a1 + f64(b1[e])
            hv = gelu(a1)
        h = bfv(hv)
        y = W2 @ h + (f64(b2[e]) if act != wl.SWIGLU else 0.0)
        dyv = gate * D
        dy = bfv(dyv)
        dh = W2.T @ dy
        a1s = bfv(a1)                                    # the stored pre-activations the derivative reads
        if act == wl.SWIGLU:
            a3s = bfv(a3)
            sg = 1.0 / (1.0 + np.exp(-a1s))
            da1v = dh * a3s * sg * (1.0 + a1s * (1.0 - sg))
            da3v = dh * a1s * sg
            da3 = bfv(da3v)
            points["a3"].append(a3)
            points["da3"].append(da3v)
        else:
            da1v = dh * dgelu(a1s)
        da1 = bfv(da1v)
        for k_, v in (("h", hv), ("dy", dyv), ("a1", a1), ("da1", da1v)):
            points[k_].append(v)
        dgate = float(D @ y)
        assert gr["dgate"][t, 0] == pytest.approx(dgate, rel=1e-12, abs=1e-15)
        dl = -p * p[e] * dgate                           # raw softmax: dl_c = p_c (dg [c = e] - p_e dg)
        dl[e] += p[e] * dgate
        np.testing.assert_allclose(gr["dlogits"][t], dl, rtol=1e-12, atol=1e-15)
        dx[t] = W1.T @ da1 + D + dl @ Wr
        if act == wl.SWIGLU:
            dx[t] += f64(w3[e]).T @ da3
            dW3[e] += np.outer(da3, X)
        dW1[e] += np.outer(da1, X)
        dW2[e] += np.outer(dy, h)
        db1[e] += da1
        db2[e] += dy
        dWr += np.outer(dl, X)
        np.testing.assert_allclose(base["out"][t], gate * y + X, rtol=1e-12, atol=1e-15)
    for name, vals in points.items():                    # every rounding point is live
        if vals:
            v = np.concatenate([np.atleast_1d(u) for u in vals])
            assert np.any(bfv(v) != v), name
    tol = dict(rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(gr["dx"], dx, **tol)
    np.testing.assert_allclose(gr["dw_router"], dWr, **tol)
    np.testing.assert_allclose(gr["dw1"], dW1, **tol)
    np.testing.assert_allclose(gr["dw2"], dW2, **tol)
    if act == wl.SWIGLU:
        np.testing.assert_allclose(gr["dw3"], dW3, **tol)
    else:
        np.testing.assert_allclose(gr["db1"], db1, **tol)
        np.testing.assert_allclose(gr["db2"], db2, **tol)
