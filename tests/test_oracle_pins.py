"""Pins of the CPU oracle to what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: numbers
printed on (or hand-derived from formulas printed on) the pages, closed
forms, invariants, library routines (numpy / scipy / torch CPU), and brute
force on tiny inputs.  Marked ``not gpu`` implicitly (no marker).
"""
import dataclasses
import itertools
import math

import numpy as np
import pytest
import scipy.special as sp
import torch

from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl


def _cfg(**kw):
    base = dict(name="t", index=9, T=16, d=8, E=4, k=2, F=12, activation=wl.GELU,
                score_fn=wl.SOFTMAX, dtype=wl.F32, router_bias=True, expert_bias=True)
    base.update(kw)
    return wl.Workload(**base)


# ------------------------------------------------------------ parameter counts
def test_param_counts_compare_moe_vs_dense(golden):
    g = golden("moe_vs_dense_768.json")
    pc = orc.param_counts(g["d_model"], g["d_ff"], g["num_experts"], g["top_k"], gated=False)
    dense = pc["expert"]  # the dense FFN of the same width is one expert
    assert dense == g["dense"]
    assert pc["router"] == g["router"]
    assert pc["total"] == g["moe_total"]
    assert pc["active"] == g["moe_active"]
    assert f"{pc['total'] / dense:.1f}" == g["total_over_dense_1dp"]
    assert f"{pc['active'] / dense:.1f}" == g["active_over_dense_1dp"]
    assert f"{pc['total'] / pc['active']:.1f}" == g["efficiency_1dp"]


def test_param_counts_mixtral(golden):
    g = golden("mixtral_params.json")
    pc = orc.param_counts(g["d_model"], g["d_ff"], g["num_experts"], g["top_k"], gated=True)
    assert pc["expert"] == g["expert_params"] == 176_160_768
    assert pc["router"] == g["gate_params_per_layer"]
    per_layer_rest = g["attention_params_per_layer"] + g["layernorm_params_per_layer"]
    transformer = (pc["total"] + per_layer_rest) * g["layers"]
    assert transformer == g["transformer_total"]
    assert transformer + g["embed_and_output_params"] == g["total"]
    active = (pc["active"] + per_layer_rest) * g["layers"] + g["embed_and_output_params"]
    assert active == g["active"]


# ------------------------------------------------------------ capacity
def test_capacity_closed_forms(golden):
    for case in golden("capacity.json")["cases"]:
        w = _cfg(T=case["T"], E=case["E"], k=1, drop_tokens=True,
                 capacity_factor=case["cf"], min_capacity=case["min_capacity"])
        assert orc.capacity(w) == case["capacity"], case
    assert orc.capacity(wl.WORKLOADS["capacity_e128"]) == 80


# ------------------------------------------------------------ fp32 sigmoid key
def _ulp32(v):
    v = np.float32(abs(v))
    return float(np.spacing(v)) if v > 0 else float(np.finfo(np.float32).smallest_subnormal)


def test_exp32_within_two_ulp_of_exp():
    xs = np.linspace(-87.0, 88.0, 40001, dtype=np.float32)
    worst = 0.0
    for x in xs:
        got = orc.exp32(float(x))
        ref = math.exp(float(x))
        err = abs(got - ref) / _ulp32(ref)
        worst = max(worst, err)
    assert worst <= 2.0, worst
    assert orc.exp32(0.0) == 1.0
    assert orc.exp32(100.0) == math.inf
    assert orc.exp32(-100.0) == 0.0
    assert math.isnan(orc.exp32(float("nan")))


def test_sigmoid32_properties():
    assert orc.sigmoid32(0.0) == 0.5
    xs = np.sort(np.random.default_rng(3).uniform(-20, 20, 20000).astype(np.float32))
    vals = np.array([orc.sigmoid32(float(x)) for x in xs], dtype=np.float64)
    assert np.all(np.diff(vals) >= 0.0)                       # monotone
    ref = sp.expit(xs.astype(np.float64))
    err = np.abs(vals - ref) / np.array([_ulp32(r) for r in ref])
    assert err.max() <= 3.0                                   # a few ulp of the exact value
    assert orc.sigmoid32(200.0) == 1.0 and orc.sigmoid32(-200.0) == 0.0


# ------------------------------------------------------------ elementwise
def test_activations_against_library():
    xs = np.linspace(-6, 6, 241)
    for x in xs:
        assert abs(orc.gelu(x) - x * sp.ndtr(x)) < 1e-14          # GELU(x) = x * Phi(x)
        assert abs(orc.silu(x) - x * sp.expit(x)) < 1e-14
    assert abs(orc.gelu(1.0) - 0.8413447460685429) < 1e-15        # Phi(1)


def test_round_bf16_matches_bit_rounding():
    g = np.random.default_rng(4)
    v = np.concatenate([g.standard_normal(4000), g.uniform(-1e4, 1e4, 1000)]).astype(np.float32)
    a = np.array([orc.round_bf16(float(x)) for x in v])
    b = wl.bf16_to_f32(wl.bf16_round(v)).astype(np.float64)
    assert np.array_equal(a, b)
    assert orc.round_bf16(1.0 + 2.0 ** -8) == 1.0                # tie -> even
    assert orc.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # tie -> even (up)


# ------------------------------------------------------------ router logits
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
def test_router_logits_against_matmul(dtype):
    w = _cfg(T=37, d=24, E=6, dtype=dtype)
    inp = wl.make_inputs(w)
    inp["b_router"] = np.linspace(-1, 1, w.E).astype(np.float32)
    got = orc.router_logits(w, inp)
    X = inp["x"] if dtype == wl.F32 else wl.bf16_to_f32(inp["x"])
    W = inp["w_router"] if dtype == wl.F32 else wl.bf16_to_f32(inp["w_router"])
    ref = X.astype(np.float64) @ W.astype(np.float64).T + inp["b_router"].astype(np.float64)
    assert np.all(np.abs(got.astype(np.float64) - ref) <= np.spacing(np.abs(ref).astype(np.float32)))


# ------------------------------------------------------------ routing
def _topk_by_sort(keys, k):
    return [e for _, e in sorted(((-float(v), e) for e, v in enumerate(keys)))[:k]]


@pytest.mark.parametrize("E,k", [(4, 1), (4, 2), (8, 2), (8, 8), (16, 3), (64, 8)])
def test_route_softmax_selection_gates_lse(E, k):
    w = _cfg(T=200, E=E, k=k)
    g = np.random.default_rng(E * 10 + k)
    lg = g.standard_normal((w.T, E)).astype(np.float32)
    lg[::5] = np.round(lg[::5] * 2) / 2                      # plenty of exact ties
    r = orc.route(w, lg)
    for t in range(w.T):
        assert list(r["idx"][t]) == _topk_by_sort(lg[t], k)
    np.testing.assert_allclose(r["gate"].sum(1), 1.0, atol=1e-15)
    probs = sp.softmax(lg.astype(np.float64), axis=1)
    sel = np.take_along_axis(probs, r["idx"].astype(np.int64), 1)
    np.testing.assert_allclose(r["gate"], sel / sel.sum(1, keepdims=True), rtol=1e-12)
    np.testing.assert_allclose(r["lse"], sp.logsumexp(lg.astype(np.float64), axis=1), rtol=1e-14)
    np.testing.assert_allclose(r["prob_sum"], probs.sum(0), rtol=1e-12)
    if k == 1:
        assert np.all(r["gate"] == 1.0)
        assert np.array_equal(r["idx"][:, 0], np.argmax(lg, axis=1))   # argmax: first maximum
    if k == E:
        assert all(sorted(r["idx"][t]) == list(range(E)) for t in range(w.T))


def test_route_without_renormalisation_returns_probabilities():
    w = _cfg(T=50, E=8, k=2, renormalize=False)
    lg = np.random.default_rng(1).standard_normal((w.T, w.E)).astype(np.float32)
    r = orc.route(w, lg)
    probs = sp.softmax(lg.astype(np.float64), axis=1)
    np.testing.assert_allclose(r["gate"], np.take_along_axis(probs, r["idx"].astype(np.int64), 1),
                               rtol=1e-12)


def test_route_top2_worked_example(golden):
    g = golden("top2_gate_example.json")
    w = _cfg(T=1, E=g["num_experts"], k=g["top_k"])
    r = orc.route(w, np.array([g["logits"]], np.float32))
    assert list(r["idx"][0]) == g["expected_idx"]
    np.testing.assert_allclose(r["gate"][0], g["expected_gates"], atol=1e-6)


def test_route_sigmoid_keys_bias_and_gates():
    w = _cfg(T=300, E=32, k=4, score_fn=wl.SIGMOID)
    g = np.random.default_rng(7)
    lg = g.standard_normal((w.T, w.E)).astype(np.float32)
    b = g.uniform(-0.1, 0.1, w.E).astype(np.float32)
    r = orc.route(w, lg, b)
    for t in range(w.T):
        keys = [np.float32(np.float32(orc.sigmoid32(float(v))) + b[e]) for e, v in enumerate(lg[t])]
        assert list(r["idx"][t]) == _topk_by_sort(keys, w.k)
    sig = sp.expit(lg.astype(np.float64))
    sel = np.take_along_axis(sig, r["idx"].astype(np.int64), 1)
    np.testing.assert_allclose(r["gate"], sel / sel.sum(1, keepdims=True), rtol=1e-12)
    # the selection bias moves the choice but never the gate value
    r0 = orc.route(w, lg, np.zeros(w.E, np.float32))
    assert not np.array_equal(r0["idx"], r["idx"])


def test_route_bruteforce_subsets_tiny():
    """Top-k = the k-subset whose smallest key beats every excluded key
    (ties: lower index), checked by enumerating all C(E,k) subsets."""
    w = _cfg(T=60, E=6, k=3)
    lg = np.round(np.random.default_rng(11).standard_normal((w.T, w.E)) * 2).astype(np.float32) / 2
    r = orc.route(w, lg)
    for t in range(w.T):
        def better(a, b):  # a ranks before b
            return lg[t, a] > lg[t, b] or (lg[t, a] == lg[t, b] and a < b)
        valid = [s for s in itertools.combinations(range(w.E), w.k)
                 if all(better(a, b) for a in s for b in range(w.E) if b not in s)]
        assert len(valid) == 1
        assert set(r["idx"][t]) == set(valid[0])


# ------------------------------------------------------------ dispatch
def _check_dispatch_invariants(w, idx, dsp, cap):
    S = w.T * w.k
    counts, kept, off, perm, inv = (dsp[n] for n in ("counts", "kept", "offsets", "perm", "inv"))
    assert np.array_equal(counts, np.bincount(idx.reshape(-1), minlength=w.E))
    assert np.array_equal(kept, np.minimum(counts, cap))
    assert off[0] == 0 and np.array_equal(np.diff(off), kept)
    nk = off[-1]
    assert np.all(perm[nk:] == -1) and np.all(perm[:nk] >= 0)
    kept_slots = np.nonzero(inv >= 0)[0]
    assert len(kept_slots) == nk
    assert np.array_equal(perm[inv[kept_slots]], kept_slots)          # perm o inv = id
    assert np.array_equal(inv[perm[:nk]], np.arange(nk))               # inv o perm = id
    flat = idx.reshape(-1)
    for e in range(w.E):
        seg = perm[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)
        prio = (seg % w.k) * w.T + seg // w.k
        assert np.all(np.diff(prio) > 0)                                 # priority order
        assert len(seg) <= cap
    # the dropped slots of an expert are exactly its lowest-priority ones
    for e in range(w.E):
        slots = np.nonzero(flat == e)[0]
        prio = (slots % w.k) * w.T + slots // w.k
        order = slots[np.argsort(prio)]
        assert np.all(inv[order[:kept[e]]] >= 0) and np.all(inv[order[kept[e]:]] == -1)


@pytest.mark.parametrize("drop", [False, True])
@pytest.mark.parametrize("E,k,T", [(4, 2, 64), (8, 1, 333), (16, 4, 129), (128, 1, 1000)])
def test_dispatch_invariants(E, k, T, drop):
    w = _cfg(T=T, E=E, k=k, drop_tokens=drop, capacity_factor=1.0, min_capacity=4)
    g = np.random.default_rng(E + k + T)
    pop = np.exp(g.standard_normal(E) * 1.5)
    idx = np.stack([g.choice(E, size=k, replace=False, p=pop / pop.sum()) for _ in range(T)]).astype(np.int32)
    dsp = orc.dispatch(w, idx)
    _check_dispatch_invariants(w, idx, dsp, orc.capacity(w))


def test_dispatch_all_on_one_expert_keeps_first_tokens():
    w = _cfg(T=50, E=4, k=1, drop_tokens=True, capacity_factor=1.0, min_capacity=4)
    cap = orc.capacity(w)  # ceil(12.5) = 13
    assert cap == 13
    idx = np.full((w.T, 1), 2, np.int32)
    d = orc.dispatch(w, idx)
    assert d["counts"].tolist() == [0, 0, 50, 0] and d["kept"].tolist() == [0, 0, 13, 0]
    assert d["perm"][:13].tolist() == list(range(13))
    assert np.all(d["inv"][13:] == -1) and d["inv"][:13].tolist() == list(range(13))


def test_dispatch_priority_rank_major_hand_case():
    # T=3, k=2: slots s = t*2 + j.  Priority: (t0,j0),(t1,j0),(t2,j0),(t0,j1),(t1,j1),(t2,j1)
    w = _cfg(T=3, E=2, k=2, drop_tokens=True, capacity_factor=1.0, min_capacity=2)
    idx = np.array([[0, 1], [1, 0], [0, 1]], np.int32)
    d = orc.dispatch(w, idx)
    # expert 0 gets slots (t0,j0)=0, (t2,j0)=4, (t1,j1)=3 -> keeps first 2 by priority: 0, 4
    # expert 1 gets (t1,j0)=2, (t0,j1)=1, (t2,j1)=5 -> keeps 2, 1
    assert d["counts"].tolist() == [3, 3] and d["kept"].tolist() == [2, 2]
    assert d["perm"].tolist() == [0, 4, 2, 1, -1, -1]
    assert d["inv"].tolist() == [0, 3, 2, -1, 1, -1]


# ------------------------------------------------------------ stats
def test_aux_loss_is_one_under_uniform_routing():
    E, T = 4, 16
    w = _cfg(T=T, E=E, k=1)
    v = np.array([2.0, 0.5, -0.25, -1.0], np.float32)
    lg = np.stack([np.roll(v, t % E) for t in range(T)])   # argmax = t mod E, probs cycle
    r = orc.route(w, lg)
    dsp = orc.dispatch(w, r["idx"])
    assert dsp["counts"].tolist() == [4, 4, 4, 4]
    st = orc.stats(w, dsp["counts"], dsp["kept"], r["prob_sum"], r["lse"])
    np.testing.assert_allclose(st["P"], 1 / E, rtol=1e-14)
    assert abs(st["aux"] - 1.0) < 1e-14


def test_aux_loss_collapse_and_zloss_closed_form():
    E, T = 8, 32
    w = _cfg(T=T, E=E, k=2)
    lg = np.zeros((T, E), np.float32)
    r = orc.route(w, lg)
    dsp = orc.dispatch(w, r["idx"])
    st = orc.stats(w, dsp["counts"], dsp["kept"], r["prob_sum"], r["lse"])
    assert abs(st["z"] - math.log(E) ** 2) < 1e-13            # lse of zeros = ln E
    # every token on experts 0 and 1 with P concentrated on expert 0
    lg2 = np.full((T, E), -80.0, np.float32)
    lg2[:, 0], lg2[:, 1] = 40.0, 0.0
    r2 = orc.route(w, lg2)
    d2 = orc.dispatch(w, r2["idx"])
    st2 = orc.stats(w, d2["counts"], d2["kept"], r2["prob_sum"], r2["lse"])
    # f = (1/2, 1/2, 0...), P_0 -> 1  =>  aux -> E * 1/2
    assert abs(st2["aux"] - E / 2) < 1e-9
    np.testing.assert_allclose(st2["f"][:2], [0.5, 0.5])


def test_monitoring_metrics(golden):
    g = golden("monitoring.json")
    w = _cfg(T=g["T"], E=g["E"], k=g["k"])
    st = orc.stats(w, np.array(g["counts"]), np.array(g["kept"]), np.zeros(w.E), np.zeros(w.T))
    for key, val in g["expected"].items():
        assert abs(st[key] - val) < 1e-15, key
    st0 = orc.stats(w, np.array([5, 0, 4, 3]), np.array([5, 0, 4, 3]), np.zeros(4), np.zeros(w.T))
    assert st0["imbalance"] == math.inf and st0["utilization"] == 0.75


def test_bias_update_sign_pattern():
    w = _cfg(T=8, E=4, k=4)                         # S = 32, mean load 8
    b = np.array([0.05, -0.02, 0.0, 0.1], np.float32)
    out = orc.bias_update(w, np.array([10, 8, 6, 8]), b, 0.001)
    g = np.float32(0.001)
    expect = np.array([b[0] - g, b[1], b[2] + g, b[3]], np.float32)  # fp32 add of +-gamma
    assert np.array_equal(out, expect)


# ------------------------------------------------------------ experts / layer
def _f64(a, dtype):
    a = a if dtype == wl.F32 else wl.bf16_to_f32(a)
    return torch.tensor(np.asarray(a, dtype=np.float64))


@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("dtype", [wl.F32, wl.BF16])
@pytest.mark.parametrize("act", [wl.GELU, wl.RELU, wl.SWIGLU])
def test_single_expert_layer_is_a_dense_ffn(act, dtype, residual):
    """E=1, k=1: the layer is one dense FFN (torch CPU float64 as the
    library), plus x when the residual is on.  For bf16 storage the
    activation output is rounded to bf16 before the second Linear."""
    w = _cfg(T=9, d=16, E=1, k=1, F=40, activation=act, expert_bias=act != wl.SWIGLU,
             dtype=dtype, residual=residual)
    inp = wl.make_inputs(w)
    if act != wl.SWIGLU:
        g = np.random.default_rng(2)
        b1 = g.standard_normal((1, w.F)).astype(np.float32) * 0.1
        b2 = g.standard_normal((1, w.d)).astype(np.float32) * 0.1
        inp["b1"] = b1 if dtype == wl.F32 else wl.bf16_round(b1)
        inp["b2"] = b2 if dtype == wl.F32 else wl.bf16_round(b2)
    ref = orc.layer(w, inp)
    assert np.all(ref["gate"] == 1.0)
    X, W1, W2 = _f64(inp["x"], dtype), _f64(inp["w1"][0], dtype), _f64(inp["w2"][0], dtype)
    if act == wl.SWIGLU:
        W3 = _f64(inp["w3"][0], dtype)
        H = torch.nn.functional.silu(X @ W1.T) * (X @ W3.T)
    else:
        A = torch.nn.functional.linear(X, W1, _f64(inp["b1"][0], dtype))
        H = torch.nn.functional.gelu(A) if act == wl.GELU else torch.relu(A)
    if dtype == wl.BF16:  # bf16 storage of H (numpy bit rounding of the fp32 value)
        H = torch.tensor(wl.bf16_to_f32(wl.bf16_round(H.numpy().astype(np.float32))).astype(np.float64))
    Y = H @ W2.T
    if act != wl.SWIGLU:
        Y = Y + _f64(inp["b2"][0], dtype)
    if residual:
        Y = Y + X
    np.testing.assert_allclose(ref["out"], Y.numpy(), rtol=1e-12, atol=1e-13)


def _tiny_variants():
    yield wl.WORKLOADS["tiny_fp32"]
    base = _cfg(T=40, d=16, E=6, k=2, F=24, dtype=wl.BF16)
    yield base.with_(name="gelu_bf16_bias")
    yield base.with_(name="relu_cap", activation=wl.RELU, drop_tokens=True, capacity_factor=1.0,
                     min_capacity=2)
    yield base.with_(name="swiglu_shared_res", activation=wl.SWIGLU, expert_bias=False,
                     router_bias=False, num_shared=1, residual=True)
    yield base.with_(name="sigmoid_k3", score_fn=wl.SIGMOID, k=3, activation=wl.SWIGLU,
                     expert_bias=False, num_shared=1, residual=True)


@pytest.mark.parametrize("w", list(_tiny_variants()), ids=lambda w: w.name)
def test_sparse_loop_equals_bruteforce_dense(w):
    inp = wl.make_inputs(w)
    if w.score_fn == wl.SIGMOID and "sel_bias" not in inp:
        inp["sel_bias"] = np.random.default_rng(5).uniform(-0.1, 0.1, w.E).astype(np.float32)
    if w.expert_bias and w.name != "tiny_fp32":
        pass
    ref = orc.layer(w, inp)
    allv, dense = orc.dense_all(w, inp, ref["idx"], ref["gate"], ref["inv"])
    np.testing.assert_allclose(ref["out"], dense, rtol=0, atol=1e-12)
    # every expert evaluation of the brute force path equals the single-row path
    X = inp["x"] if w.dtype == wl.F32 else wl.bf16_to_f32(inp["x"])
    for t in (0, w.T - 1):
        for e in range(w.E):
            np.testing.assert_array_equal(allv[t, e], orc.expert_row(w, inp, e, X[t]))


def test_dropped_slot_contributes_nothing():
    w = _cfg(T=30, d=8, E=3, k=1, F=16, drop_tokens=True, capacity_factor=1.0, min_capacity=1)
    inp = wl.make_inputs(w)
    inp["b_router"] = np.array([5.0, 0.0, 0.0], np.float32)     # most tokens want expert 0
    ref = orc.layer(w, inp)
    dropped = np.nonzero(ref["inv"] < 0)[0]
    assert len(dropped) > 0
    np.testing.assert_array_equal(ref["out"][dropped], 0.0)    # no residual, no shared


def test_sigmoid_keys_block_matches_scalar_spec():
    g = np.random.default_rng(9)
    lg = g.standard_normal((7, 33)).astype(np.float32) * 4
    b = g.uniform(-0.1, 0.1, 33).astype(np.float32)
    keys = orc.sigmoid_keys(lg, b)
    for t in range(7):
        for e in range(33):
            assert keys[t, e] == np.float32(np.float32(orc.sigmoid32(float(lg[t, e]))) + b[e])


def test_expert_rows_parallel_equals_single_row():
    w = _cfg(T=12, d=16, E=3, k=1, F=24, activation=wl.SWIGLU, expert_bias=False, num_shared=1,
             dtype=wl.BF16)
    inp = wl.make_inputs(w)
    X = wl.bf16_to_f32(inp["x"]).astype(np.float64)
    ex = np.array([0, 2, 1, -1, 0, 2, -1, 1, 1, 0, 2, -1], np.int32)
    y = orc.expert_rows(w, inp, ex, X)
    for i, e in enumerate(ex):
        if e >= 0:
            np.testing.assert_array_equal(y[i], orc.expert_row(w, inp, e, X[i]))
    # the shared expert rows equal the layer's shared contribution (routed part removed)
    lay = orc.layer(w, inp)
    routed = np.stack([lay["gate"][t, 0] * orc.expert_row(w, inp, lay["idx"][t, 0], X[t]) for t in range(w.T)])
    shared_rows = np.nonzero(ex == -1)[0]
    np.testing.assert_allclose(lay["out"][shared_rows] - routed[shared_rows], y[shared_rows], atol=1e-12)



# ------------------------------------------------------------ hash routing
def test_hash_routing_properties():
    """Hash routing is a fixed token -> expert map with no router (the
    survey page's hash-layer digest): the same token always gets the same
    experts, choices are distinct and in range, k = E gives every expert,
    and the first choice is close to uniform over experts."""
    g = np.random.default_rng(12)
    tok = g.integers(0, 32000, 60000).astype(np.int32)
    for E, k in [(1, 1), (8, 2), (16, 16), (128, 1), (256, 8)]:
        r = orc.route_hash(len(tok), E, k, tok)
        idx = r["idx"]
        assert idx.min() >= 0 and idx.max() < E
        assert all(len(set(row)) == k for row in idx[:2000])
        np.testing.assert_allclose(r["gate"], 1.0 / k)
        # same token id -> same choices
        first = {}
        for t in range(3000):
            key = int(tok[t])
            if key in first:
                assert list(idx[t]) == first[key]
            else:
                first[key] = list(idx[t])
        if k == E:
            assert all(sorted(row) == list(range(E)) for row in idx[:500])
        if E >= 8 and k == 1:
            # uniformity over distinct ids (a repeated id repeats its expert by design)
            uniq = np.arange(100000, dtype=np.int32)
            counts = np.bincount(orc.route_hash(len(uniq), E, 1, uniq)["idx"][:, 0], minlength=E)
            expect = len(uniq) / E
            chi2 = float(((counts - expect) ** 2 / expect).sum())
            assert chi2 < E + 6 * np.sqrt(2 * E)          # ~6 sigma of a chi-square(E-1)


def test_fmix32_closed_forms():
    # fmix32 is a bijection with fmix32(0) = 0 and no other fixed structure;
    # check the zero point, injectivity on a block, and avalanche (one input
    # bit flips about half of the output bits)
    assert orc.fmix32(0) == 0
    vals = [orc.fmix32(i) for i in range(1, 20001)]
    assert len(set(vals)) == len(vals)
    flips = [bin(orc.fmix32(i) ^ orc.fmix32(i ^ 1)).count("1") for i in range(1, 2001)]
    assert 14 < float(np.mean(flips)) < 18


def test_fmix32_murmur3_test_vectors():
    """MurmurHash3_x86_32 of the empty input with seed s is fmix32(s) (no
    blocks, no tail, length 0), so the finalizer's published test vectors
    for the empty input pin it: seed 0 -> 0, seed 1 -> 0x514E28B7, seed
    0xFFFFFFFF -> 0x81F16F39 (MurmurHash3, A. Appleby, SMHasher
    verification values)."""
    assert orc.fmix32(0) == 0
    assert orc.fmix32(1) == 0x514E28B7
    assert orc.fmix32(0xFFFFFFFF) == 0x81F16F39


def _golden_stride():
    # floor(2^32 / phi) = floor(2^31 (sqrt(5) - 1)), in integers
    return ((1 << 31) * (math.isqrt(5 << 128) - (1 << 64))) >> 64


def test_hash_choices_use_the_golden_ratio_stride():
    """Choice j hashes token_id + j * floor(2^32 / phi) (mod 2^32); where the
    keys of a token do not collide, every choice is that hash mod E."""
    stride = _golden_stride()
    assert stride == 0x9E3779B9
    E, k = 64, 3
    tok = np.arange(5000, dtype=np.int32) * 7 + 3
    r = orc.route_hash(len(tok), E, k, tok)
    checked = 0
    for t, tid in enumerate(tok):
        raw = [orc.fmix32((int(tid) + j * stride) & 0xFFFFFFFF) % E for j in range(k)]
        if len(set(raw)) == k:
            assert list(r["idx"][t]) == raw
            checked += 1
    assert checked > 4000


def test_hash_collision_moves_up_cyclically():
    """A choice that an earlier choice of the same token took moves to the
    next expert up, wrapping at E."""
    stride = _golden_stride()
    E = 5
    tok = np.arange(4000, dtype=np.int32)
    r = orc.route_hash(len(tok), E, 2, tok)
    hits = wraps = 0
    for t, tid in enumerate(tok):
        a = orc.fmix32(int(tid)) % E
        b = orc.fmix32((int(tid) + stride) & 0xFFFFFFFF) % E
        assert r["idx"][t, 0] == a
        if a == b:
            assert r["idx"][t, 1] == (a + 1) % E
            hits += 1
            wraps += a == E - 1
        else:
            assert r["idx"][t, 1] == b
    assert hits > 400 and wraps > 50


def test_hash_collision_moves_to_next_free_expert():
    """With E = 2, k = 2 the second choice must be the expert the first did
    not take, whatever the hash of the second key is."""
    tok = np.arange(100, dtype=np.int32)
    r = orc.route_hash(100, 2, 2, tok)
    assert all(sorted(row) == [0, 1] for row in r["idx"])
    first = np.array([orc.fmix32(int(t)) % 2 for t in tok])
    np.testing.assert_array_equal(r["idx"][:, 0], first)



# ------------------------------------------------------------ expert-choice routing
def test_expert_choice_selection_against_sort():
    w = _cfg(T=300, E=8, k=1, capacity_factor=2.0, min_capacity=4)
    g = np.random.default_rng(21)
    lg = g.standard_normal((w.T, w.E)).astype(np.float32)
    lg[::4] = np.round(lg[::4] * 2) / 2                      # ties
    ec = orc.route_expert_choice(w, lg)
    C = ec["C"]
    assert C == int(np.ceil(300 / 8 * 2.0)) == 75
    for e in range(w.E):
        seg = ec["row_token"][e * C:(e + 1) * C]
        want = sorted(t for _, t in sorted((-float(lg[t, e]), t) for t in range(w.T))[:C])
        assert list(seg) == want                              # top-C, ties to lower index, token order
        for r, t in enumerate(seg):
            assert ec["tok_row"][t, e] == e * C + r
    assert np.all((ec["tok_row"] >= 0).sum(0) == C)           # every expert exactly C tokens
    probs = sp.softmax(lg.astype(np.float64), axis=1)
    mask = ec["tok_row"] >= 0
    np.testing.assert_allclose(ec["tok_gate"][mask], probs[mask], rtol=1e-12)
    assert np.all(ec["tok_gate"][~mask] == 0)


def test_expert_choice_ties_at_the_capacity_boundary():
    """Logits in {0, 1}: about half the tokens tie at the C-th largest
    value; the expert takes the ties with the lowest token indices (a
    stable sort of the negated logits, first C, back in token order)."""
    w = _cfg(T=301, E=6, k=1, capacity_factor=1.7, min_capacity=0)
    g = np.random.default_rng(5)
    lg = g.integers(0, 2, (w.T, w.E)).astype(np.float32)
    ec = orc.route_expert_choice(w, lg)
    C = ec["C"]
    for e in range(w.E):
        order = np.argsort(-lg[:, e], kind="stable")
        assert lg[order[C - 1], e] == lg[order[C], e]          # the boundary really is a tie
        np.testing.assert_array_equal(ec["row_token"][e * C:(e + 1) * C], np.sort(order[:C]))


def test_expert_choice_capacity_closed_forms():
    """C = min(T, max(min_capacity, ceil(T / E * capacity_factor))), on
    values where T / E * capacity_factor is not within rounding of an
    integer."""
    for T, E, cf, mc, want in [(301, 6, 1.7, 0, 86), (10, 3, 1.0, 0, 4), (10, 4, 1.5, 0, 4), (10, 4, 1.5, 5, 5),
                               (3, 1, 2.0, 0, 3), (7, 7, 1.0, 0, 1), (1000, 8, 0.01, 2, 2)]:
        w = _cfg(T=T, E=E, k=1, capacity_factor=cf, min_capacity=mc)
        assert orc.ec_capacity(w) == want, (T, E, cf, mc)


def test_expert_choice_full_capacity_is_the_dense_soft_mixture():
    """C = T: every expert takes every token, so the layer is the dense
    softmax-weighted mixture of all experts (EfficientMoE-style brute force
    with all E experts and no renormalisation)."""
    w = _cfg(T=24, d=8, E=4, k=1, F=12, capacity_factor=4.0, min_capacity=0, renormalize=False)
    inp = wl.make_inputs(w)
    lg = orc.router_logits(w, inp)
    ec = orc.route_expert_choice(w, lg)
    assert ec["C"] == w.T and np.all(ec["tok_row"] >= 0)
    out = orc.forward_tokens_ec(w, inp, ec, np.arange(w.T))
    allv, _ = orc.dense_all(w, inp, np.zeros((w.T, 1), np.int32), np.ones((w.T, 1)), None)
    probs = sp.softmax(lg.astype(np.float64), axis=1)
    np.testing.assert_allclose(out, np.einsum("te,ted->td", probs, allv), rtol=1e-12, atol=1e-13)
