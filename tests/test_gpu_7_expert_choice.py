"""Expert-choice routing on the GPU: the selection is compared bit for bit
with the oracle fed the same fp32 logits (ties, signed zeros, batches above
the shared-memory key cache, one token, an empty batch), the gates to fp32
rounding, and the whole layer through moe_forward_expert_choice against the
oracle's expert-choice layer."""
import dataclasses

import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl
from tests.gpu_util import dev, float_check, host, weights

pytestmark = pytest.mark.gpu


def _w(T, E, cf, min_capacity=0, dtype=wl.F32, d=64):
    return wl.Workload("ec", 70, T=T, d=d, E=E, k=1, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                       dtype=dtype, router_bias=False, expert_bias=False, capacity_factor=cf,
                       min_capacity=min_capacity)


def run_select(w, logits):
    cfg = moe.config_for(w)
    C = moe.moe_ec_capacity(cfg)
    assert C == orc.ec_capacity(w)
    T, E = w.T, w.E
    i32 = dict(dtype=torch.int32, device="cuda")
    row_token = torch.full((max(E * C, 1),), -7, **i32)
    tok_row = torch.full((max(T, 1), E), -7, **i32)
    tok_gate = torch.full((max(T, 1), E), -7.0, dtype=torch.float32, device="cuda")
    offsets = torch.full((E + 1,), -7, **i32)
    lg = dev(np.ascontiguousarray(logits, np.float32)) if T else torch.empty(0, E, device="cuda")
    moe.moe_route_expert_choice(cfg, lg, row_token, tok_row, tok_gate, offsets)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    return dict(C=C, row_token=host(row_token)[:E * C], tok_row=host(tok_row)[:T], tok_gate=host(tok_gate)[:T],
                offsets=host(offsets))


def check_select(w, logits, got):
    ref = orc.route_expert_choice(w, logits)
    C = ref["C"]
    np.testing.assert_array_equal(got["row_token"], ref["row_token"])
    np.testing.assert_array_equal(got["tok_row"], ref["tok_row"])
    np.testing.assert_array_equal(got["offsets"], np.arange(w.E + 1) * C)
    np.testing.assert_allclose(got["tok_gate"], ref["tok_gate"], rtol=2e-6, atol=1e-30)
    # every expert holds exactly C tokens, each once, in token order
    rt = got["row_token"].reshape(w.E, C)
    assert np.all(np.diff(rt, axis=1) > 0)
    return ref


@pytest.mark.parametrize("T,E,cf,kind", [(1000, 8, 2.0, "normal"), (4097, 64, 1.0, "normal"),
                                         (3000, 16, 2.0, "ties"), (2500, 5, 1.5, "signed_zero"),
                                         (50000, 4, 0.08, "normal"), (50000, 3, 0.06, "ties"),
                                         (1, 4, 1.0, "normal"), (777, 256, 3.0, "normal"),
                                         (300, 1024, 2.0, "normal"), (100, 4, 100.0, "normal")])
def test_expert_choice_selection_bit_exact(T, E, cf, kind):
    g = np.random.default_rng(T * 31 + E)
    if kind == "ties":
        lg = g.integers(0, 4, (T, E)).astype(np.float32)
    elif kind == "signed_zero":
        lg = g.integers(-1, 2, (T, E)).astype(np.float32)
        lg[(lg == 0) & (g.random((T, E)) < 0.5)] = -0.0
    else:
        lg = (g.standard_normal((T, E)) * 2).astype(np.float32)
    w = _w(T, E, cf)
    check_select(w, lg, run_select(w, lg))


def test_expert_choice_empty_batch():
    w = _w(0, 8, 2.0)
    got = run_select(w, np.zeros((0, 8), np.float32))
    assert got["C"] == 0 and got["offsets"].tolist() == [0] * 9


def test_expert_choice_rejects_bad_capacity_factor():
    cfg = moe.config_for(_w(10, 4, 1.0))
    cfg.capacity_factor = 0.0
    with pytest.raises(moe.MoEError):
        moe.moe_ec_capacity(cfg)


def _logit_bound(w, inp, got_logits):
    ref_lg = orc.router_logits(w, inp)
    X = inp["x"] if w.dtype == wl.F32 else wl.bf16_to_f32(inp["x"])
    W = inp["w_router"] if w.dtype == wl.F32 else wl.bf16_to_f32(inp["w_router"])
    absdot = np.abs(X).astype(np.float64) @ np.abs(W).astype(np.float64).T
    err = np.abs(got_logits.astype(np.float64) - ref_lg.astype(np.float64))
    bound = (w.d / 32 + 32) * 2.0 ** -24 * absdot + 2.0 ** -23 * np.abs(ref_lg)
    assert np.all(err <= bound), f"logit error {err.max():.3e} above bound"
    return ref_lg, 2.0 * float(err.max()) + 1e-30


EC_LAYERS = [("tiny_fp32", 64, None, None), ("quickstart_bf16", 1000, 96, None), ("capacity_e128", 2000, 96, None),
             ("mixtral", 512, 12, None), ("deepseek_v3", 256, 16, 8.0)]


@pytest.mark.parametrize("name,T,ntok,cf", EC_LAYERS)
def test_expert_choice_layer(name, T, ntok, cf):
    base = wl.WORKLOADS[name].scaled(T)
    w = dataclasses.replace(base, capacity_factor=float(cf if cf else base.k))
    inp = wl.make_inputs(w)
    layer = moe.ExpertChoiceLayer(moe.config_for(w), weights(inp))
    out = layer.forward(dev(inp["x"]))
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    got = {k: host(v) for k, v in layer.io.items()}
    got_out = host(out)
    ref_lg, margin = _logit_bound(w, inp, got["logits"])
    # the selection, from the layer's own fp32 logits, is exact
    C = layer.capacity
    sel = dict(row_token=got["row_token"][:w.E * C], tok_row=got["tok_row"], tok_gate=got["tok_gate"],
               offsets=got["offsets"])
    ec = check_select(w, got["logits"], sel)
    # and valid against the oracle's logits up to the logit error
    for e in range(w.E):
        chosen = np.zeros(w.T, bool)
        chosen[ec["row_token"][e * C:(e + 1) * C]] = True
        if chosen.all():
            continue
        assert ref_lg[chosen, e].min() >= ref_lg[~chosen, e].max() - margin, e
    tokens = np.arange(w.T) if ntok is None else wl.sample_tokens(w, ntok)
    unchosen = np.all(ec["tok_row"] < 0, axis=1)
    zero = unchosen & (not w.residual) & (w.num_shared == 0)
    zt = tokens[zero[tokens]]
    if len(zt):
        assert np.all(got_out[zt] == 0.0)
    tokens = tokens[~zero[tokens]]
    out_ref = orc.forward_tokens_ec(w, inp, ec, tokens)
    float_check(got_out[tokens], out_ref, w, f"{name} expert choice out", out_rounding=True)


def test_expert_choice_layer_full_capacity_is_dense_soft_mixture():
    """C = T: every expert takes every token, so the layer is the dense
    softmax-weighted mixture of all experts (brute force)."""
    w = dataclasses.replace(wl.WORKLOADS["tiny_fp32"], capacity_factor=1e4)
    inp = wl.make_inputs(w)
    layer = moe.ExpertChoiceLayer(moe.config_for(w), weights(inp))
    assert layer.capacity == w.T
    out = host(layer.forward(dev(inp["x"])))
    lg = orc.router_logits(w, inp).astype(np.float64)
    p = np.exp(lg - lg.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    wk = dataclasses.replace(w, k=w.E)
    idx = np.tile(np.arange(w.E, dtype=np.int32), (w.T, 1))
    _, dense = orc.dense_all(wk, inp, idx, p, None)
    float_check(out, dense, w, "expert choice C=T vs dense mixture")


def test_expert_choice_layer_empty_batch():
    w = dataclasses.replace(wl.WORKLOADS["quickstart_bf16"].scaled(0), capacity_factor=2.0)
    inp = wl.make_inputs(w)
    layer = moe.ExpertChoiceLayer(moe.config_for(w), weights(inp))
    out = layer.forward(dev(inp["x"]))
    torch.cuda.synchronize()
    assert out.shape == (0, w.d) and moe.moe_check_device_error() == 0
