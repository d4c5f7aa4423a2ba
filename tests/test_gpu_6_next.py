"""The next rows of the scope table on the GPU: hash routing (bit-exact
against the oracle), the hash-routed layer through moe_forward_from_routing,
and the capacity variants (k > 1 with token dropping, the evaluation
capacity factor 2.0, Switch-style top-1 gating by the raw probability)."""
import math

import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl
from tests.gpu_util import dev, float_check, host, weights
from tests.test_gpu_4_layer import check_layer, run_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("E,k,T", [(1, 1, 100), (8, 2, 5000), (16, 16, 333), (128, 1, 4097), (256, 8, 2048),
                                   (1024, 16, 999)])
def test_route_hash_bit_exact(E, k, T):
    g = np.random.default_rng(E + k)
    tok = g.integers(-2**31, 2**31 - 1, T, dtype=np.int64).astype(np.int32)
    tok[: T // 3] = g.integers(0, 32000, T // 3)                 # vocabulary-sized ids too
    w = wl.Workload(f"h{E}", 70, T=T, d=64, E=E, k=k, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                    dtype=wl.BF16, router_bias=False, expert_bias=False)
    cfg = moe.config_for(w)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    gw = torch.empty(T, k, dtype=torch.float32, device="cuda")
    moe.moe_route_hash(cfg, dev(tok), idx, gw)
    torch.cuda.synchronize()
    ref = orc.route_hash(T, E, k, tok)
    np.testing.assert_array_equal(host(idx), ref["idx"])
    np.testing.assert_array_equal(host(gw), np.float32(1.0 / k))


@pytest.mark.parametrize("name,T,ntok", [("quickstart_bf16", 1500, 64), ("mixtral", 300, 10),
                                         ("deepseek_v3", 256, 12), ("tiny_fp32", 64, None)])
def test_hash_routed_layer(name, T, ntok):
    w = wl.WORKLOADS[name].scaled(T)
    inp = wl.make_inputs(w)
    tok = np.random.default_rng(T).integers(0, 32000, w.T).astype(np.int32)
    layer = moe.MoELayer(moe.config_for(w), weights(inp), dev(inp["sel_bias"]) if "sel_bias" in inp else None)
    out = host(layer.forward_hashed(dev(inp["x"]), dev(tok)))
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    ref_r = orc.route_hash(w.T, w.E, w.k, tok)
    ref_d = orc.dispatch(w, ref_r["idx"])
    for key in ("counts", "kept", "offsets"):
        np.testing.assert_array_equal(host(layer.io[key]), ref_d[key], err_msg=key)
    tokens = np.arange(w.T) if ntok is None else wl.sample_tokens(w, ntok)
    out_ref = orc.forward_tokens(w, inp, ref_r["idx"], ref_r["gate"], ref_d["inv"], tokens)
    float_check(out[tokens], out_ref, w, f"{w.name} hash out")
    st = layer.stats()
    assert math.isnan(st["aux_loss"]) and math.isnan(st["z_loss"])   # no router probabilities
    assert st["total_kept"] == int(ref_d["kept"].sum())


CAPACITY_VARIANTS = [
    # k > 1 with token dropping (rank-major priority decides who is dropped)
    dict(name="top2_drop", T=3000, E=16, k=2, capacity_factor=1.0, min_capacity=4, drop_tokens=True),
    # the evaluation capacity factor of the DeepSpeed guide
    dict(name="eval_cf2", T=3000, E=32, k=1, capacity_factor=2.0, min_capacity=4, drop_tokens=True),
    # Switch-style top-1: the gate is the raw softmax probability (no renormalisation)
    dict(name="switch_raw_prob", T=2000, E=8, k=1, renormalize=False),
    # top-2 without renormalisation and with dropping
    dict(name="top2_raw_drop", T=2500, E=8, k=2, renormalize=False, capacity_factor=1.25, drop_tokens=True),
]


@pytest.mark.parametrize("v", CAPACITY_VARIANTS, ids=lambda v: v["name"])
def test_capacity_and_gating_variants(v):
    kw = dict(v)
    name = kw.pop("name")
    w = wl.Workload(name, 80, d=256, F=512, activation=wl.GELU, score_fn=wl.SOFTMAX, dtype=wl.BF16,
                    router_bias=True, expert_bias=True, **kw)
    inp = wl.make_inputs(w)
    inp["b_router"] = np.random.default_rng(7).standard_normal(w.E).astype(np.float32)   # skewed load
    _, got = run_layer(w, inp)
    ref_r, ref_d, _ = check_layer(w, inp, got, wl.sample_tokens(w, 64))
    if w.drop_tokens:
        assert got["stats"]["dropped"] > 0
