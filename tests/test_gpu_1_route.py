"""Router parity on the GPU: moe_route_from_logits (bit-exact integers from
the same fp32 logits) and moe_route (logits from x within the fp32
accumulation bound; integer choices exact wherever the key gap exceeds the
measured logit error, valid otherwise)."""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl
from tests.gpu_util import dev, host, keys_of, topk_valid

pytestmark = pytest.mark.gpu

NAMES = list(wl.WORKLOADS)


def _run_from_logits(w, logits, sel_bias):
    cfg = moe.config_for(w)
    T, E, k = w.T, w.E, w.k
    lg = dev(logits)
    sb = dev(sel_bias) if sel_bias is not None else None
    idx = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    tw = torch.empty(T, k, dtype=torch.float32, device="cuda")
    lse = torch.empty(T, dtype=torch.float32, device="cuda")
    P = torch.empty(E, dtype=torch.float32, device="cuda")
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(moe.moe_workspace_size(cfg, moe.MOE_WS_ROUTE), 1), dtype=torch.uint8, device="cuda")
    moe.moe_route_from_logits(cfg, lg, sb, idx, tw, lse, P, cnt, ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    return dict(idx=host(idx), w=host(tw), lse=host(lse), P=host(P), counts=host(cnt))


def _check_route_exact(w, logits, sel_bias, got):
    ref = orc.route(w, logits, sel_bias)
    np.testing.assert_array_equal(got["idx"], ref["idx"])
    np.testing.assert_array_equal(got["counts"], np.bincount(ref["idx"].reshape(-1), minlength=w.E))
    np.testing.assert_allclose(got["w"], ref["gate"], rtol=0, atol=2e-6)
    np.testing.assert_allclose(got["lse"], ref["lse"], rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(got["P"], ref["prob_sum"] / w.T, rtol=2e-5, atol=1e-7)


@pytest.mark.parametrize("name", NAMES)
def test_route_from_logits_bit_exact(name):
    w = wl.WORKLOADS[name]
    lg = wl.make_logits(w, ties=True)
    sb = wl.make_inputs(w, with_weights=False).get("sel_bias")
    _check_route_exact(w, lg, sb, _run_from_logits(w, lg, sb))


@pytest.mark.parametrize("E,k,score,renorm,T", [
    (1, 1, wl.SOFTMAX, True, 77), (4, 4, wl.SOFTMAX, True, 333), (8, 1, wl.SOFTMAX, False, 1000),
    (16, 3, wl.SIGMOID, True, 1001), (24, 5, wl.SOFTMAX, False, 257), (32, 8, wl.SIGMOID, False, 999),
    (48, 2, wl.SOFTMAX, True, 1234), (128, 16, wl.SIGMOID, True, 515), (300, 6, wl.SOFTMAX, True, 100),
    (1024, 16, wl.SIGMOID, True, 70), (1024, 2, wl.SOFTMAX, True, 33), (64, 64 // 4, wl.SOFTMAX, True, 1),
])
def test_route_from_logits_shapes(E, k, score, renorm, T):
    w = wl.Workload(f"r{E}_{k}", 20 + E % 7, T=T, d=64, E=E, k=k, F=64, activation=wl.GELU,
                    score_fn=score, dtype=wl.BF16, router_bias=False, expert_bias=False,
                    renormalize=renorm)
    g = np.random.default_rng(E * 1000 + k)
    lg = g.standard_normal((T, E)).astype(np.float32)
    lg[::3] = np.round(lg[::3] * 2) / 2          # exact ties
    lg[1::11] = 0.0                              # whole rows tied
    sb = g.uniform(-0.1, 0.1, E).astype(np.float32) if score == wl.SIGMOID else None
    _check_route_exact(w, lg, sb, _run_from_logits(w, lg, sb))


def test_route_empty_batch():
    w = wl.WORKLOADS["quickstart_bf16"].scaled(0)
    got = _run_from_logits(w, np.zeros((0, w.E), np.float32), None)
    assert got["counts"].tolist() == [0] * w.E and np.all(got["P"] == 0)


def _route_from_x(w, inp):
    cfg = moe.config_for(w)
    T, E, k = w.T, w.E, w.k
    x = dev(inp["x"])
    wr = dev(inp["w_router"])
    br = dev(inp["b_router"]) if "b_router" in inp else None
    sb = dev(inp["sel_bias"]) if "sel_bias" in inp else None
    logits = torch.empty(T, E, dtype=torch.float32, device="cuda")
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    tw = torch.empty(T, k, dtype=torch.float32, device="cuda")
    lse = torch.empty(T, dtype=torch.float32, device="cuda")
    P = torch.empty(E, dtype=torch.float32, device="cuda")
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(moe.moe_workspace_size(cfg, moe.MOE_WS_ROUTE), 1), dtype=torch.uint8, device="cuda")
    moe.moe_route(cfg, x, wr, br, sb, logits, idx, tw, lse, P, cnt, ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    return dict(logits=host(logits), idx=host(idx), w=host(tw), lse=host(lse), P=host(P), counts=host(cnt))


def check_route_from_x(w, inp, got, report=None):
    """Logits within the fp32 accumulation bound; choices exact where the
    oracle's key gap exceeds twice the measured logit error."""
    ref_lg = orc.router_logits(w, inp)
    X = inp["x"] if w.dtype == wl.F32 else wl.bf16_to_f32(inp["x"])
    W = inp["w_router"] if w.dtype == wl.F32 else wl.bf16_to_f32(inp["w_router"])
    absdot = np.abs(X).astype(np.float64) @ np.abs(W).astype(np.float64).T
    err = np.abs(got["logits"].astype(np.float64) - ref_lg.astype(np.float64))
    # fp32 sum of d products: |err| <= (d/32 + 32) * 2^-24 * sum|x w| covers a
    # per-lane sequential sum plus a tree, and any tensor-core order
    bound = (w.d / 32 + 32) * 2.0 ** -24 * absdot + 2.0 ** -23 * np.abs(ref_lg)
    assert np.all(err <= bound), f"logit error {err.max():.3e} above bound"
    margin = 2.0 * float(err.max()) + 1e-30
    sb = inp.get("sel_bias")
    ref = orc.route(w, ref_lg, sb)
    keys = keys_of(w, ref_lg, sb)
    srt = -np.sort(-keys, axis=1)
    k = w.k
    # set boundary: k-th vs (k+1)-th key; order: every adjacent gap in the top k (+1)
    set_gap = srt[:, k - 1] - (srt[:, k] if k < w.E else -np.inf)
    ext = np.concatenate([srt[:, :k], (srt[:, k:k + 1] if k < w.E else np.full((w.T, 1), -np.inf))], axis=1)
    order_gap = np.min(ext[:, :-1] - ext[:, 1:], axis=1)
    clear = order_gap > margin
    set_clear = set_gap > margin
    np.testing.assert_array_equal(got["idx"][clear], ref["idx"][clear])
    for t in np.nonzero(~clear)[0]:
        sel = got["idx"][t]
        assert len(set(sel)) == k
        if set_clear[t]:
            assert sorted(sel) == sorted(ref["idx"][t]), t
        assert topk_valid(sel, keys[t], margin), t
        ks = keys[t][sel]
        assert np.all(ks[:-1] >= ks[1:] - margin), t          # descending within the margin
    np.testing.assert_array_equal(got["counts"], np.bincount(got["idx"].reshape(-1), minlength=w.E))
    # gates / lse / P from the GPU's own logits within fp32 rounding of the oracle's
    np.testing.assert_allclose(got["lse"][clear], ref["lse"][clear], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(got["w"][clear], ref["gate"][clear], atol=1e-4)
    np.testing.assert_allclose(got["P"], ref["prob_sum"] / max(w.T, 1), rtol=1e-4, atol=1e-6)
    if report is not None:
        report.append((w.name, float(err.max()), int((~clear).sum())))
    return ref, int((~clear).sum())


@pytest.mark.parametrize("name,T", [("tiny_fp32", 64), ("quickstart_bf16", 1000), ("capacity_e128", 1000),
                                    ("mixtral", 700), ("deepseek_v3", 300)])
def test_route_from_x(name, T):
    w = wl.WORKLOADS[name].scaled(T)
    inp = wl.make_inputs(w, with_weights=False)
    check_route_from_x(w, inp, _route_from_x(w, inp))


@pytest.mark.parametrize("E,dtype", [(40, wl.BF16), (64, wl.F32), (96, wl.BF16), (33, wl.F32)])
def test_route_from_x_other_paths(E, dtype):
    """Router logits on the CUDA-core tile kernel (fp32, or E not a multiple
    of 32) and on the tensor cores with N = 96."""
    w = wl.Workload(f"rx{E}", 30 + E % 5, T=333, d=128, E=E, k=2, F=64, activation=wl.GELU,
                    score_fn=wl.SOFTMAX, dtype=dtype, router_bias=True, expert_bias=False)
    inp = wl.make_inputs(w, with_weights=False)
    check_route_from_x(w, inp, _route_from_x(w, inp))


@pytest.mark.parametrize("E,k,score,renorm,bias,T", [
    (5, 2, wl.SOFTMAX, 1, True, 333), (8, 1, wl.SOFTMAX, 0, False, 4097), (13, 3, wl.SIGMOID, 1, True, 1000),
    (16, 4, wl.SOFTMAX, 1, False, 129), (24, 6, wl.SIGMOID, 1, False, 777), (32, 8, wl.SOFTMAX, 0, True, 2048),
    (32, 16, wl.SIGMOID, 0, True, 95)])
def test_route_from_x_fused_gemm_epilogue(E, k, score, renorm, bias, T):
    """bf16 with E <= 32: the router GEMM routes in its epilogue (one thread
    per token, expert bound 8 / 16 / 32), including its per-block partials."""
    w = wl.Workload(f"rf{E}_{k}", 50 + E, T=T, d=256, E=E, k=k, F=64, activation=wl.GELU, score_fn=score,
                    dtype=wl.BF16, router_bias=bias, expert_bias=False, renormalize=renorm)
    inp = wl.make_inputs(w, with_weights=False)
    check_route_from_x(w, inp, _route_from_x(w, inp))
