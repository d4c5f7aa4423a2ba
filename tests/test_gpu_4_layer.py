"""Whole-layer parity on the GPU through moe_forward (the call the benchmark
times): output, intermediates, statistics, the bias update, determinism and
the empty batch."""
import ctypes as C

import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl
from tests.gpu_util import as_f32, dev, float_check, host, weights
from tests.test_gpu_1_route import check_route_from_x

pytestmark = pytest.mark.gpu


def run_layer(w, inp):
    cfg = moe.config_for(w)
    layer = moe.MoELayer(cfg, weights(inp), dev(inp["sel_bias"]) if "sel_bias" in inp else None)
    out = layer.forward(dev(inp["x"]))
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    got = {k: host(v) for k, v in layer.io.items() if k != "stats"}
    got["out"] = host(out)
    got["stats"] = layer.stats()
    return layer, got


def check_layer(w, inp, got, tokens, report=None):
    """Routing from x (exact where unambiguous), dispatch, output, stats."""
    ref_r, n_near = check_route_from_x(w, inp, dict(logits=got["logits"], idx=got["topk_idx"],
                                                    w=got["topk_w"], lse=got["lse"], P=got["prob_mean"],
                                                    counts=got["counts"]))
    ref_d = orc.dispatch(w, ref_r["idx"])
    S = w.T * w.k
    if n_near == 0:
        for key in ("counts", "kept", "offsets"):
            np.testing.assert_array_equal(got[key], ref_d[key], err_msg=key)
        np.testing.assert_array_equal(got["perm"][:S], ref_d["perm"])
        np.testing.assert_array_equal(got["inv"].reshape(-1)[:S], ref_d["inv"])
        ok_tokens = tokens
    else:
        # a near-tie flipped a choice: compare tokens whose route and slots agree
        same = np.all(got["topk_idx"] == ref_r["idx"], axis=1)
        inv_g = got["inv"].reshape(w.T, w.k)
        inv_same = np.all((inv_g >= 0) == (ref_d["inv"].reshape(w.T, w.k) >= 0), axis=1)
        ok_tokens = np.array([t for t in tokens if same[t] and inv_same[t]])
    # tokens whose every slot was dropped, in a layer without residual or
    # shared expert, output exact zeros; the float bar is measured on the rows
    # the layer computes (zero rows would only deflate the RMS it uses)
    inv2 = ref_d["inv"].reshape(w.T, w.k)
    structural_zero = np.all(inv2 < 0, axis=1) & (not w.residual) & (w.num_shared == 0)
    zero_tok = np.array([t for t in ok_tokens if structural_zero[t]], dtype=np.int64)
    if len(zero_tok):
        assert np.all(got["out"][zero_tok] == 0.0)
    ok_tokens = np.array([t for t in ok_tokens if not structural_zero[t]], dtype=np.int64)
    out_ref = orc.forward_tokens(w, inp, ref_r["idx"], ref_r["gate"], ref_d["inv"], ok_tokens)
    float_check(got["out"][ok_tokens], out_ref, w, f"{w.name} out", report)
    st = orc.stats(w, ref_d["counts"], ref_d["kept"], ref_r["prob_sum"], ref_r["lse"])
    gs = got["stats"]
    if n_near == 0:
        assert gs["dropped"] == st["dropped"]
        assert gs["total_kept"] == int(ref_d["kept"].sum())
        np.testing.assert_allclose(got["f"], st["f"], rtol=1e-6)
        assert abs(gs["utilization"] - st["utilization"]) < 1e-6
        assert (gs["imbalance"] == st["imbalance"]) or abs(gs["imbalance"] - st["imbalance"]) < 1e-5 * st["imbalance"]
        assert abs(gs["drop_rate"] - st["drop_rate"]) < 1e-7
    np.testing.assert_allclose(gs["aux_loss"], st["aux"], rtol=1e-4)
    np.testing.assert_allclose(gs["z_loss"], st["z"], rtol=1e-4)
    assert gs["capacity"] == (orc.capacity(w) if w.drop_tokens else -1)
    return ref_r, ref_d, n_near


LAYER_CASES = [("tiny_fp32", 64, None), ("quickstart_bf16", 1000, 96), ("capacity_e128", 2000, 128),
               ("mixtral", 256, 12), ("deepseek_v3", 200, 24)]


@pytest.mark.parametrize("name,T,ntok", LAYER_CASES)
def test_layer_forward(name, T, ntok):
    w = wl.WORKLOADS[name].scaled(T)
    inp = wl.make_inputs(w)
    _, got = run_layer(w, inp)
    tokens = np.arange(T) if ntok is None else wl.sample_tokens(w, ntok)
    check_layer(w, inp, got, tokens)


def test_tiny_layer_against_bruteforce():
    """The fp32 Quick Start layer against the EfficientMoE brute-force form."""
    w = wl.WORKLOADS["tiny_fp32"]
    inp = wl.make_inputs(w)
    _, got = run_layer(w, inp)
    ref = orc.layer(w, inp)
    _, dense = orc.dense_all(w, inp, ref["idx"], ref["gate"], ref["inv"])
    float_check(got["out"], dense, w, "tiny vs brute force")


@pytest.mark.parametrize("name,T,ntok", LAYER_CASES)
def test_layer_deterministic(name, T, ntok):
    """Two forwards of the same layer on the same inputs, each with its own
    buffers and workspace: every output and intermediate bit-identical."""
    w = wl.WORKLOADS[name].scaled(T)
    inp = wl.make_inputs(w)
    _, a = run_layer(w, inp)
    _, b = run_layer(w, inp)
    for key in ("out", "logits", "topk_idx", "topk_w", "lse", "prob_mean", "counts", "kept", "offsets", "perm",
                "inv", "f"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=f"{name} {key}")
    assert a["stats"] == b["stats"]


def test_bias_update_bit_exact():
    w = wl.WORKLOADS["deepseek_v3"].scaled(512)
    inp = wl.make_inputs(w)
    layer, got = run_layer(w, inp)
    b0 = host(layer.sel_bias).copy()
    moe.bias_update(layer, w.bias_gamma)
    torch.cuda.synchronize()
    ref = orc.bias_update(w, got["counts"], b0, w.bias_gamma)
    np.testing.assert_array_equal(host(layer.sel_bias), ref)
    # the update moves overloaded experts down and idle ones up by exactly gamma
    mean = w.T * w.k / w.E
    d = host(layer.sel_bias) - b0
    assert np.all(d[got["counts"] > mean] < 0) and np.all(d[got["counts"] < mean] > 0)


def test_layer_empty_batch():
    w = wl.WORKLOADS["quickstart_bf16"].scaled(0)
    inp = wl.make_inputs(w)
    _, got = run_layer(w, inp)
    assert got["out"].shape == (0, w.d)
    assert got["counts"].tolist() == [0] * w.E
    assert got["stats"]["total_kept"] == 0


def test_layer_single_token_and_k_equals_E():
    w = wl.Workload("k_eq_E", 60, T=1, d=128, E=4, k=4, F=128, activation=wl.GELU, score_fn=wl.SOFTMAX,
                    dtype=wl.BF16, router_bias=True, expert_bias=True, residual=True)
    inp = wl.make_inputs(w)
    _, got = run_layer(w, inp)
    check_layer(w, inp, got, np.arange(1))


def test_layer_capacity_all_drop_but_capacity():
    """Every token prefers one expert: exactly C tokens (the first C) are
    processed by it, the rest output zero (no residual, no shared)."""
    w = wl.Workload("collapse", 61, T=600, d=128, E=8, k=1, F=128, activation=wl.RELU, score_fn=wl.SOFTMAX,
                    dtype=wl.BF16, router_bias=True, expert_bias=True, drop_tokens=True,
                    capacity_factor=1.0, min_capacity=4)
    inp = wl.make_inputs(w)
    inp["b_router"] = np.array([0, 0, 0, 40.0, 0, 0, 0, 0], np.float32)
    _, got = run_layer(w, inp)
    cap = orc.capacity(w)
    assert got["kept"].tolist() == [0, 0, 0, cap, 0, 0, 0, 0]
    assert np.all(got["out"][cap:] == 0.0)          # dropped rows: exactly zero
    check_layer(w, inp, got, np.arange(0, w.T, 3))


def test_host_batches_pipeline_matches_forward():
    """MoELayer.run_host_batches (uploads, compute and downloads overlapped on
    three streams) returns exactly what forward returns for every batch."""
    w = wl.WORKLOADS["quickstart_bf16"].scaled(1000)
    inp = wl.make_inputs(w)
    layer, got = run_layer(w, inp)
    x0 = dev(inp["x"])
    x1 = x0.flip(0).contiguous()                      # a second, different batch
    xs = [torch.empty_like(x0, device="cpu").pin_memory() for _ in range(2)]
    xs[0].copy_(x0)
    xs[1].copy_(x1)
    outs = [torch.empty(w.T, w.d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    layer.run_host_batches(xs, outs, 5)
    torch.cuda.synchronize()
    ref0 = layer.forward(x0).cpu()
    ref1 = layer.forward(x1).cpu()
    torch.cuda.synchronize()
    assert torch.equal(outs[0], ref0)                 # step 4 used batch 0
    assert torch.equal(outs[1], ref1)                 # step 3 used batch 1
    np.testing.assert_array_equal(host(ref0), got["out"])


@pytest.mark.parametrize("name,T", [("tiny_fp32", 64), ("quickstart_bf16", 1000), ("deepseek_v3", 200)])
def test_graph_replay_matches_forward(name, T):
    """MoELayer.graphed: replays of the captured forward, on new inputs
    copied into the captured x buffer, give exactly the eager forward's
    output, routing and statistics for those inputs."""
    w = wl.WORKLOADS[name].scaled(T)
    inp = wl.make_inputs(w)
    layer, first = run_layer(w, inp)
    x = dev(inp["x"])
    out = torch.empty(w.T, w.d, dtype=layer.out_dtype(), device="cuda")
    g = layer.graphed(x, out)
    torch.cuda.synchronize()
    x0 = x.clone()
    x1 = (x0.flip(0) * 0.5).contiguous()             # a second, different batch
    for xb in (x1, x0, x1):
        x.copy_(xb)
        g.replay()
        torch.cuda.synchronize()
        got_out, got_idx, got_stats = out.clone(), layer.io["topk_idx"].clone(), layer.stats()
        ref = layer.forward(xb)
        torch.cuda.synchronize()
        assert torch.equal(got_out, ref), name
        assert torch.equal(got_idx, layer.io["topk_idx"]), name
        assert got_stats == layer.stats(), name
    assert moe.moe_check_device_error() == 0
    np.testing.assert_array_equal(host(layer.forward(x0)), first["out"])


def run_steps(w, inp):
    """The layer as the separate calls of the C ABI, each with its own
    workspace: moe_route -> moe_permute -> moe_expert_ffn (-> moe_shared_ffn)
    -> moe_combine -> moe_stats (raw expert outputs, gates applied in the
    combine)."""
    cfg = moe.config_for(w)
    T, E, k, d = w.T, w.E, w.k, w.d
    S = T * k
    W = weights(inp)
    f32, i32 = dict(dtype=torch.float32, device="cuda"), dict(dtype=torch.int32, device="cuda")
    ws = lambda which: torch.empty(max(moe.moe_workspace_size(cfg, which), 1), dtype=torch.uint8, device="cuda")
    x = dev(inp["x"])
    sb = dev(inp["sel_bias"]) if "sel_bias" in inp else None
    o = dict(logits=torch.empty(T, E, **f32), topk_idx=torch.empty(T, k, **i32), topk_w=torch.empty(T, k, **f32),
             lse=torch.empty(T, **f32), prob_mean=torch.empty(E, **f32), counts=torch.empty(E, **i32),
             counts2=torch.empty(E, **i32), kept=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
             perm=torch.empty(S, **i32), inv=torch.empty(S, **i32), f=torch.empty(E, **f32))
    moe.moe_route(cfg, x, W["w_router"], W.get("b_router"), sb, o["logits"], o["topk_idx"], o["topk_w"], o["lse"],
                  o["prob_mean"], o["counts"], ws(moe.MOE_WS_ROUTE))
    x_perm = torch.empty(S, d, dtype=x.dtype, device="cuda")
    moe.moe_permute(cfg, x, o["topk_idx"], o["counts2"], o["kept"], o["offsets"], o["perm"], o["inv"], x_perm,
                    ws(moe.MOE_WS_PERMUTE))
    y = torch.empty(S, d, **f32)
    moe.moe_expert_ffn(cfg, x_perm, o["offsets"], W["w1"], W.get("b1"), W.get("w3"), W["w2"], W.get("b2"), y,
                       ws(moe.MOE_WS_EXPERT_FFN))
    z = None
    if w.num_shared:
        z = torch.empty(T, d, **f32)
        moe.moe_shared_ffn(cfg, x, W["shared_w1"], W.get("shared_w3"), W["shared_w2"], z, ws(moe.MOE_WS_SHARED_FFN))
    out = torch.empty(T, d, dtype=x.dtype, device="cuda")
    moe.moe_combine(cfg, y, o["inv"], o["topk_w"], z, x, out)
    st = torch.empty(C.sizeof(moe.MoEStats), dtype=torch.uint8, device="cuda")
    moe.moe_stats(cfg, o["counts2"], o["kept"], o["prob_mean"], o["lse"], o["f"], st)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    got = {k2: host(v) for k2, v in o.items()}
    got["out"] = host(out)
    got["stats"] = moe.stats_from_buffer(st)
    return got


@pytest.mark.parametrize("name,T,ntok", [c for c in LAYER_CASES if c[0] != "tiny_fp32"] + [("tiny_fp32", 64, None)])
def test_step_by_step_calls_match_oracle_and_forward(name, T, ntok):
    """Every call of the boundary chained by hand gives the oracle's layer,
    and the same routing, dispatch and statistics as moe_forward."""
    w = wl.WORKLOADS[name].scaled(T)
    inp = wl.make_inputs(w)
    got = run_steps(w, inp)
    np.testing.assert_array_equal(got["counts"], got["counts2"])     # router and dispatch agree
    tokens = np.arange(T) if ntok is None else wl.sample_tokens(w, ntok)
    check_layer(w, inp, got, tokens)
    _, fwd = run_layer(w, inp)
    for key in ("logits", "topk_idx", "topk_w", "lse", "counts", "kept", "offsets", "perm", "inv", "f"):
        np.testing.assert_array_equal(got[key], fwd[key], err_msg=key)
    assert got["stats"]["total_kept"] == fwd["stats"]["total_kept"]
    # the two combines add the same terms in a different fp32 order
    float_check(got["out"], fwd["out"], w, f"{name} steps vs forward")
