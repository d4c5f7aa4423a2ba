"""Expert FFN parity on the GPU (tcgen05 grouped GEMM for bf16 layers,
CUDA cores for fp32): y_perm rows against the oracle's expert evaluation of
the same token row, fed the oracle's dispatch."""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl
from tests.gpu_util import as_f32, dev, float_check, host, weights

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[0, 1], ids=["single_cta", "cta_pair"])
def gemm_kernel(request):
    """Run the test with the single-CTA tcgen05 kernel, then with the CTA-pair
    (cta_group::2) kernel (the MOE_OPT_GEMM_PAIR option, read per launch)."""
    moe.moe_set_option(moe.MOE_OPT_GEMM_PAIR, request.param)
    yield request.param
    moe.moe_set_option(moe.MOE_OPT_GEMM_PAIR, -1)


def oracle_dispatch(w, inp):
    lg = wl.make_logits(w, ties=False)
    r = orc.route(w, lg, inp.get("sel_bias"))
    return r, orc.dispatch(w, r["idx"])


def run_expert_ffn(w, inp, d_ref, expect_flag=0):
    """y_perm rows 0 .. offsets[E]-1 of moe_expert_ffn on the oracle's
    dispatch; the device error flag must read expect_flag afterwards."""
    cfg = moe.config_for(w)
    S, d = w.T * w.k, w.d
    X = inp["x"]
    nk = int(d_ref["offsets"][-1])
    xp = np.zeros((max(S, 1), d), X.dtype)
    xp[:nk] = X[d_ref["perm"][:nk] // w.k]             # host-side gather of the rows
    W = weights(inp)
    y = torch.full((max(S, 1), d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(moe.moe_workspace_size(cfg, moe.MOE_WS_EXPERT_FFN), 1), dtype=torch.uint8, device="cuda")
    moe.moe_expert_ffn(cfg, dev(xp), dev(d_ref["offsets"]), W["w1"], W.get("b1"), W.get("w3"), W["w2"],
                       W.get("b2"), y, ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == expect_flag
    return host(y)[:nk]


def sample_rows(d_ref, n, seed=0):
    """Sampled rows incl. the first and last row of every non-empty segment."""
    off = d_ref["offsets"]
    nk = int(off[-1])
    rows = set()
    for e in range(len(off) - 1):
        if off[e + 1] > off[e]:
            rows |= {int(off[e]), int(off[e + 1]) - 1}
    g = np.random.default_rng(seed)
    if nk:
        rows |= set(g.choice(nk, size=min(n, nk), replace=False).tolist())
    return np.array(sorted(rows), np.int64)


def check_ffn(w, inp, d_ref, y_gpu, nrows, report=None):
    rows = sample_rows(d_ref, nrows)
    if len(rows) == 0:
        return
    slots = d_ref["perm"][rows]
    tok = slots // w.k
    X = as_f32(inp["x"]).astype(np.float64)
    # expert of each row from the segment it sits in
    experts = np.searchsorted(d_ref["offsets"], rows, side="right") - 1
    ref = orc.expert_rows(w, inp, experts.astype(np.int32), X[tok])
    float_check(y_gpu[rows], ref, w, f"{w.name} y_perm", report)


CASES = [("tiny_fp32", 64, 10**9), ("quickstart_bf16", 1000, 96), ("capacity_e128", 1500, 160),
         ("mixtral", 300, 24), ("deepseek_v3", 200, 64)]


@pytest.mark.parametrize("name,T,nrows", CASES)
def test_expert_ffn(name, T, nrows, gemm_kernel):
    w = wl.WORKLOADS[name].scaled(T)
    inp = wl.make_inputs(w)
    _, d_ref = oracle_dispatch(w, inp)
    y = run_expert_ffn(w, inp, d_ref)
    check_ffn(w, inp, d_ref, y, nrows)


@pytest.mark.parametrize("act", [wl.RELU, wl.GELU, wl.SWIGLU])
def test_expert_ffn_ragged_segments(act, gemm_kernel):
    """Segments of 0, 1, 127, 128, 129, 255, 256, 257, 300 and 600 rows."""
    sizes = [0, 1, 127, 128, 129, 255, 0, 256, 257, 300, 600, 64]
    E = len(sizes)
    T = sum(sizes)
    w = wl.Workload(f"rag{act}", 50 + act, T=T, d=128, E=E, k=1, F=192, activation=act, score_fn=wl.SOFTMAX,
                    dtype=wl.BF16, router_bias=False, expert_bias=act != wl.SWIGLU)
    inp = wl.make_inputs(w)
    idx = np.concatenate([np.full(s, e, np.int32) for e, s in enumerate(sizes)])[:, None]
    d_ref = orc.dispatch(w, idx)
    y = run_expert_ffn(w, inp, d_ref)
    check_ffn(w, inp, d_ref, y, 10**9)


def test_shared_ffn(gemm_kernel):
    w = wl.WORKLOADS["deepseek_v3"].scaled(300)
    inp = wl.make_inputs(w)
    cfg = moe.config_for(w)
    W = weights(inp)
    z = torch.full((w.T, w.d), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.moe_workspace_size(cfg, moe.MOE_WS_SHARED_FFN), dtype=torch.uint8, device="cuda")
    moe.moe_shared_ffn(cfg, dev(inp["x"]), W["shared_w1"], W["shared_w3"], W["shared_w2"], z, ws)
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    X = as_f32(inp["x"]).astype(np.float64)
    toks = np.array(sorted({0, 1, 127, 128, 255, w.T - 1} | set(range(3, w.T, 17))))
    ref = orc.expert_rows(w, inp, np.full(len(toks), -1, np.int32), X[toks])
    float_check(host(z)[toks], ref, w, "shared z")
