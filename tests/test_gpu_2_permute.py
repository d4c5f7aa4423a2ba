"""Dispatch parity on the GPU: counts, kept, offsets, the permutation, its
inverse and the copied rows must equal the oracle's bit for bit, fed the
oracle's own top-k choices."""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl
from tests.gpu_util import dev, host

pytestmark = pytest.mark.gpu


def run_permute(w, x, idx):
    cfg = moe.config_for(w)
    T, E, k, d = w.T, w.E, w.k, w.d
    S = T * k
    xd = dev(x)
    idd = dev(np.ascontiguousarray(idx, np.int32))
    i32 = dict(dtype=torch.int32, device="cuda")
    counts = torch.full((E,), -5, **i32)
    kept = torch.full((E,), -5, **i32)
    offsets = torch.full((E + 1,), -5, **i32)
    perm = torch.full((max(S, 1),), -5, **i32)
    inv = torch.full((max(S, 1),), -5, **i32)
    xp = torch.zeros(max(S, 1), d, dtype=xd.dtype, device="cuda")
    ws = torch.empty(max(moe.moe_workspace_size(cfg, moe.MOE_WS_PERMUTE), 1), dtype=torch.uint8, device="cuda")
    moe.moe_permute(cfg, xd, idd, counts, kept, offsets, perm, inv, xp, ws)
    torch.cuda.synchronize()
    err = moe.moe_check_device_error()
    return dict(counts=host(counts), kept=host(kept), offsets=host(offsets), perm=host(perm)[:S],
                inv=host(inv)[:S], x_perm=host(xp)[:S], err=err)


def check_permute(w, x, idx, got):
    ref = orc.dispatch(w, idx)
    assert got["err"] == 0
    for key in ("counts", "kept", "offsets", "perm", "inv"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    nk = int(ref["offsets"][-1])
    X = x if w.dtype == wl.F32 else wl.bf16_to_f32(x)
    np.testing.assert_array_equal(got["x_perm"][:nk], X[ref["perm"][:nk] // w.k])
    return ref


def _oracle_idx(w):
    lg = wl.make_logits(w)
    return orc.route(w, lg, wl.make_inputs(w, with_weights=False).get("sel_bias"))["idx"]


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_permute_bit_exact_full_size(name):
    w = wl.WORKLOADS[name]
    x = wl.make_inputs(w, with_weights=False)["x"]
    idx = _oracle_idx(w)
    ref = check_permute(w, x, idx, run_permute(w, x, idx))
    if w.drop_tokens:
        assert ref["kept"].max() <= orc.capacity(w) == 80
        assert (ref["counts"] - ref["kept"]).sum() > 0    # the skewed router does drop


@pytest.mark.parametrize("case", ["one_expert_capacity", "k_equals_E", "single_token", "ragged_many_chunks",
                                  "empty_experts", "e1024_drop", "fp32_k3_drop", "two_pass_80k_slots",
                                  "chunked_160k_slots"])
def test_permute_edge_cases(case):
    g = np.random.default_rng(len(case))
    if case == "one_expert_capacity":
        w = wl.Workload(case, 40, T=5000, d=64, E=16, k=1, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.BF16, router_bias=False, expert_bias=False, drop_tokens=True,
                        capacity_factor=1.25, min_capacity=4)
        idx = np.full((w.T, 1), 3, np.int32)
    elif case == "k_equals_E":
        w = wl.Workload(case, 41, T=777, d=128, E=8, k=8, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.BF16, router_bias=False, expert_bias=False)
        idx = np.stack([g.permutation(8) for _ in range(w.T)]).astype(np.int32)
    elif case == "single_token":
        w = wl.Workload(case, 42, T=1, d=64, E=4, k=2, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.BF16, router_bias=False, expert_bias=False, drop_tokens=True,
                        capacity_factor=1.0, min_capacity=0)
        idx = np.array([[2, 0]], np.int32)
    elif case == "ragged_many_chunks":
        w = wl.Workload(case, 43, T=9999, d=64, E=37, k=3, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.BF16, router_bias=False, expert_bias=False, drop_tokens=True,
                        capacity_factor=0.9, min_capacity=4)
        pop = np.exp(g.standard_normal(w.E) * 2)
        idx = np.stack([g.choice(w.E, 3, replace=False, p=pop / pop.sum()) for _ in range(w.T)]).astype(np.int32)
    elif case == "empty_experts":
        w = wl.Workload(case, 44, T=3000, d=64, E=64, k=2, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.BF16, router_bias=False, expert_bias=False)
        idx = np.stack([g.choice([5, 9, 60], 2, replace=False) for _ in range(w.T)]).astype(np.int32)
    elif case == "e1024_drop":
        w = wl.Workload(case, 45, T=4100, d=64, E=1024, k=4, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.BF16, router_bias=False, expert_bias=False, drop_tokens=True,
                        capacity_factor=2.0, min_capacity=4)
        pop = np.exp(g.standard_normal(w.E) * 1.5)
        idx = np.stack([g.choice(w.E, 4, replace=False, p=pop / pop.sum()) for _ in range(w.T)]).astype(np.int32)
    elif case == "two_pass_80k_slots":
        # far above the one-CTA dispatch limit: 40 chunks x 64 experts, the two-launch dispatch
        w = wl.Workload(case, 48, T=40000, d=64, E=64, k=2, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.BF16, router_bias=False, expert_bias=False, drop_tokens=True,
                        capacity_factor=1.1, min_capacity=4)
        pop = np.exp(g.standard_normal(w.E))
        idx = np.stack([g.choice(w.E, 2, replace=False, p=pop / pop.sum()) for _ in range(w.T)]).astype(np.int32)
    elif case == "chunked_160k_slots":
        # a chunk table of 79 x 128 entries, above the two-launch limit: the
        # histogram, scan and rank kernels with the workspace tables
        w = wl.Workload(case, 51, T=40000, d=64, E=128, k=4, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.BF16, router_bias=False, expert_bias=False, drop_tokens=True,
                        capacity_factor=1.1, min_capacity=4)
        pop = np.exp(g.standard_normal(w.E))
        idx = np.stack([g.choice(w.E, 4, replace=False, p=pop / pop.sum()) for _ in range(w.T)]).astype(np.int32)
    else:
        w = wl.Workload(case, 46, T=2049, d=36, E=6, k=3, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                        dtype=wl.F32, router_bias=False, expert_bias=False, drop_tokens=True,
                        capacity_factor=1.0, min_capacity=4)
        idx = np.stack([g.choice(w.E, 3, replace=False) for _ in range(w.T)]).astype(np.int32)
    x = wl.make_inputs(w, with_weights=False)["x"]
    check_permute(w, x, idx, run_permute(w, x, idx))


def test_permute_empty_batch():
    w = wl.WORKLOADS["mixtral"].scaled(0)
    got = run_permute(w, np.zeros((0, w.d), np.uint16), np.zeros((0, w.k), np.int32))
    assert got["counts"].tolist() == [0] * w.E and got["offsets"].tolist() == [0] * (w.E + 1)


@pytest.mark.parametrize("T", [100, 6000], ids=["one_cta", "two_launch"])
def test_permute_flags_out_of_range_expert(T):
    """An index outside [0, E) is skipped (slot dropped) and raises the
    library's device error flag, read back as MOE_ERR_INVALID_ARG."""
    w = wl.Workload("bad_idx", 47, T=T, d=64, E=8, k=2, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                    dtype=wl.BF16, router_bias=False, expert_bias=False)
    g = np.random.default_rng(1)
    idx = np.stack([g.choice(8, 2, replace=False) for _ in range(w.T)]).astype(np.int32)
    idx[17, 1] = 8
    idx[50, 0] = -1
    x = wl.make_inputs(w, with_weights=False)["x"]
    got = run_permute(w, x, idx)
    assert got["err"] == 1
    assert got["inv"][17 * 2 + 1] == -1 and got["inv"][50 * 2] == -1
    assert moe.moe_check_device_error() == 0   # read clears the flag


@pytest.mark.parametrize("T", [1001, 5001], ids=["one_cta", "two_launch"])
def test_permute_unaligned_topk_idx(T):
    """topk_idx need not be 16-byte aligned: a view starting 4 bytes into a
    buffer gives the same dispatch."""
    w = wl.Workload("unaligned", 49, T=T, d=64, E=16, k=2, F=64, activation=wl.GELU, score_fn=wl.SOFTMAX,
                    dtype=wl.BF16, router_bias=False, expert_bias=False)
    g = np.random.default_rng(3)
    idx = np.stack([g.choice(w.E, 2, replace=False) for _ in range(w.T)]).astype(np.int32)
    x = wl.make_inputs(w, with_weights=False)["x"]
    cfg = moe.config_for(w)
    S = w.T * w.k
    buf = torch.zeros(S + 4, dtype=torch.int32, device="cuda")
    buf[1:S + 1] = torch.from_numpy(idx.reshape(-1)).cuda()
    view = buf[1:S + 1]
    assert view.data_ptr() % 16 == 4
    i32 = dict(dtype=torch.int32, device="cuda")
    outs = [torch.empty(w.E, **i32), torch.empty(w.E, **i32), torch.empty(w.E + 1, **i32),
            torch.empty(S, **i32), torch.empty(S, **i32)]
    xd = dev(x)
    xp = torch.zeros(S, w.d, dtype=xd.dtype, device="cuda")
    ws = torch.empty(moe.moe_workspace_size(cfg, moe.MOE_WS_PERMUTE), dtype=torch.uint8, device="cuda")
    moe.moe_permute(cfg, xd, view, *outs, xp, ws)
    torch.cuda.synchronize()
    got = dict(counts=host(outs[0]), kept=host(outs[1]), offsets=host(outs[2]), perm=host(outs[3]),
               inv=host(outs[4]), x_perm=host(xp), err=moe.moe_check_device_error())
    check_permute(w, x, idx, got)
