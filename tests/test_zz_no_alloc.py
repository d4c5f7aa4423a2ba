"""moe_permute_noalloc: the dispatch for callers that cannot allocate device
memory (no workspace; its scratch is a fixed array inside the library).

Two calls in a row with different layers.  Each is compared with the
oracle's dispatch (counts, kept, offsets, the permutation and its inverse
bit-exact, every copied row equal to its token's row of x) and with
moe_permute, which uses a caller workspace, on the same inputs.  The second
call runs on scratch that still holds the first call's tables.  A further
call must leave the device's free memory unchanged (nothing allocated), and
a layer beyond the scratch limit is refused before anything is launched.
This file is collected last, and passes alone in a fresh process too."""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
from oracle import oracle as orc
from sparse_mixture_experts_60_b300 import workloads as wl

pytestmark = pytest.mark.gpu


def _dev(a):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def _buffers(w, like):
    S = w.T * w.k
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(counts=torch.full((w.E,), -3, **i32), kept=torch.full((w.E,), -3, **i32),
                offsets=torch.full((w.E + 1,), -3, **i32), perm=torch.full((S,), -3, **i32),
                inv=torch.full((S,), -3, **i32),
                x_perm=torch.zeros(S, w.d, dtype=like.dtype, device="cuda"))


def _case(w, seed):
    g = np.random.default_rng(seed)
    pop = np.exp(g.standard_normal(w.E))
    idx = np.stack([g.choice(w.E, w.k, replace=False, p=pop / pop.sum()) for _ in range(w.T)])
    x = wl.make_inputs(w, with_weights=False)["x"]
    return _dev(x), _dev(idx.astype(np.int32))


def _run_both(w, x, idx):
    cfg = moe.config_for(w)
    a = _buffers(w, x)
    ws = torch.empty(moe.moe_workspace_size(cfg, moe.MOE_WS_PERMUTE), dtype=torch.uint8, device="cuda")
    moe.moe_permute(cfg, x, idx, a["counts"], a["kept"], a["offsets"], a["perm"], a["inv"], a["x_perm"], ws)
    b = _buffers(w, x)
    moe.moe_permute_noalloc(cfg, x, idx, b["counts"], b["kept"], b["offsets"], b["perm"], b["inv"],
                            b["x_perm"])
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    return a, b


def _host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def test_noalloc_permute_matches_oracle_and_workspace_permute_on_two_calls():
    first = wl.WORKLOADS["capacity_e128"].scaled(6000)           # E=128, k=1, token dropping
    second = wl.WORKLOADS["deepseek_v3"].scaled(2500)            # E=256, k=8, different table sizes
    for w, seed in ((first, 1), (second, 2)):
        x, idx = _case(w, seed)
        a, b = _run_both(w, x, idx)
        ref = orc.dispatch(w, _host(idx))
        S = w.T * w.k
        for key in ("counts", "kept", "offsets"):
            np.testing.assert_array_equal(_host(b[key]), ref[key], err_msg=f"{w.name} {key}")
        np.testing.assert_array_equal(_host(b["perm"])[:S], ref["perm"], err_msg=w.name)
        np.testing.assert_array_equal(_host(b["inv"])[:S], ref["inv"], err_msg=w.name)
        for key in ("counts", "kept", "offsets", "perm", "inv"):
            assert torch.equal(a[key], b[key]), (w.name, key)
        nk = int(ref["offsets"][-1])
        rows = _host(b["x_perm"])[:nk]
        np.testing.assert_array_equal(rows, _host(x)[ref["perm"][:nk] // w.k], err_msg=w.name)
        assert torch.equal(a["x_perm"][:nk], b["x_perm"][:nk]), w.name
        if w.drop_tokens:
            assert int((ref["counts"] - ref["kept"]).sum()) > 0        # the first call really dropped


def test_noalloc_permute_allocates_nothing():
    w = wl.WORKLOADS["mixtral"].scaled(3000)
    x, idx = _case(w, 3)
    cfg = moe.config_for(w)
    b = _buffers(w, x)
    args = (cfg, x, idx, b["counts"], b["kept"], b["offsets"], b["perm"], b["inv"], b["x_perm"])
    moe.moe_permute_noalloc(*args)                  # first call on the device: the one-time set-up
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        moe.moe_permute_noalloc(*args)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert moe.moe_check_device_error() == 0


def test_noalloc_permute_rejects_layers_beyond_its_scratch():
    # ceil(132000 / 2048) * 1024 = 66560 > 65536 table entries; every buffer
    # is a real device tensor of the layer's full size (small at d = 64)
    w = wl.Workload("beyond_scratch", 70, T=16500, d=64, E=1024, k=8, F=64, activation=wl.RELU,
                    score_fn=wl.SOFTMAX, dtype=wl.BF16, router_bias=False, expert_bias=False)
    x, idx = _case(w, 4)
    cfg = moe.config_for(w)
    b = _buffers(w, x)
    with pytest.raises(moe.MoEError, match="static scratch limit"):
        moe.moe_permute_noalloc(cfg, x, idx, b["counts"], b["kept"], b["offsets"], b["perm"], b["inv"],
                                b["x_perm"])
    torch.cuda.synchronize()
    assert int(b["counts"][0].item()) == -3          # refused before any launch: outputs untouched
    # one slot fewer per chunk table row fits: ceil(131072 / 2048) * 1024 = 65536
    w2 = w.with_(T=16384, name="at_scratch_limit")
    x2, idx2 = _case(w2, 5)
    b2 = _buffers(w2, x2)
    moe.moe_permute_noalloc(moe.config_for(w2), x2, idx2, b2["counts"], b2["kept"], b2["offsets"], b2["perm"],
                            b2["inv"], b2["x_perm"])
    torch.cuda.synchronize()
    assert moe.moe_check_device_error() == 0
    ref = orc.dispatch(w2, _host(idx2))
    np.testing.assert_array_equal(_host(b2["inv"]), ref["inv"])
