"""moe_permute_noalloc: the dispatch for callers that cannot allocate device
memory (no workspace; its scratch is a fixed array inside the library).

Two calls in a row with different layers, each compared with moe_permute
(which uses a caller workspace) on the same inputs: counts, kept, offsets,
the permutation, its inverse and the copied rows must be identical.  The
second call runs on scratch that still holds the first call's tables.
This file is collected last, and passes alone in a fresh process too."""
import numpy as np
import pytest
import torch

import sparse_mixture_experts_60_b300 as moe
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


def test_noalloc_permute_matches_workspace_permute_on_two_calls():
    first = wl.WORKLOADS["capacity_e128"].scaled(6000)           # E=128, k=1, token dropping
    second = wl.WORKLOADS["deepseek_v3"].scaled(2500)            # E=256, k=8, different table sizes
    for w, seed in ((first, 1), (second, 2)):
        x, idx = _case(w, seed)
        a, b = _run_both(w, x, idx)
        for key in ("counts", "kept", "offsets", "perm", "inv"):
            assert torch.equal(a[key], b[key]), (w.name, key)
        nk = int(a["offsets"][-1].item())
        assert torch.equal(a["x_perm"][:nk], b["x_perm"][:nk]), w.name
        if w.drop_tokens:
            assert int((a["counts"] - a["kept"]).sum().item()) > 0      # the first call really dropped


def test_noalloc_permute_rejects_layers_beyond_its_scratch():
    w = wl.WORKLOADS["deepseek_v3"].scaled(70000)    # ceil(560000/2048) * 256 > 65536
    cfg = moe.config_for(w)
    with pytest.raises(moe.MoEError, match="static scratch limit"):
        moe.moe_permute_noalloc(cfg, 16, 16, 16, 16, 16, 16, 16, 16)
