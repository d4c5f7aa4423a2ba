"""The C-ABI library: it builds, loads without a GPU, exports every entry
point the header declares, sizes workspaces, and rejects bad arguments on
the host before launching anything.  No test here needs a GPU."""
import ctypes as C
import os
import re
import subprocess

import pytest

import sparse_mixture_experts_60_b300 as moe
from sparse_mixture_experts_60_b300 import _lib, build as mbuild
from sparse_mixture_experts_60_b300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_b300.h")


@pytest.fixture(scope="module")
def L():
    mbuild.build()
    return _lib.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 13
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (moe_[a-z_]+)$", out, flags=re.M))
    assert set(names) <= exported, set(names) - exported
    for n in names:
        assert hasattr(L, n)
    assert L.moe_version() == 1


def test_library_does_not_link_the_driver():
    out = subprocess.run(["ldd", _lib.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_struct_layouts_match_header(tmp_path):
    """sizeof and field offsets of every ABI struct, from the header compiled
    by the host C compiler, equal the ctypes mirrors of the binding."""
    structs = {"moe_config_t": _lib.MoEConfig, "moe_stats_t": _lib.MoEStats, "moe_weights_t": _lib.MoEWeights,
               "moe_forward_io_t": _lib.MoEForwardIO, "moe_ec_io_t": _lib.MoEECIO, "moe_saved_t": _lib.MoESaved,
               "moe_grads_t": _lib.MoEGrads, "moe_backward_opts_t": _lib.MoEBackwardOpts}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "moe_b300.h"', "int main(void) {"]
    for cname, py in structs.items():
        lines.append(f'printf("{cname} %zu\\n", sizeof({cname}));')
        for fname, _ in py._fields_:
            lines.append(f'printf("{cname}.{fname} %zu\\n", offsetof({cname}, {fname}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.splitlines())
    for cname, py in structs.items():
        assert int(got[cname]) == C.sizeof(py), cname
        for fname, _ in py._fields_:
            assert int(got[f"{cname}.{fname}"]) == getattr(py, fname).offset, (cname, fname)


def _ws_expect(w):
    """Workspace bytes recomputed from the layout rules (256-byte aligned regions)."""
    a = lambda n: (n + 255) // 256 * 256
    T, E, k, d, F = w.T, w.E, w.k, w.d, w.F
    S = T * k
    eb = 4 if w.dtype == wl.F32 else 2
    nblk = -(-T // 32)
    nch = -(-S // 2048)
    route = 2 * a(nblk * E * 4) + a(nblk * 4)
    perm = 2 * a(max(nch * E, 8192) * 4) + a(S * 4)
    ffn = a(S * F * eb)
    shared = a(T * F * eb) if w.num_shared else 0
    fwd = route + perm + ffn + shared + a(S * d * eb) + a(S * d * 4) + (a(T * d * 4) if w.num_shared else 0)
    fwd += a(T * E * 4) + 4 * a(S * 4) + a(T * 4) + 4 * a(E * 4) + a((E + 1) * 4) + a(32)
    return dict(route=route, perm=perm, ffn=ffn, shared=shared, fwd=fwd)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_workspace_sizes(L, name):
    w = wl.WORKLOADS[name]
    cfg = moe.config_for(w)
    exp = _ws_expect(w)
    assert moe.moe_workspace_size(cfg, moe.MOE_WS_ROUTE) == exp["route"]
    assert moe.moe_workspace_size(cfg, moe.MOE_WS_PERMUTE) == exp["perm"]
    assert moe.moe_workspace_size(cfg, moe.MOE_WS_EXPERT_FFN) == exp["ffn"]
    assert moe.moe_workspace_size(cfg, moe.MOE_WS_SHARED_FFN) == exp["shared"]
    assert moe.moe_workspace_size(cfg, moe.MOE_WS_FORWARD) == exp["fwd"]
    # the forward's workspace covers every single call
    assert exp["fwd"] >= max(exp["route"], exp["perm"], exp["ffn"], exp["shared"])


def _status(fn, *args):
    return fn(*args)


BAD_CFGS = [
    (dict(num_experts=0), 1), (dict(num_experts=1025), 1), (dict(top_k=0), 1), (dict(top_k=9), 1),
    (dict(top_k=17, num_experts=32), 1), (dict(num_tokens=-1), 1), (dict(score_fn=2), 1),
    (dict(activation=3), 1), (dict(dtype=2), 1), (dict(num_shared=2), 2),
    (dict(drop_tokens=1, capacity_factor=0.0), 1), (dict(min_capacity=-1), 1),
    (dict(d_model=1000), 2), (dict(d_ff=100), 2), (dict(num_tokens=2**31), 2),
]


@pytest.mark.parametrize("patch,code", BAD_CFGS)
def test_bad_config_rejected_on_host(L, patch, code):
    base = dict(num_tokens=64, d_model=1024, num_experts=8, top_k=2, d_ff=4096)
    kw = {**base, **{k: v for k, v in patch.items() if k in base}}
    cfg = moe.make_config(**kw)
    for k, v in patch.items():
        setattr(cfg, k, v)
    n = C.c_size_t(0)
    assert L.moe_workspace_size(C.byref(cfg), 0, C.byref(n)) == code
    assert len(_lib.last_error()) > 0
    with pytest.raises(moe.MoEError):
        moe.moe_workspace_size(cfg)


def test_null_and_alignment_rejected_before_launch(L):
    cfg = moe.make_config(64, 1024, 8, 2, 4096)
    P = 0x10000  # never dereferenced: validation fails first
    # null x
    st = L.moe_route(C.byref(cfg), None, P, None, None, P, P, P, P, P, P, P, 1 << 30, None)
    assert st == 1 and "x" in _lib.last_error()
    # misaligned x
    st = L.moe_route(C.byref(cfg), P + 2, P, None, None, P, P, P, P, P, P, P, 1 << 30, None)
    assert st == 3
    # sigmoid scoring without a selection bias
    cfg2 = moe.make_config(64, 1024, 8, 2, 4096, score_fn=moe.SIGMOID)
    st = L.moe_route(C.byref(cfg2), P, P, None, None, P, P, P, P, P, P, P, 1 << 30, None)
    assert st == 1 and "sel_bias" in _lib.last_error()
    # workspace too small
    need = moe.moe_workspace_size(cfg, moe.MOE_WS_ROUTE)
    st = L.moe_route(C.byref(cfg), P, P, None, None, P, P, P, P, P, P, P, need - 1, None)
    assert st == 4
    # SwiGLU without w3
    cfg3 = moe.make_config(64, 1024, 8, 2, 4096, activation=moe.SWIGLU)
    st = L.moe_expert_ffn(C.byref(cfg3), P, P, P, None, None, P, None, P, P, 1 << 40, None)
    assert st == 1 and "w3" in _lib.last_error()
    # shared FFN on a layer without a shared expert
    st = L.moe_shared_ffn(C.byref(cfg), P, P, P, P, P, P, 1 << 40, None)
    assert st == 1
    # residual without x
    cfg4 = moe.make_config(64, 1024, 8, 2, 4096, residual=True)
    st = L.moe_combine(C.byref(cfg4), P, P, P, None, None, P, None)
    assert st == 1
    # forward with a null weight struct
    st = L.moe_forward(C.byref(cfg), None, P, None, P, None, P, 1 << 40, None)
    assert st == 1
    # non-finite gamma
    st = L.moe_bias_update(C.byref(cfg), P, P, float("nan"), None)
    assert st == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.lib()


def test_c_program_links_and_calls_the_host_entry_points(L, tmp_path):
    """A plain C program compiled against the header and linked with the
    library (no Python, no GPU) sizes workspaces, gets the expert-choice
    capacity, and reads back the host-side error of a bad call."""
    src = tmp_path / "user.c"
    src.write_text(r'''
#include <stdio.h>
#include <string.h>
#include "moe_b300.h"
int main(void) {
    moe_config_t c;
    memset(&c, 0, sizeof c);
    c.num_tokens = 16384; c.d_model = 4096; c.num_experts = 8; c.top_k = 2; c.d_ff = 14336;
    c.score_fn = MOE_SCORE_SOFTMAX; c.activation = MOE_ACT_SWIGLU; c.dtype = MOE_DTYPE_BF16;
    c.renormalize = 1; c.residual = 1; c.capacity_factor = 2.0f;
    size_t fwd = 0, bwd = 0;
    if (moe_workspace_size(&c, MOE_WS_FORWARD, &fwd) != MOE_OK) return 1;
    if (moe_workspace_size(&c, MOE_WS_BACKWARD, &bwd) != MOE_OK) return 2;
    int64_t cap = 0;
    if (moe_ec_capacity(&c, &cap) != MOE_OK) return 3;
    c.top_k = 0;
    size_t n = 0;
    moe_status_t st = moe_workspace_size(&c, MOE_WS_FORWARD, &n);
    char msg[256];
    moe_last_error(msg, sizeof msg);
    printf("%d %zu %zu %lld %d %s\n", moe_version(), fwd, bwd, (long long)cap, (int)st, msg);
    return 0;
}
''')
    exe = tmp_path / "user"
    libdir = os.path.dirname(_lib.LIB_PATH)
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                    "-L", libdir, "-lmoe_b300", "-Wl,-rpath," + libdir], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, (r.returncode, r.stderr)
    ver, fwd, bwd, cap, st, *msg = r.stdout.split()
    w = wl.WORKLOADS["mixtral"]
    assert int(ver) == L.moe_version()
    assert int(fwd) == _ws_expect(w)["fwd"]
    assert int(fwd) == moe.moe_workspace_size(moe.config_for(w), moe.MOE_WS_FORWARD)
    assert int(bwd) > 0
    assert int(cap) == 4096                        # ceil(16384 / 8 * 2.0)
    assert int(st) == 1 and msg                    # MOE_ERR_INVALID_ARG with a message


def test_options_are_checked_on_host(L):
    """moe_set_option / moe_get_option: defaults, range checks, round trip
    (host state only, nothing is launched)."""
    assert moe.moe_get_option(moe.MOE_OPT_PDL) == 1
    assert moe.moe_get_option(moe.MOE_OPT_GEMM_PAIR) == -1
    assert moe.moe_get_option(moe.MOE_OPT_WAIT_LIMIT_NS) == 2_000_000_000
    assert moe.moe_get_option(moe.MOE_OPT_GEMM_BAND) == -1
    with pytest.raises(moe.MoEError, match="out of range"):
        moe.moe_set_option(moe.MOE_OPT_GEMM_BAND, -2)
    with pytest.raises(moe.MoEError, match="out of range"):
        moe.moe_set_option(moe.MOE_OPT_WAIT_LIMIT_NS, -1)
    with pytest.raises(moe.MoEError, match="out of range"):
        moe.moe_set_option(moe.MOE_OPT_GEMM_PAIR, 2)
    with pytest.raises(moe.MoEError, match="out of range"):
        moe.moe_set_option(moe.MOE_OPT_PDL, 5)
    with pytest.raises(moe.MoEError, match="unknown option"):
        moe.moe_set_option(99, 0)
    with pytest.raises(moe.MoEError, match="unknown option"):
        moe.moe_get_option(99)
    try:
        moe.moe_set_option(moe.MOE_OPT_GEMM_PAIR, 0)
        assert moe.moe_get_option(moe.MOE_OPT_GEMM_PAIR) == 0
        moe.moe_set_option(moe.MOE_OPT_WAIT_LIMIT_NS, 12345)
        assert moe.moe_get_option(moe.MOE_OPT_WAIT_LIMIT_NS) == 12345
    finally:
        moe.moe_set_option(moe.MOE_OPT_GEMM_PAIR, -1)
        moe.moe_set_option(moe.MOE_OPT_WAIT_LIMIT_NS, 2_000_000_000)
