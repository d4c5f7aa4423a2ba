"""ctypes wrapper of the plain CPU oracle (``moe_oracle.c``).

TEST INFRASTRUCTURE: only the tests, the package smoke check and the
benchmark's CPU-baseline leg use this module.  It never imports the product
package; a layer description is any object with the attributes
``T d E k F score_fn activation renormalize drop_tokens min_capacity
capacity_factor num_shared residual dtype`` (the workload generator's
``Workload`` has them).

Parity unpinned: the floating-point layer output of the bf16 workloads has
no printed worked example on the pages; it is pinned only through the
brute-force path, the E=1 dense special case, and the closed forms checked
in the oracle tests.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from typing import Dict, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11",
          "-shared", "-fPIC", "-Wall", "-Wno-unused-function"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp contraction off: every fp32 and fp64
    operation is rounded on its own, as written)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(C.Structure):
    _fields_ = [("T", C.c_int64), ("d", C.c_int32), ("E", C.c_int32), ("k", C.c_int32),
                ("F", C.c_int32), ("score_fn", C.c_int32), ("activation", C.c_int32),
                ("renormalize", C.c_int32), ("drop_tokens", C.c_int32),
                ("min_capacity", C.c_int32), ("num_shared", C.c_int32), ("residual", C.c_int32),
                ("dtype", C.c_int32), ("capacity_factor", C.c_double)]


class _Tensors(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("x", "w_router", "b_router", "sel_bias", "w1", "b1", "w3", "w2", "b2",
                 "sw1", "sw3", "sw2")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            L.orc_num_threads.restype = C.c_int
            L.orc_exp32.restype = C.c_float
            L.orc_exp32.argtypes = [C.c_float]
            L.orc_sigmoid32.restype = C.c_float
            L.orc_sigmoid32.argtypes = [C.c_float]
            L.orc_round_bf16.restype = C.c_double
            L.orc_round_bf16.argtypes = [C.c_double]
            L.orc_gelu.restype = C.c_double
            L.orc_gelu.argtypes = [C.c_double]
            L.orc_silu.restype = C.c_double
            L.orc_silu.argtypes = [C.c_double]
            L.orc_capacity.restype = C.c_int64
            L.orc_capacity.argtypes = [P]
            L.orc_router_logits.argtypes = [P, P, P]
            L.orc_route.argtypes = [P, P, P, P, P, P, P]
            L.orc_dispatch.argtypes = [P] * 7
            L.orc_expert_row.argtypes = [P, P, C.c_int64, P, P]
            L.orc_forward_tokens.argtypes = [P, P, P, P, P, P, C.c_int64, P]
            L.orc_dense_all.argtypes = [P] * 7
            L.orc_stats.argtypes = [P] * 8
            L.orc_bias_update.argtypes = [P, P, P, C.c_float]
            L.orc_param_counts.argtypes = [C.c_int64] * 4 + [C.c_int, P]
            L.orc_sigmoid_keys.argtypes = [P, P, C.c_int64, C.c_int64, P]
            L.orc_expert_rows.argtypes = [P, P, C.c_int64, P, P, P]
            L.orc_fmix32.restype = C.c_uint32
            L.orc_fmix32.argtypes = [C.c_uint32]
            L.orc_route_hash.argtypes = [C.c_int64, C.c_int32, C.c_int32, P, P, P]
            L.orc_ec_capacity.restype = C.c_int64
            L.orc_ec_capacity.argtypes = [C.c_int64, C.c_int32, C.c_double, C.c_int32]
            L.orc_route_expert_choice.argtypes = [C.c_int64, C.c_int32, C.c_int64, P, P, P, P]
            L.orc_backward.argtypes = [P] * 8 + [C.c_double, C.c_double, P]
            L.orc_backward_units.argtypes = [P] * 7 + [C.c_int64] + [P] * 4
            _lib = L
    return _lib


def num_threads() -> int:
    return lib().orc_num_threads()


def _cfg(w) -> _Cfg:
    return _Cfg(T=w.T, d=w.d, E=w.E, k=w.k, F=w.F, score_fn=w.score_fn, activation=w.activation,
                renormalize=int(w.renormalize), drop_tokens=int(w.drop_tokens),
                min_capacity=w.min_capacity, num_shared=w.num_shared, residual=int(w.residual),
                dtype=w.dtype, capacity_factor=float(np.float32(w.capacity_factor)))


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _tensors(inp: Dict[str, np.ndarray]) -> _Tensors:
    g = inp.get
    return _Tensors(x=_p(g("x")), w_router=_p(g("w_router")), b_router=_p(g("b_router")),
                    sel_bias=_p(g("sel_bias")), w1=_p(g("w1")), b1=_p(g("b1")), w3=_p(g("w3")),
                    w2=_p(g("w2")), b2=_p(g("b2")), sw1=_p(g("shared_w1")),
                    sw3=_p(g("shared_w3")), sw2=_p(g("shared_w2")))


def _c(a, dt):
    return np.ascontiguousarray(a, dtype=dt)


# ---------------------------------------------------------------- steps
def exp32(a: float) -> float:
    return lib().orc_exp32(float(a))


def sigmoid32(a: float) -> float:
    return lib().orc_sigmoid32(float(a))


def sigmoid_keys(logits: np.ndarray, sel_bias: Optional[np.ndarray]) -> np.ndarray:
    """fp32 selection keys sigmoid32(logit) + b_e of a [T, E] logit block."""
    lg = _c(logits, np.float32)
    sb = None if sel_bias is None else _c(sel_bias, np.float32)
    out = np.empty_like(lg)
    lib().orc_sigmoid_keys(lg.ctypes.data, _p(sb), lg.shape[0], lg.shape[1], out.ctypes.data)
    return out


def round_bf16(v: float) -> float:
    return lib().orc_round_bf16(float(v))


def gelu(v: float) -> float:
    return lib().orc_gelu(float(v))


def silu(v: float) -> float:
    return lib().orc_silu(float(v))


def capacity(w) -> int:
    c = _cfg(w)
    return int(lib().orc_capacity(C.byref(c)))


def router_logits(w, inp) -> np.ndarray:
    c, tn = _cfg(w), _tensors(inp)
    out = np.empty((w.T, w.E), np.float32)
    lib().orc_router_logits(C.byref(c), C.byref(tn), out.ctypes.data)
    return out


def route(w, logits: np.ndarray, sel_bias: Optional[np.ndarray] = None):
    """-> dict(idx [T,k] int32, gate [T,k] f64, lse [T] f64, prob_sum [E] f64)"""
    c = _cfg(w)
    logits = _c(logits, np.float32)
    sb = None if sel_bias is None else _c(sel_bias, np.float32)
    idx = np.empty((w.T, w.k), np.int32)
    gate = np.empty((w.T, w.k), np.float64)
    lse = np.empty(w.T, np.float64)
    ps = np.empty(w.E, np.float64)
    lib().orc_route(C.byref(c), logits.ctypes.data, _p(sb), idx.ctypes.data, gate.ctypes.data,
                    lse.ctypes.data, ps.ctypes.data)
    return dict(idx=idx, gate=gate, lse=lse, prob_sum=ps)


def fmix32(h: int) -> int:
    return int(lib().orc_fmix32(h & 0xFFFFFFFF))


def route_hash(T: int, E: int, k: int, token_ids: np.ndarray):
    """-> dict(idx [T,k] int32, gate [T,k] f64) of hash routing."""
    tid = _c(token_ids, np.int32)
    idx = np.empty((T, k), np.int32)
    gate = np.empty((T, k), np.float64)
    lib().orc_route_hash(T, E, k, tid.ctypes.data, idx.ctypes.data, gate.ctypes.data)
    return dict(idx=idx, gate=gate)


def ec_capacity(w) -> int:
    return int(lib().orc_ec_capacity(w.T, w.E, float(np.float32(w.capacity_factor)), w.min_capacity))


def route_expert_choice(w, logits: np.ndarray):
    """-> dict(C, row_token [E*C], tok_row [T,E], tok_gate [T,E] f64)."""
    Cc = ec_capacity(w)
    lg = _c(logits, np.float32)
    row_token = np.empty(max(w.E * Cc, 1), np.int32)[: w.E * Cc]
    tok_row = np.empty((w.T, w.E), np.int32)
    tok_gate = np.empty((w.T, w.E), np.float64)
    lib().orc_route_expert_choice(w.T, w.E, Cc, lg.ctypes.data, row_token.ctypes.data, tok_row.ctypes.data,
                                  tok_gate.ctypes.data)
    return dict(C=Cc, row_token=row_token, tok_row=tok_row, tok_gate=tok_gate)


def forward_tokens_ec(w, inp, ec, tokens) -> np.ndarray:
    """Layer output under expert-choice routing: out_t = sum over the experts
    that chose t (expert order) of gate * E_e(x_t), + shared + residual."""
    import dataclasses as _dc
    wk = _dc.replace(w, k=w.E) if _dc.is_dataclass(w) else w
    idx = np.tile(np.arange(w.E, dtype=np.int32), (w.T, 1))
    return forward_tokens(wk, inp, idx, ec["tok_gate"], ec["tok_row"].reshape(-1), tokens)


def dispatch(w, idx: np.ndarray):
    """-> dict(counts, kept [E], offsets [E+1], perm [S], inv [S]) all int32"""
    c = _cfg(w)
    idx = _c(idx, np.int32)
    S = w.T * w.k
    counts = np.empty(w.E, np.int32)
    kept = np.empty(w.E, np.int32)
    offsets = np.empty(w.E + 1, np.int32)
    perm = np.empty(max(S, 1), np.int32)[:S]
    inv = np.empty(max(S, 1), np.int32)[:S]
    lib().orc_dispatch(C.byref(c), idx.ctypes.data, counts.ctypes.data, kept.ctypes.data,
                       offsets.ctypes.data, perm.ctypes.data, inv.ctypes.data)
    return dict(counts=counts, kept=kept, offsets=offsets, perm=perm, inv=inv)


def expert_row(w, inp, e: int, xrow: np.ndarray) -> np.ndarray:
    c, tn = _cfg(w), _tensors(inp)
    xv = _c(xrow, np.float64)
    y = np.empty(w.d, np.float64)
    lib().orc_expert_row(C.byref(c), C.byref(tn), int(e), xv.ctypes.data, y.ctypes.data)
    return y


def expert_rows(w, inp, experts, xrows) -> np.ndarray:
    """y[i] = E_{experts[i]}(xrows[i]) in parallel; a negative expert id -s-1
    selects shared expert s."""
    c, tn = _cfg(w), _tensors(inp)
    ex = _c(experts, np.int32)
    xv = _c(xrows, np.float64)
    y = np.empty((len(ex), w.d), np.float64)
    lib().orc_expert_rows(C.byref(c), C.byref(tn), len(ex), ex.ctypes.data, xv.ctypes.data, y.ctypes.data)
    return y


def forward_tokens(w, inp, idx, gate, inv, tokens) -> np.ndarray:
    c, tn = _cfg(w), _tensors(inp)
    idx = _c(idx, np.int32)
    gate = _c(gate, np.float64)
    inv = None if inv is None else _c(inv, np.int32)
    tokens = _c(tokens, np.int64)
    out = np.empty((len(tokens), w.d), np.float64)
    lib().orc_forward_tokens(C.byref(c), C.byref(tn), idx.ctypes.data, gate.ctypes.data, _p(inv),
                             tokens.ctypes.data, len(tokens), out.ctypes.data)
    return out


def dense_all(w, inp, idx, gate, inv):
    """Brute force: (all-experts tensor [T,E,d], layer output [T,d])."""
    c, tn = _cfg(w), _tensors(inp)
    idx = _c(idx, np.int32)
    gate = _c(gate, np.float64)
    inv = None if inv is None else _c(inv, np.int32)
    allv = np.empty((w.T, w.E, w.d), np.float64)
    out = np.empty((w.T, w.d), np.float64)
    lib().orc_dense_all(C.byref(c), C.byref(tn), idx.ctypes.data, gate.ctypes.data, _p(inv),
                        allv.ctypes.data, out.ctypes.data)
    return allv, out


def stats(w, counts, kept, prob_sum, lse):
    """-> dict(f, P, aux, z, dropped, imbalance, utilization, drop_rate)"""
    c = _cfg(w)
    counts = _c(counts, np.int32)
    kept = _c(kept, np.int32)
    prob_sum = _c(prob_sum, np.float64)
    lse = _c(lse, np.float64)
    f = np.empty(w.E, np.float64)
    P = np.empty(w.E, np.float64)
    s = np.empty(6, np.float64)
    lib().orc_stats(C.byref(c), counts.ctypes.data, kept.ctypes.data, prob_sum.ctypes.data,
                    lse.ctypes.data, f.ctypes.data, P.ctypes.data, s.ctypes.data)
    return dict(f=f, P=P, aux=s[0], z=s[1], dropped=int(s[2]), imbalance=s[3],
                utilization=s[4], drop_rate=s[5])


def bias_update(w, counts, bias, gamma: float) -> np.ndarray:
    c = _cfg(w)
    counts = _c(counts, np.int32)
    b = np.array(bias, dtype=np.float32, copy=True)
    lib().orc_bias_update(C.byref(c), counts.ctypes.data, b.ctypes.data, float(gamma))
    return b


def param_counts(d: int, F: int, E: int, k: int, gated: bool):
    out = np.empty(4, np.int64)
    lib().orc_param_counts(d, F, E, k, int(gated), out.ctypes.data)
    return dict(expert=int(out[0]), router=int(out[1]), total=int(out[2]), active=int(out[3]))


class _Grads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("dx", "dw_router", "db_router", "dw1", "db1", "dw3", "dw2", "db2",
                                          "dsw1", "dsw3", "dsw2", "dgate", "dlogits")]


def backward(w, inp, fwd, dout, aux_coef: float = 0.0, z_coef: float = 0.0, units=None):
    """Gradients (fp64) of sum_t <dout_t, out_t> + aux_coef * L_aux +
    z_coef * L_z for the forward ``fwd`` (``layer``'s routing and dispatch:
    logits, idx, gate, inv, counts).  Returns a dict keyed like the C
    orc_grads fields; weight gradients of absent weights are None.
    ``units``: compute the expert weight gradients only for these units
    (u = expert * F + f, experts >= E being shared experts) and return them
    as rows: dw1_rows / dw3_rows [n, d], dw2_cols [n, d], db1_units [n]."""
    c, tn = _cfg(w), _tensors(inp)
    T, d, E, k, F, S = w.T, w.d, w.E, w.k, w.F, w.num_shared
    gated = w.activation == 2
    full = units is None
    z = lambda *shape: np.zeros(shape) if full else None
    out = dict(dx=np.zeros((T, d)), dw_router=np.zeros((E, d)), db_router=np.zeros(E),
               dw1=z(E, F, d), db1=z(E, F) if "b1" in inp else None,
               dw3=z(E, F, d) if gated else None, dw2=z(E, d, F),
               db2=np.zeros((E, d)) if "b2" in inp else None,
               dsw1=z(S, F, d) if S else None, dsw3=z(S, F, d) if S and gated else None,
               dsw2=z(S, d, F) if S else None, dgate=np.zeros((T, k)), dlogits=np.zeros((T, E)))
    g = _Grads(**{n: _p(out[n]) for n, _ in _Grads._fields_})
    lg = _c(fwd["logits"], np.float32)
    idx = _c(fwd["idx"], np.int32)
    gate = _c(fwd["gate"], np.float64)
    inv = _c(fwd["inv"], np.int32)
    counts = _c(fwd["counts"], np.int32)
    dout = _c(dout, np.float64)
    lib().orc_backward(C.byref(c), C.byref(tn), lg.ctypes.data, idx.ctypes.data, gate.ctypes.data,
                       inv.ctypes.data, counts.ctypes.data, dout.ctypes.data, float(aux_coef), float(z_coef),
                       C.byref(g))
    if not full:
        u = _c(units, np.int64)
        n = len(u)
        out.update(units=u, dw1_rows=np.zeros((n, d)), dw3_rows=np.zeros((n, d)) if gated else None,
                   dw2_cols=np.zeros((n, d)), db1_units=np.zeros(n))
        lib().orc_backward_units(C.byref(c), C.byref(tn), idx.ctypes.data, gate.ctypes.data, inv.ctypes.data,
                                 dout.ctypes.data, u.ctypes.data, n, out["dw1_rows"].ctypes.data,
                                 _p(out["dw3_rows"]), out["dw2_cols"].ctypes.data, out["db1_units"].ctypes.data)
    return out


def loss(w, inp, dout, aux_coef: float = 0.0, z_coef: float = 0.0) -> float:
    """sum_t <dout_t, out_t> + aux_coef * L_aux + z_coef * L_z of the layer
    (the scalar the backward differentiates)."""
    r = layer(w, inp)
    return float(np.sum(np.asarray(dout, np.float64) * r["out"]) + aux_coef * r["stats"]["aux"]
                 + z_coef * r["stats"]["z"])


def layer(w, inp, tokens=None):
    """Whole reference layer: routing for every token, outputs for `tokens`
    (all tokens when None).  Returns a dict of every intermediate."""
    logits = router_logits(w, inp)
    r = route(w, logits, inp.get("sel_bias"))
    dsp = dispatch(w, r["idx"])
    st = stats(w, dsp["counts"], dsp["kept"], r["prob_sum"], r["lse"])
    if tokens is None:
        tokens = np.arange(w.T, dtype=np.int64)
    out = forward_tokens(w, inp, r["idx"], r["gate"], dsp["inv"], tokens)
    return dict(logits=logits, tokens=np.asarray(tokens), out=out, **r, **dsp, stats=st)
