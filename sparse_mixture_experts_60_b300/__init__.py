"""B300-native (sm_103a) forward of a token-choice top-k Mixture-of-Experts
FFN layer.

The functions below carry the names of the C ABI in ``include/moe_b300.h``
and only marshal arguments: torch CUDA tensors become device pointers, the
current torch stream becomes the launch stream, and a non-zero status
becomes a ``MoEError``.  Every step of the layer runs in the CUDA library
``libmoe_b300.so`` (build it with ``python -m
sparse_mixture_experts_60_b300.build``); nothing here computes.

``MoELayer`` is a convenience owner of weights, workspace and intermediate
buffers (allocated with torch) around ``moe_forward``.
"""
from __future__ import annotations

import ctypes as C
from typing import Dict, Optional

from ._lib import (MOE_OPT_GEMM_BAND, MOE_OPT_GEMM_PAIR, MOE_OPT_PDL, MOE_OPT_WAIT_LIMIT_NS,  # noqa: F401
                   MOE_BWD_STAGE_EVENTS, MOE_STAGE_EVENTS, MOE_WS_BACKWARD, MoEBackwardOpts, MOE_WS_EXPERT_CHOICE, MOE_WS_EXPERT_FFN,  # noqa: F401
                   MOE_WS_FORWARD, MOE_WS_PERMUTE, MOE_WS_ROUTE, MOE_WS_SHARED_FFN, MoEConfig, MoEECIO, MoEGrads,
                   MoESaved, MoEError, MoEForwardIO, MoEStats, MoEWeights, check,
                   last_error, lib)

SOFTMAX, SIGMOID = 0, 1
GELU, RELU, SWIGLU = 0, 1, 2
F32, BF16 = 0, 1


def make_config(num_tokens: int, d_model: int, num_experts: int, top_k: int, d_ff: int, *,
                score_fn: int = SOFTMAX, activation: int = GELU, dtype: int = BF16,
                renormalize: bool = True, drop_tokens: bool = False, min_capacity: int = 4,
                num_shared: int = 0, residual: bool = False, capacity_factor: float = 1.0) -> MoEConfig:
    return MoEConfig(num_tokens=num_tokens, d_model=d_model, num_experts=num_experts, top_k=top_k,
                     d_ff=d_ff, score_fn=score_fn, activation=activation, dtype=dtype,
                     renormalize=int(renormalize), drop_tokens=int(drop_tokens),
                     min_capacity=min_capacity, num_shared=num_shared, residual=int(residual),
                     capacity_factor=capacity_factor)


def config_for(w) -> MoEConfig:
    """MoEConfig of a layer description with the attributes T d E k F score_fn
    activation dtype renormalize drop_tokens min_capacity num_shared residual
    capacity_factor (for example a ``workloads.Workload``)."""
    return make_config(w.T, w.d, w.E, w.k, w.F, score_fn=w.score_fn, activation=w.activation,
                       dtype=w.dtype, renormalize=w.renormalize, drop_tokens=w.drop_tokens,
                       min_capacity=w.min_capacity, num_shared=w.num_shared, residual=w.residual,
                       capacity_factor=w.capacity_factor)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ws(ws):
    if ws is None:
        return None, 0
    return _ptr(ws), ws.numel() * ws.element_size()


def moe_workspace_size(cfg: MoEConfig, which: int = MOE_WS_FORWARD) -> int:
    n = C.c_size_t(0)
    check(lib().moe_workspace_size(C.byref(cfg), which, C.byref(n)))
    return n.value


def moe_route(cfg, x, w_router, b_router, sel_bias, logits, topk_idx, topk_w, lse, prob_mean, counts,
              ws, stream=None) -> None:
    p, n = _ws(ws)
    check(lib().moe_route(C.byref(cfg), _ptr(x), _ptr(w_router), _ptr(b_router), _ptr(sel_bias),
                          _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _ptr(lse), _ptr(prob_mean),
                          _ptr(counts), p, n, _stream(stream)))


def moe_route_from_logits(cfg, logits, sel_bias, topk_idx, topk_w, lse, prob_mean, counts, ws,
                          stream=None) -> None:
    p, n = _ws(ws)
    check(lib().moe_route_from_logits(C.byref(cfg), _ptr(logits), _ptr(sel_bias), _ptr(topk_idx),
                                      _ptr(topk_w), _ptr(lse), _ptr(prob_mean), _ptr(counts), p, n,
                                      _stream(stream)))


def moe_permute(cfg, x, topk_idx, counts, kept, offsets, perm, inv, x_perm, ws, stream=None) -> None:
    p, n = _ws(ws)
    check(lib().moe_permute(C.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(kept),
                            _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(x_perm), p, n, _stream(stream)))


def moe_permute_noalloc(cfg, x, topk_idx, counts, kept, offsets, perm, inv, x_perm, stream=None) -> None:
    """moe_permute without a workspace: for callers that cannot allocate
    device memory (the scratch is a fixed 512 KB array inside the library;
    see include/moe_b300.h for the size limit and the first-call set-up)."""
    check(lib().moe_permute_noalloc(C.byref(cfg), _ptr(x), _ptr(topk_idx), _ptr(counts), _ptr(kept),
                                    _ptr(offsets), _ptr(perm), _ptr(inv), _ptr(x_perm), _stream(stream)))


def moe_expert_ffn(cfg, x_perm, offsets, w1, b1, w3, w2, b2, y_perm, ws, stream=None) -> None:
    p, n = _ws(ws)
    check(lib().moe_expert_ffn(C.byref(cfg), _ptr(x_perm), _ptr(offsets), _ptr(w1), _ptr(b1), _ptr(w3),
                               _ptr(w2), _ptr(b2), _ptr(y_perm), p, n, _stream(stream)))


def moe_shared_ffn(cfg, x, shared_w1, shared_w3, shared_w2, z, ws, stream=None) -> None:
    p, n = _ws(ws)
    check(lib().moe_shared_ffn(C.byref(cfg), _ptr(x), _ptr(shared_w1), _ptr(shared_w3),
                               _ptr(shared_w2), _ptr(z), p, n, _stream(stream)))


def moe_combine(cfg, y_perm, inv, topk_w, shared_out, x, out, stream=None) -> None:
    check(lib().moe_combine(C.byref(cfg), _ptr(y_perm), _ptr(inv), _ptr(topk_w), _ptr(shared_out),
                            _ptr(x), _ptr(out), _stream(stream)))


def moe_stats(cfg, counts, kept, prob_mean, lse, f, stats, stream=None) -> None:
    """``stats`` is a CUDA buffer of at least ``ctypes.sizeof(MoEStats)`` bytes."""
    check(lib().moe_stats(C.byref(cfg), _ptr(counts), _ptr(kept), _ptr(prob_mean), _ptr(lse), _ptr(f),
                          _ptr(stats), _stream(stream)))


def moe_bias_update(cfg, counts, sel_bias, gamma: float, stream=None) -> None:
    check(lib().moe_bias_update(C.byref(cfg), _ptr(counts), _ptr(sel_bias), float(gamma),
                                _stream(stream)))


def weights_struct(w: Dict) -> MoEWeights:
    g = w.get
    return MoEWeights(w_router=_ptr(g("w_router")), b_router=_ptr(g("b_router")), w1=_ptr(g("w1")),
                      b1=_ptr(g("b1")), w3=_ptr(g("w3")), w2=_ptr(g("w2")), b2=_ptr(g("b2")),
                      shared_w1=_ptr(g("shared_w1")), shared_w3=_ptr(g("shared_w3")),
                      shared_w2=_ptr(g("shared_w2")))


def io_struct(io: Optional[Dict], stage_events=None) -> Optional[MoEForwardIO]:
    """``stage_events``: None or a sequence of MOE_STAGE_EVENTS raw
    cudaEvent_t handles (ints), recorded by moe_forward at stage boundaries."""
    if io is None and stage_events is None:
        return None
    io = io or {}
    s = MoEForwardIO(**{k: _ptr(io.get(k)) for k, _ in MoEForwardIO._fields_ if k != "stage_events"})
    if stage_events is not None:
        arr = (C.c_void_p * MOE_STAGE_EVENTS)(*[int(e) for e in stage_events])
        s._events_keepalive = arr
        s.stage_events = C.cast(arr, C.c_void_p)
    return s


def moe_forward(cfg, weights: Dict, x, sel_bias, out, io: Optional[Dict], ws, stream=None,
                stage_events=None) -> None:
    """``weights``: dict of CUDA tensors keyed like ``MoEWeights`` fields;
    ``io``: dict of optional intermediate output tensors keyed like
    ``MoEForwardIO`` fields (missing keys stay in the workspace);
    ``stage_events``: optional MOE_STAGE_EVENTS raw cudaEvent_t handles."""
    p, n = _ws(ws)
    wst = weights_struct(weights)
    ios = io_struct(io, stage_events)
    check(lib().moe_forward(C.byref(cfg), C.byref(wst), _ptr(x), _ptr(sel_bias), _ptr(out),
                            C.byref(ios) if ios is not None else None, p, n, _stream(stream)))


def moe_forward_from_routing(cfg, weights: Dict, x, topk_idx, topk_w, out, io: Optional[Dict], ws, stream=None,
                             stage_events=None) -> None:
    """The layer from caller-given routing (topk_idx [T,k], topk_w [T,k])."""
    p, n = _ws(ws)
    wst = weights_struct(weights)
    ios = io_struct(io, stage_events)
    check(lib().moe_forward_from_routing(C.byref(cfg), C.byref(wst), _ptr(x), _ptr(topk_idx), _ptr(topk_w),
                                         _ptr(out), C.byref(ios) if ios is not None else None, p, n,
                                         _stream(stream)))


def moe_route_hash(cfg, token_ids, topk_idx, topk_w, stream=None) -> None:
    """Hash routing of token ids [T] (int32) into topk_idx / topk_w [T,k]."""
    check(lib().moe_route_hash(C.byref(cfg), _ptr(token_ids), _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


def moe_ec_capacity(cfg) -> int:
    """Tokens per expert under expert-choice routing."""
    c = C.c_int64(0)
    check(lib().moe_ec_capacity(C.byref(cfg), C.byref(c)))
    return c.value


def moe_route_expert_choice(cfg, logits, row_token, tok_row, tok_gate, offsets, stream=None) -> None:
    """Expert-choice routing of fp32 logits [T,E] into row_token [E*C],
    tok_row [T,E], tok_gate [T,E] and offsets [E+1]."""
    check(lib().moe_route_expert_choice(C.byref(cfg), _ptr(logits), _ptr(row_token), _ptr(tok_row),
                                        _ptr(tok_gate), _ptr(offsets), _stream(stream)))


def ec_io_struct(io: Optional[Dict], stage_events=None) -> Optional[MoEECIO]:
    if io is None and stage_events is None:
        return None
    io = io or {}
    s = MoEECIO(**{k: _ptr(io.get(k)) for k, _ in MoEECIO._fields_ if k != "stage_events"})
    if stage_events is not None:
        arr = (C.c_void_p * MOE_STAGE_EVENTS)(*[int(e) for e in stage_events])
        s._events_keepalive = arr
        s.stage_events = C.cast(arr, C.c_void_p)
    return s


def moe_forward_expert_choice(cfg, weights: Dict, x, out, io: Optional[Dict], ws, stream=None,
                              stage_events=None) -> None:
    """The layer under expert-choice routing; ``io`` keyed like ``MoEECIO``."""
    p, n = _ws(ws)
    wst = weights_struct(weights)
    ios = ec_io_struct(io, stage_events)
    check(lib().moe_forward_expert_choice(C.byref(cfg), C.byref(wst), _ptr(x), _ptr(out),
                                          C.byref(ios) if ios is not None else None, p, n, _stream(stream)))


def moe_backward(cfg, weights: Dict, x, dout, saved: Dict, grads: Dict, ws, aux_coef: float = 0.0,
                 z_coef: float = 0.0, stream=None, stage_events=None) -> None:
    """Layer backward; ``saved`` keyed like ``MoESaved``, ``grads`` (fp32
    output tensors) keyed like ``MoEGrads`` (missing keys: not computed);
    ``stage_events``: optional MOE_BWD_STAGE_EVENTS raw cudaEvent_t handles."""
    p, n = _ws(ws)
    wst = weights_struct(weights)
    sv = MoESaved(**{k: _ptr(saved.get(k)) for k, _ in MoESaved._fields_})
    gr = MoEGrads(**{k: _ptr(grads.get(k)) for k, _ in MoEGrads._fields_})
    opts = MoEBackwardOpts(aux_coef=float(aux_coef), z_coef=float(z_coef))
    if stage_events is not None:
        arr = (C.c_void_p * MOE_BWD_STAGE_EVENTS)(*[int(e) for e in stage_events])
        opts._events_keepalive = arr
        opts.stage_events = C.cast(arr, C.c_void_p)
    check(lib().moe_backward(C.byref(cfg), C.byref(wst), _ptr(x), _ptr(dout), C.byref(sv), C.byref(gr),
                             C.byref(opts), p, n, _stream(stream)))


def moe_check_device_error() -> int:
    code = C.c_int32(0)
    check(lib().moe_check_device_error(C.byref(code)))
    return code.value


def moe_set_option(option: int, value: int) -> None:
    """Process-wide switch (MOE_OPT_PDL, MOE_OPT_GEMM_PAIR, MOE_OPT_WAIT_LIMIT_NS, MOE_OPT_GEMM_BAND)."""
    check(lib().moe_set_option(int(option), int(value)))


def moe_get_option(option: int) -> int:
    v = C.c_int64(0)
    check(lib().moe_get_option(int(option), C.byref(v)))
    return v.value


def stats_from_buffer(buf) -> Dict:
    """Decode a CUDA (or CPU) byte tensor holding one moe_stats_t."""
    raw = bytes(buf.detach().cpu().numpy().tobytes())[:C.sizeof(MoEStats)]
    s = MoEStats.from_buffer_copy(raw)
    return {k: getattr(s, k) for k, _ in MoEStats._fields_}


class _HostPipeline:
    """Overlapped host-buffer batches for a layer class with ``cfg``,
    ``device``, ``out_dtype()`` and ``forward(x, out, stream)``."""

    def run_host_batches(self, x_hosts, out_hosts, n_steps: int, stream=None):
        """Run ``n_steps`` batches from host memory with the copies overlapped:
        batch i is uploaded on a copy stream while batch i-1 computes, and its
        output is downloaded on another copy stream while batch i+1 computes.
        ``x_hosts`` / ``out_hosts``: sequences of pinned host tensors, used
        round-robin (step i reads ``x_hosts[i % len]`` and writes
        ``out_hosts[i % len]``).  Every step copies its whole input in and its
        whole output out.  Returns after enqueueing; synchronise to wait."""
        import torch
        comp = stream or torch.cuda.current_stream()
        if not hasattr(self, "_pipe"):
            dev = self.device
            T, d = self.cfg.num_tokens, self.cfg.d_model
            xdt = x_hosts[0].dtype
            self._pipe = dict(
                h2d=torch.cuda.Stream(device=dev), d2h=torch.cuda.Stream(device=dev),
                xd=[torch.empty(T, d, dtype=xdt, device=dev) for _ in range(2)],
                od=[torch.empty(T, d, dtype=self.out_dtype(), device=dev) for _ in range(2)])
        P = self._pipe
        P["h2d"].wait_stream(comp)       # the first upload follows earlier work on `comp`
        x_ready = [torch.cuda.Event() for _ in range(2)]
        x_free = [torch.cuda.Event() for _ in range(2)]
        o_ready = [torch.cuda.Event() for _ in range(2)]
        o_free = [torch.cuda.Event() for _ in range(2)]
        for i in range(n_steps):
            b = i % 2
            if i >= 2:
                P["h2d"].wait_event(x_free[b])            # batch i-2 no longer reads xd[b]
            with torch.cuda.stream(P["h2d"]):
                P["xd"][b].copy_(x_hosts[i % len(x_hosts)], non_blocking=True)
                x_ready[b].record(P["h2d"])
            comp.wait_event(x_ready[b])
            if i >= 2:
                comp.wait_event(o_free[b])                # batch i-2's output left od[b]
            self.forward(P["xd"][b], P["od"][b], comp)
            x_free[b].record(comp)
            o_ready[b].record(comp)
            P["d2h"].wait_event(o_ready[b])
            with torch.cuda.stream(P["d2h"]):
                out_hosts[i % len(out_hosts)].copy_(P["od"][b], non_blocking=True)
                o_free[b].record(P["d2h"])
        comp.wait_stream(P["d2h"])


class MoELayer(_HostPipeline):
    """Owner of one layer's device weights, workspace and intermediate
    buffers.  ``weights``: dict of CUDA tensors (``w_router``, ``b_router``,
    ``w1``, ``b1``, ``w3``, ``w2``, ``b2``, ``shared_w1``, ``shared_w3``,
    ``shared_w2``), ``sel_bias``: CUDA fp32 [E] for sigmoid scoring."""

    def __init__(self, cfg: MoEConfig, weights: Dict, sel_bias=None, device="cuda"):
        import torch
        self.cfg = cfg
        self.weights = weights
        self.sel_bias = sel_bias
        self.device = torch.device(device)
        T, E, k = cfg.num_tokens, cfg.num_experts, cfg.top_k
        dev = self.device
        self.ws = torch.empty(max(moe_workspace_size(cfg), 1), dtype=torch.uint8, device=dev)
        i32, f32 = torch.int32, torch.float32
        self.io = dict(logits=torch.empty(T, E, dtype=f32, device=dev),
                       topk_idx=torch.empty(T, k, dtype=i32, device=dev),
                       topk_w=torch.empty(T, k, dtype=f32, device=dev),
                       lse=torch.empty(T, dtype=f32, device=dev),
                       prob_mean=torch.empty(E, dtype=f32, device=dev),
                       counts=torch.empty(E, dtype=i32, device=dev),
                       kept=torch.empty(E, dtype=i32, device=dev),
                       offsets=torch.empty(E + 1, dtype=i32, device=dev),
                       perm=torch.empty(T * k, dtype=i32, device=dev),
                       inv=torch.empty(T * k, dtype=i32, device=dev),
                       f=torch.empty(E, dtype=f32, device=dev),
                       stats=torch.empty(C.sizeof(MoEStats), dtype=torch.uint8, device=dev))

    def out_dtype(self):
        import torch
        return torch.float32 if self.cfg.dtype == F32 else torch.bfloat16

    def forward(self, x, out=None, stream=None, stage_events=None):
        import torch
        if out is None:
            out = torch.empty(self.cfg.num_tokens, self.cfg.d_model, dtype=self.out_dtype(),
                              device=self.device)
        moe_forward(self.cfg, self.weights, x, self.sel_bias, out, self.io, self.ws, stream, stage_events)
        return out

    def graphed(self, x, out):
        """A CUDA graph of ``forward(x, out)`` on these two device buffers:
        one eager forward first (it also sets up the library's per-device
        state), then a capture on torch's capture stream.  ``g.replay()``
        runs the whole layer with one launch from the host: copy new inputs
        into ``x`` first, read the result from ``out``.  The graph is valid
        while the layer, ``x`` and ``out`` live and the layer's weights keep
        their addresses."""
        import torch
        self.forward(x, out)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            self.forward(x, out)
        return g

    def forward_host(self, x_host, out_host, x_dev=None, out_dev=None, stream=None):
        """End-to-end call from host buffers (pinned for overlap): copy x in,
        run the layer, copy out back; asynchronous on the stream."""
        import torch
        st = stream or torch.cuda.current_stream()
        with torch.cuda.stream(st):
            if x_dev is None:
                x_dev = torch.empty(x_host.shape, dtype=x_host.dtype, device=self.device)
            x_dev.copy_(x_host, non_blocking=True)
            out_dev = self.forward(x_dev, out_dev, st)
            out_host.copy_(out_dev, non_blocking=True)
        return out_host

    def forward_hashed(self, x, token_ids, out=None, stream=None, stage_events=None):
        """The layer with hash routing of ``token_ids`` [T] instead of the router."""
        import torch
        if out is None:
            out = torch.empty(self.cfg.num_tokens, self.cfg.d_model, dtype=self.out_dtype(), device=self.device)
        moe_route_hash(self.cfg, token_ids, self.io["topk_idx"], self.io["topk_w"], stream)
        moe_forward_from_routing(self.cfg, self.weights, x, self.io["topk_idx"], self.io["topk_w"], out, self.io,
                                 self.ws, stream, stage_events)
        return out

    def stats(self) -> Dict:
        return stats_from_buffer(self.io["stats"])


class TrainingLayer(MoELayer):
    """A layer whose forward keeps what the backward needs (x_perm, the
    first GEMM's pre-activations, H, the expert outputs) and whose backward
    returns fp32 gradients of sum <dout, out> + aux_coef L_aux + z_coef L_z."""

    def __init__(self, cfg: MoEConfig, weights: Dict, sel_bias=None, device="cuda"):
        import torch
        super().__init__(cfg, weights, sel_bias, device)
        T, k, d, F = cfg.num_tokens, cfg.top_k, cfg.d_model, cfg.d_ff
        nF = 2 * F if cfg.activation == SWIGLU else F
        dt, dev = self.out_dtype(), self.device
        R = max(T * k, 1)
        self.io.update(x_perm=torch.empty(R, d, dtype=dt, device=dev),
                       pre_act=torch.empty(R, nF, dtype=torch.bfloat16, device=dev),
                       hidden=torch.empty(R, F, dtype=dt, device=dev),
                       y_perm=torch.empty(R, d, dtype=torch.float32, device=dev))
        if cfg.num_shared:
            self.io.update(shared_pre_act=torch.empty(max(T, 1), nF, dtype=torch.bfloat16, device=dev),
                           shared_hidden=torch.empty(max(T, 1), F, dtype=dt, device=dev))
        self.bws = torch.empty(max(moe_workspace_size(cfg, MOE_WS_BACKWARD), 1), dtype=torch.uint8, device=dev)
        self._x = None

    def forward(self, x, out=None, stream=None, stage_events=None):
        self._x = x
        return super().forward(x, out, stream, stage_events)

    def saved(self) -> Dict:
        return {k: self.io.get(k) for k, _ in MoESaved._fields_}

    def new_grads(self) -> Dict:
        import torch
        cfg, w = self.cfg, self.weights
        T, d, E, F = cfg.num_tokens, cfg.d_model, cfg.num_experts, cfg.d_ff
        f32 = dict(dtype=torch.float32, device=self.device)
        g = dict(dx=torch.empty(max(T, 1), d, **f32), dw_router=torch.empty(E, d, **f32),
                 dw1=torch.empty(E, F, d, **f32), dw2=torch.empty(E, d, F, **f32))
        if w.get("b_router") is not None:
            g["db_router"] = torch.empty(E, **f32)
        if cfg.activation == SWIGLU:
            g["dw3"] = torch.empty(E, F, d, **f32)
        if w.get("b1") is not None:
            g["db1"] = torch.empty(E, F, **f32)
        if w.get("b2") is not None:
            g["db2"] = torch.empty(E, d, **f32)
        if cfg.num_shared:
            g["shared_dw1"] = torch.empty(F, d, **f32)
            g["shared_dw2"] = torch.empty(d, F, **f32)
            if cfg.activation == SWIGLU:
                g["shared_dw3"] = torch.empty(F, d, **f32)
        return g

    def backward(self, dout, aux_coef: float = 0.0, z_coef: float = 0.0, grads: Optional[Dict] = None,
                 stream=None, stage_events=None) -> Dict:
        g = grads if grads is not None else self.new_grads()
        moe_backward(self.cfg, self.weights, self._x, dout, self.saved(), g, self.bws, aux_coef, z_coef, stream,
                     stage_events)
        return g


class ExpertChoiceLayer(_HostPipeline):
    """One layer under expert-choice routing: device weights (as for
    ``MoELayer``), its workspace and the routing outputs."""

    def __init__(self, cfg: MoEConfig, weights: Dict, device="cuda"):
        import torch
        self.cfg = cfg
        self.weights = weights
        self.device = torch.device(device)
        T, E = cfg.num_tokens, cfg.num_experts
        self.capacity = moe_ec_capacity(cfg)
        dev = self.device
        self.ws = torch.empty(max(moe_workspace_size(cfg, MOE_WS_EXPERT_CHOICE), 1), dtype=torch.uint8, device=dev)
        i32, f32 = torch.int32, torch.float32
        self.io = dict(logits=torch.empty(T, E, dtype=f32, device=dev),
                       row_token=torch.empty(max(E * self.capacity, 1), dtype=i32, device=dev),
                       tok_row=torch.empty(T, E, dtype=i32, device=dev),
                       tok_gate=torch.empty(T, E, dtype=f32, device=dev),
                       offsets=torch.empty(E + 1, dtype=i32, device=dev))

    def out_dtype(self):
        import torch
        return torch.float32 if self.cfg.dtype == F32 else torch.bfloat16

    def forward(self, x, out=None, stream=None, stage_events=None):
        import torch
        if out is None:
            out = torch.empty(self.cfg.num_tokens, self.cfg.d_model, dtype=self.out_dtype(), device=self.device)
        moe_forward_expert_choice(self.cfg, self.weights, x, out, self.io, self.ws, stream, stage_events)
        return out


def bias_update(layer: MoELayer, gamma: float, stream=None) -> None:
    """Aux-loss-free balancing step after ``layer.forward``."""
    moe_bias_update(layer.cfg, layer.io["counts"], layer.sel_bias, gamma, stream)
