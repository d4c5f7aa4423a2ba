"""Run one MoE layer of a given shape on random device weights, for use
under an external profiler (one process, one GPU, no timing of its own).

    python -m sparse_mixture_experts_60_b300.layer_run --tokens 2048 --d-model 7168 \\
        --experts 16 --top-k 1 --d-ff 2048 --train --steps 1

Each step is ``moe_forward`` (with ``--train``: the training forward, then
``moe_backward`` with aux_coef 0.01 and z_coef 0.001).  Weights are bf16
with standard deviation 0.02, x and dout standard normal, all drawn on the
device from a fixed seed.  The launches of one step, in order: router GEMM
(routing in its epilogue when E <= 32, else logits GEMM + routing kernel),
dispatch, FFN1, FFN2, combine, statistics; then the backward's combine,
router, dh, dx, dx assembly, dW2, dW1 (and dW3), router weight gradient.
"""
from __future__ import annotations

import argparse

from . import (BF16, GELU, RELU, SIGMOID, SOFTMAX, SWIGLU, MoELayer, TrainingLayer, make_config,
               moe_check_device_error)


def main(argv=None) -> int:
    import torch

    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--tokens", type=int, required=True)
    ap.add_argument("--d-model", type=int, required=True)
    ap.add_argument("--experts", type=int, required=True)
    ap.add_argument("--top-k", type=int, required=True)
    ap.add_argument("--d-ff", type=int, required=True)
    ap.add_argument("--activation", choices=["gelu", "relu", "swiglu"], default="swiglu")
    ap.add_argument("--score", choices=["softmax", "sigmoid"], default="softmax")
    ap.add_argument("--shared", type=int, default=0, help="shared experts (0 or 1)")
    ap.add_argument("--train", action="store_true")
    ap.add_argument("--steps", type=int, default=1)
    a = ap.parse_args(argv)
    act = {"gelu": GELU, "relu": RELU, "swiglu": SWIGLU}[a.activation]
    score = SOFTMAX if a.score == "softmax" else SIGMOID
    T, d, E, k, F = a.tokens, a.d_model, a.experts, a.top_k, a.d_ff
    cfg = make_config(T, d, E, k, F, score_fn=score, activation=act, dtype=BF16, renormalize=True,
                      drop_tokens=False, min_capacity=0, num_shared=a.shared, residual=True, capacity_factor=1.0)
    g = torch.Generator(device="cuda").manual_seed(1)

    def rnd(*shape, sd=0.02):
        return (torch.randn(*shape, device="cuda", generator=g) * sd).to(torch.bfloat16)

    w = {"w_router": rnd(E, d), "w1": rnd(E, F, d), "w2": rnd(E, d, F)}
    if act == SWIGLU:
        w["w3"] = rnd(E, F, d)
    else:
        w["b1"] = rnd(E, F)
        w["b2"] = rnd(E, d)
    if a.shared:
        w["shared_w1"] = rnd(a.shared, F, d)
        w["shared_w2"] = rnd(a.shared, d, F)
        if act == SWIGLU:
            w["shared_w3"] = rnd(a.shared, F, d)
    sel_bias = torch.zeros(E, dtype=torch.float32, device="cuda") if score == SIGMOID else None
    x = rnd(T, d, sd=1.0)
    if a.train:
        layer = TrainingLayer(cfg, w, sel_bias)
        dout = rnd(T, d, sd=1.0)
        grads = layer.new_grads()
        for _ in range(a.steps):
            layer.forward(x)
            layer.backward(dout, 0.01, 0.001, grads=grads)
    else:
        layer = MoELayer(cfg, w, sel_bias)
        out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
        for _ in range(a.steps):
            layer.forward(x, out)
    torch.cuda.synchronize()
    if moe_check_device_error():
        raise RuntimeError("device error flag set")
    print(f"ok: {a.steps} step(s) of T={T} d={d} E={E} k={k} F={F} ({a.activation}, {a.score}, "
          f"{'train' if a.train else 'forward'})")
    return 0


if __name__ == "__main__":
    raise SystemExit(main())
