"""Seeded synthetic workloads for the MoE-layer forward.

This module only *draws numbers*: shapes, value distributions and the
seeded generators that both the CUDA path and the CPU oracle are fed from.
It holds none of the layer's arithmetic (no routing, no FFN, no statistics).

Five workloads, shaped like the pages' examples:

* ``tiny_fp32``      -- "MoE Training: Mixture of Experts", Quick Start
  ``MoELayer`` at toy size in fp32 (T=64, d=32, E=4, k=2, GELU FFN 32->128->32,
  biases zero).
* ``quickstart_bf16`` -- the same Quick Start layer in bf16 at batch 4 x seq
  2048, hidden 1024, E=8, top-2, GELU FFN with d_ff = 4 * hidden.
* ``capacity_e128``  -- "MoE Training Guide" (DeepSpeed), Core MoE
  Parameters: E=128, top-1, capacity factor 1.25, min capacity 4, token
  dropping on; router logits ~N(0,1) with per-expert offsets ~N(0,1).
* ``mixtral``        -- Mixtral-8x7B-shaped layer (the Mixtral parameter
  arithmetic in the "MoE technical survey" page): d=4096, E=8, top-2,
  SwiGLU with d_ff=14336, no biases, residual added to the output.
* ``deepseek_v3``    -- "Mixture of Experts (MoE) From Scratch to DeepSeek V3"
  (shared + fine-grained experts, sigmoid routing, bias-based balancing):
  d=7168, 256 routed + 1 shared SwiGLU expert with d_ff=2048, top-8,
  selection bias b_i ~ U(-0.1, 0.1), Zipf(1.1) per-expert logit offsets.

Every tensor has its own PCG64 stream, seeded by
``SeedSequence([1000 + workload index, tensor id, expert index])``, so the
bytes do not depend on generation order or thread count.  bf16 tensors are
drawn in fp32 and rounded to nearest-even; they are returned as ``uint16``
bit patterns (``bf16_to_f32`` widens them exactly).
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional

import numpy as np

# activation / score / dtype codes (mirrored by value in the C header)
SOFTMAX, SIGMOID = 0, 1
GELU, RELU, SWIGLU = 0, 1, 2
F32, BF16 = 0, 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    T: int
    d: int
    E: int
    k: int
    F: int
    activation: int
    score_fn: int
    dtype: int
    router_bias: bool
    expert_bias: bool
    drop_tokens: bool = False
    capacity_factor: float = 1.0
    min_capacity: int = 4
    num_shared: int = 0
    residual: bool = False
    renormalize: bool = True
    batch: int = 1
    seq: int = 0
    bias_gamma: float = 0.0  # > 0: one aux-loss-free bias update after the forward

    @property
    def S(self) -> int:
        return self.T * self.k

    @property
    def gated(self) -> bool:
        return self.activation == SWIGLU

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == F32 else 2

    def scaled(self, T: int, name: Optional[str] = None) -> "Workload":
        """Same layer with a different token count (parity cases, samples)."""
        return dataclasses.replace(self, T=T, batch=1, seq=T, name=name or f"{self.name}_T{T}")

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_fp32", 0, T=64, d=32, E=4, k=2, F=128, activation=GELU,
                 score_fn=SOFTMAX, dtype=F32, router_bias=True, expert_bias=True,
                 batch=2, seq=32),
        Workload("quickstart_bf16", 1, T=8192, d=1024, E=8, k=2, F=4096, activation=GELU,
                 score_fn=SOFTMAX, dtype=BF16, router_bias=True, expert_bias=True,
                 batch=4, seq=2048),
        Workload("capacity_e128", 2, T=8192, d=1024, E=128, k=1, F=4096, activation=GELU,
                 score_fn=SOFTMAX, dtype=BF16, router_bias=True, expert_bias=True,
                 drop_tokens=True, capacity_factor=1.25, min_capacity=4, batch=1, seq=8192),
        Workload("mixtral", 3, T=16384, d=4096, E=8, k=2, F=14336, activation=SWIGLU,
                 score_fn=SOFTMAX, dtype=BF16, router_bias=False, expert_bias=False,
                 residual=True, batch=4, seq=4096),
        Workload("deepseek_v3", 4, T=4096, d=7168, E=256, k=8, F=2048, activation=SWIGLU,
                 score_fn=SIGMOID, dtype=BF16, router_bias=True, expert_bias=False,
                 num_shared=1, residual=True, batch=1, seq=4096, bias_gamma=0.001),
    ]
}

# tensor ids for the seed sequence
_TID = {"x": 1, "w_router": 2, "b_router": 3, "w1": 4, "b1": 5, "w3": 6, "w2": 7, "b2": 8,
        "sel_bias": 9, "shared_w1": 10, "shared_w3": 11, "shared_w2": 12, "logits": 13,
        "zipf_rank": 14, "sample": 15, "token_ids": 16}


def bf16_round(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> exact fp32 values."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _rng(w: Workload, name: str, sub: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([1000 + w.index, _TID[name], sub])))


def _normal(w: Workload, name: str, shape, std: float, sub: int = 0, store: Optional[int] = None):
    a = _rng(w, name, sub).standard_normal(int(np.prod(shape)), dtype=np.float32).reshape(shape)
    if std != 1.0:
        a *= np.float32(std)
    dt = w.dtype if store is None else store
    return bf16_round(a) if dt == BF16 else a


def _per_expert(w: Workload, name: str, rows: int, cols: int, std: float, n: int, threads: int):
    """[n, rows, cols] stacked expert matrices, one stream per expert."""
    dt = np.uint16 if w.dtype == BF16 else np.float32
    out = np.empty((n, rows, cols), dtype=dt)

    def job(e):
        out[e] = _normal(w, name, (rows, cols), std, sub=e)

    with ThreadPoolExecutor(max(1, threads)) as ex:
        list(ex.map(job, range(n)))
    return out


def _zipf_offsets(w: Workload) -> np.ndarray:
    """Per-expert logit offsets whose softmax popularity follows Zipf(1.1):
    a seeded random rank r_e in 1..E per expert, offset_e = -1.1 * ln(r_e)."""
    rank = _rng(w, "zipf_rank").permutation(w.E) + 1
    return (-1.1 * np.log(rank.astype(np.float64))).astype(np.float32)


def make_inputs(w: Workload, threads: int = 8, with_weights: bool = True) -> Dict[str, np.ndarray]:
    """All inputs of one workload as numpy arrays (bf16 as uint16 bits).

    Shapes: x [T,d]; w_router [E,d]; b_router [E] fp32; w1/w3 [E,F,d];
    b1 [E,F]; w2 [E,d,F]; b2 [E,d]; sel_bias [E] fp32; shared_w1/w3 [S,F,d];
    shared_w2 [S,d,F] (S = num_shared).  Weight matrices follow nn.Linear's
    [out_features, in_features] layout.
    """
    T, d, E, F = w.T, w.d, w.E, w.F
    inp: Dict[str, np.ndarray] = {"x": _normal(w, "x", (T, d), 1.0)}
    # router
    if w.name in ("capacity_e128", "deepseek_v3"):
        inp["w_router"] = _normal(w, "w_router", (E, d), 1.0 / math.sqrt(d))
    else:
        inp["w_router"] = _normal(w, "w_router", (E, d), 0.02)
    if w.router_bias:
        if w.name == "tiny_fp32":
            inp["b_router"] = np.zeros(E, np.float32)
        elif w.name == "capacity_e128":
            inp["b_router"] = _normal(w, "b_router", (E,), 1.0, store=F32)
        elif w.name == "deepseek_v3":
            inp["b_router"] = _zipf_offsets(w)
        else:
            inp["b_router"] = _normal(w, "b_router", (E,), 0.02, store=F32)
    if w.score_fn == SIGMOID:
        inp["sel_bias"] = _rng(w, "sel_bias").uniform(-0.1, 0.1, E).astype(np.float32)
    if not with_weights:
        return inp
    inp["w1"] = _per_expert(w, "w1", F, d, 0.02, E, threads)
    if w.gated:
        inp["w3"] = _per_expert(w, "w3", F, d, 0.02, E, threads)
    inp["w2"] = _per_expert(w, "w2", d, F, 0.02, E, threads)
    if w.expert_bias:
        if w.name == "tiny_fp32":
            inp["b1"] = np.zeros((E, F), np.float32)
            inp["b2"] = np.zeros((E, d), np.float32)
        else:
            inp["b1"] = _normal(w, "b1", (E, F), 0.02)
            inp["b2"] = _normal(w, "b2", (E, d), 0.02)
    if w.num_shared:
        inp["shared_w1"] = _per_expert(w, "shared_w1", F, d, 0.02, w.num_shared, threads)
        if w.gated:
            inp["shared_w3"] = _per_expert(w, "shared_w3", F, d, 0.02, w.num_shared, threads)
        inp["shared_w2"] = _per_expert(w, "shared_w2", d, F, 0.02, w.num_shared, threads)
    return inp


def make_logits(w: Workload, ties: bool = True) -> np.ndarray:
    """Synthetic fp32 router logits [T,E] for routing-only parity.

    N(0,1) plus the workload's per-expert offsets; with ``ties`` every 7th
    token has its logits snapped to a coarse grid (multiples of 1/4) so that
    equal keys occur and the lower-index tie rule is exercised.
    """
    g = _rng(w, "logits")
    lg = g.standard_normal((w.T, w.E), dtype=np.float32)
    if w.name == "capacity_e128":
        lg += _normal(w, "b_router", (w.E,), 1.0, store=F32)[None, :]
    if w.name == "deepseek_v3":
        lg += _zipf_offsets(w)[None, :]
    if ties:
        sl = slice(0, w.T, 7)
        lg[sl] = np.round(lg[sl] * 4.0) / 4.0
    return np.ascontiguousarray(lg, dtype=np.float32)


def make_token_ids(w: Workload, vocab: int = 32000) -> np.ndarray:
    """Seeded vocabulary ids [T] int32 for hash routing: ranks drawn with
    Zipf frequencies (p(r) proportional to 1/r over a 32000-entry vocabulary,
    the Mixtral tokenizer's size), mapped to ids by a fixed permutation."""
    g = _rng(w, "token_ids")
    p = 1.0 / np.arange(1, vocab + 1, dtype=np.float64)
    ranks = g.choice(vocab, size=w.T, p=p / p.sum())
    return g.permutation(vocab).astype(np.int32)[ranks]


def sample_tokens(w: Workload, n: int) -> np.ndarray:
    """A seeded, sorted sample of n distinct token indices (always includes
    the first and the last token so the ragged tail is covered)."""
    n = min(n, w.T)
    g = _rng(w, "sample")
    idx = set(g.choice(w.T, size=max(0, n - 2), replace=False).tolist()) | {0, w.T - 1}
    return np.array(sorted(idx), dtype=np.int64)
