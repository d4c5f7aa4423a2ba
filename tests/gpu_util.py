"""Helpers of the GPU parity tests: upload of generated inputs, download,
and the float tolerance of the layer.

Tolerances (floating point):
  fp32 layers: |gpu - ref| <= 1e-4 * max(|ref|, rms(ref)) per element, i.e.
               a max relative error of 1e-4 with the output RMS as the floor
               for elements near zero;
  bf16 layers: max |gpu - ref| <= 2e-2 * rms(ref).
  bf16 layers with heavy-tailed outputs (expert-choice routing, where a few
  tokens are taken by many experts): |gpu - ref| <= 2e-2 * rms(ref) +
  half_ulp_bf16(ref) per element, the second term being the rounding of the
  stored bf16 output itself, which no implementation avoids.
Integer outputs are compared for equality.
"""
from __future__ import annotations

import numpy as np
import torch

from sparse_mixture_experts_60_b300 import workloads as wl

FP32_REL = 1e-4
BF16_OF_RMS = 2e-2
REPORT = []   # (what, max_err, rms, ratio) of every float check, written at session end
WEIGHT_KEYS = ("w_router", "b_router", "w1", "b1", "w3", "w2", "b2", "shared_w1", "shared_w3", "shared_w2")


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach()
    if t.dtype == torch.bfloat16:
        return wl.bf16_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy()


def weights(inp):
    return {k: dev(inp[k]) for k in WEIGHT_KEYS if k in inp}


def as_f32(a: np.ndarray) -> np.ndarray:
    return wl.bf16_to_f32(a) if a.dtype == np.uint16 else np.asarray(a, np.float32)


def half_ulp_bf16(v: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.exp2(e - 8)


def float_check(gpu, ref, w, what="", report=None, out_rounding=False):
    """Assert the layer's float tolerance; returns (max_err, rms, ratio)."""
    g = np.asarray(gpu, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    err = np.abs(g - r)
    rms = float(np.sqrt(np.mean(r * r))) if r.size else 0.0
    if w.dtype == wl.F32:
        bound = FP32_REL * np.maximum(np.abs(r), rms)
        worst = float(np.max(err / np.maximum(bound, 1e-300))) if r.size else 0.0
        ok = bool(np.all(err <= bound))
        ratio = worst * FP32_REL
    elif out_rounding:
        ratio = float(err.max() / rms) if r.size else 0.0
        ok = bool(np.all(err <= BF16_OF_RMS * rms + half_ulp_bf16(r)))
    else:
        ratio = float(err.max() / rms) if r.size else 0.0
        ok = ratio <= BF16_OF_RMS
    rec = (what, float(err.max()) if r.size else 0.0, rms, ratio)
    REPORT.append(rec)
    if report is not None:
        report.append(rec)
    assert ok, f"{what}: max err {err.max():.3e} rms {rms:.3e} ratio {ratio:.3e}"
    return float(err.max()) if r.size else 0.0, rms, ratio


def topk_valid(sel, keys, margin):
    """Every chosen expert's key is >= every unchosen key - margin."""
    E = keys.shape[0]
    mask = np.zeros(E, bool)
    mask[sel] = True
    if mask.all():
        return True
    return keys[mask].min() >= keys[~mask].max() - margin


def keys_of(w, logits, sel_bias):
    """Selection keys as the oracle defines them (fp32)."""
    from oracle import oracle as orc
    if w.score_fn == wl.SOFTMAX:
        return np.asarray(logits, np.float32)
    return orc.sigmoid_keys(logits, sel_bias)
