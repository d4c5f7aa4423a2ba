"""The GELU epilogues of the expert GEMMs take the Gaussian CDF from the
rational approximation of erfc in Abramowitz & Stegun, Handbook of
Mathematical Functions, 7.1.26 (absolute error at most 1.5e-7 for x >= 0).
The constants are read from the CUDA source and the published bound is
checked against scipy's erfc, so a mistyped constant fails here; the GPU
parity tests of the GELU layers check the compiled epilogues end to end."""
import os
import re

import numpy as np
from scipy.special import erf, erfc

SRC = os.path.join(os.path.dirname(__file__), "..", "sparse_mixture_experts_60_b300", "csrc", "gemm_sm103.cu")


def _constants():
    src = open(SRC).read()
    body = src[src.index("struct ErfcAS7126 {"):]
    body = body[:body.index("};")]
    vals = dict(re.findall(r"\b(p|a[1-5])\s*=\s*(-?[0-9.]+)f", body))
    assert set(vals) == {"p", "a1", "a2", "a3", "a4", "a5"}, vals
    return {k: float(v) for k, v in vals.items()}


def _erfc_approx(x, c):
    t = 1.0 / (1.0 + c["p"] * x)
    return t * (c["a1"] + t * (c["a2"] + t * (c["a3"] + t * (c["a4"] + t * c["a5"])))) * np.exp(-x * x)


def test_erfc_constants_meet_published_bound():
    c = _constants()
    x = np.linspace(0.0, 12.0, 400001)
    assert np.abs(_erfc_approx(x, c) - erfc(x)).max() <= 1.5e-7


def test_gelu_and_derivative_from_the_approximation():
    c = _constants()
    a = np.linspace(-12.0, 12.0, 200001)
    half_erfc = 0.5 * _erfc_approx(np.abs(a) / np.sqrt(2.0), c)
    cdf = np.where(a >= 0, 1.0 - half_erfc, half_erfc)
    exact = 0.5 * (1.0 + erf(a / np.sqrt(2.0)))
    assert np.abs(cdf - exact).max() <= 0.75e-7
    dens = np.exp(-0.5 * a * a) / np.sqrt(2.0 * np.pi)
    assert np.abs((cdf + a * dens) - (exact + a * dens)).max() <= 0.75e-7
    # GELU(a) = a Phi(a): absolute error at most |a| * 0.75e-7
    assert np.all(np.abs(a * cdf - a * exact) <= np.abs(a) * 0.75e-7 + 1e-300)
