"""Parity at the workloads' full sizes, through MoELayer.forward exactly as
the benchmark calls it: routing integers for every token (exact where the
key order is unambiguous), the dispatch, statistics, and the layer output
on a seeded sample of tokens (including the first and last) against the
oracle, which evaluates those tokens one by one."""
import numpy as np
import pytest

from sparse_mixture_experts_60_b300 import workloads as wl
from tests.test_gpu_4_layer import check_layer, run_layer

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLES = {"tiny_fp32": None, "quickstart_bf16": 48, "capacity_e128": 96, "mixtral": 12, "deepseek_v3": 16}


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_full_size_layer(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    _, got = run_layer(w, inp)
    n = SAMPLES[name]
    tokens = np.arange(w.T) if n is None else wl.sample_tokens(w, n)
    check_layer(w, inp, got, tokens)
