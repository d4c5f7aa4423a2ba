"""Parity at the workloads' full sizes, through MoELayer.forward exactly as
the benchmark calls it: routing integers for every token (exact where the
key order is unambiguous), the dispatch, statistics, and the layer output
against the oracle, which evaluates the chosen tokens one by one.

Token choice: for the Mixtral-shaped and DeepSeek-V3-style layers, one
token from every 128-row tile of every expert segment of x_perm (a seeded
row inside the tile, plus the last row of each segment), so that every M
tile the expert GEMMs compute (and, through the full output rows, every N
tile) is checked; for the other workloads a seeded sample (all tokens of
the tiny layer)."""
import numpy as np
import pytest

from sparse_mixture_experts_60_b300 import workloads as wl
from tests.test_gpu_4_layer import check_layer, run_layer

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLES = {"tiny_fp32": None, "quickstart_bf16": 48, "capacity_e128": 96, "mixtral": "tiles",
           "deepseek_v3": "tiles"}
TILE_ROWS = 128


def tokens_per_tile(w, got, seed=0):
    """One token per TILE_ROWS-row tile of every expert segment (a seeded row
    inside the tile) and the token of each segment's last row."""
    off = got["offsets"].astype(np.int64)
    perm = got["perm"].astype(np.int64)
    g = np.random.default_rng(seed)
    toks = set()
    for e in range(w.E):
        lo, hi = int(off[e]), int(off[e + 1])
        for r0 in range(lo, hi, TILE_ROWS):
            r = int(g.integers(r0, min(r0 + TILE_ROWS, hi)))
            toks.add(int(perm[r]) // w.k)
        if hi > lo:
            toks.add(int(perm[hi - 1]) // w.k)
    return np.array(sorted(toks), np.int64)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_full_size_layer(name):
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w)
    _, got = run_layer(w, inp)
    n = SAMPLES[name]
    if n is None:
        tokens = np.arange(w.T)
    elif n == "tiles":
        tokens = tokens_per_tile(w, got)
        n_tiles = sum(-(-int(c) // TILE_ROWS) for c in got["kept"])
        assert len(tokens) >= min(n_tiles, w.T) // w.k      # tokens can share tiles only through their k rows
    else:
        tokens = wl.sample_tokens(w, n)
    check_layer(w, inp, got, tokens)
