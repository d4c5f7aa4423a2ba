"""The bounded device-side waits of the tensor-core GEMM, made to run out on
purpose.  Every wait of the GEMM kernels on a copy or MMA barrier gives up
after MOE_OPT_WAIT_LIMIT_NS; a kernel whose wait gives up leaves its loops,
lets the copies and MMAs it already issued land, releases its tensor memory,
returns, and raises MOE_ERR_DEVICE_TIMEOUT.  With the limit at 0 ns the
first wait that does not succeed at once gives up (the epilogue's wait for
the first accumulator always does: a tile's main loop takes microseconds),
so the call must end with that status and without a fault or a hang; the
same call with the default limit must then be exact again, which shows the
context was left usable."""
import numpy as np
import pytest

import sparse_mixture_experts_60_b300 as moe
from sparse_mixture_experts_60_b300 import workloads as wl
from tests.test_gpu_3_ffn import check_ffn, oracle_dispatch, run_expert_ffn

pytestmark = pytest.mark.gpu

MOE_ERR_DEVICE_TIMEOUT = 6


def test_gemm_wait_limit_runs_out_then_next_call_is_exact():
    w = wl.WORKLOADS["quickstart_bf16"].scaled(600)       # 1200 expert rows over 8 experts, K = 1024 / 4096
    inp = wl.make_inputs(w)
    _, d_ref = oracle_dispatch(w, inp)
    default = moe.moe_get_option(moe.MOE_OPT_WAIT_LIMIT_NS)
    assert default == 2_000_000_000
    moe.moe_set_option(moe.MOE_OPT_GEMM_PAIR, 0)          # the one-CTA kernel's abort path
    try:
        moe.moe_set_option(moe.MOE_OPT_WAIT_LIMIT_NS, 0)
        run_expert_ffn(w, inp, d_ref, expect_flag=MOE_ERR_DEVICE_TIMEOUT)
    finally:
        moe.moe_set_option(moe.MOE_OPT_WAIT_LIMIT_NS, default)
        moe.moe_set_option(moe.MOE_OPT_GEMM_PAIR, -1)
    assert moe.moe_check_device_error() == 0              # the flag was read and cleared
    y = run_expert_ffn(w, inp, d_ref)                     # flag must stay 0
    check_ffn(w, inp, d_ref, y, 200)

