"""ctypes declarations of the C ABI in ``include/moe_b300.h``.

Loading fails loudly (``RuntimeError``) when ``libmoe_b300.so`` has not been
built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmoe_b300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED",
                3: "MOE_ERR_BAD_ALIGNMENT", 4: "MOE_ERR_WORKSPACE_TOO_SMALL", 5: "MOE_ERR_CUDA",
                6: "MOE_ERR_DEVICE_TIMEOUT"}
MOE_OPT_PDL, MOE_OPT_GEMM_PAIR, MOE_OPT_WAIT_LIMIT_NS, MOE_OPT_GEMM_BAND = 0, 1, 2, 3
(MOE_WS_FORWARD, MOE_WS_ROUTE, MOE_WS_PERMUTE, MOE_WS_EXPERT_FFN, MOE_WS_SHARED_FFN, MOE_WS_EXPERT_CHOICE,
 MOE_WS_BACKWARD) = range(7)


class MoEConfig(C.Structure):
    _fields_ = [("num_tokens", C.c_int64), ("d_model", C.c_int32), ("num_experts", C.c_int32),
                ("top_k", C.c_int32), ("d_ff", C.c_int32), ("score_fn", C.c_int32),
                ("activation", C.c_int32), ("dtype", C.c_int32), ("renormalize", C.c_int32),
                ("drop_tokens", C.c_int32), ("min_capacity", C.c_int32), ("num_shared", C.c_int32),
                ("residual", C.c_int32), ("capacity_factor", C.c_float)]


class MoEStats(C.Structure):
    _fields_ = [("aux_loss", C.c_float), ("z_loss", C.c_float), ("imbalance", C.c_float),
                ("utilization", C.c_float), ("drop_rate", C.c_float), ("dropped", C.c_int32),
                ("capacity", C.c_int32), ("total_kept", C.c_int32)]


class MoEWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w_router", "b_router", "w1", "b1", "w3", "w2", "b2",
                                          "shared_w1", "shared_w3", "shared_w2")]


MOE_STAGE_EVENTS = 8


class MoEForwardIO(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("logits", "topk_idx", "topk_w", "lse", "prob_mean",
                                          "counts", "kept", "offsets", "perm", "inv", "f", "stats",
                                          "stage_events", "x_perm", "pre_act", "hidden", "y_perm",
                                          "shared_pre_act", "shared_hidden")]


class MoESaved(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("topk_idx", "topk_w", "logits", "inv", "offsets", "counts", "x_perm",
                                          "pre_act", "hidden", "y_perm", "shared_pre_act", "shared_hidden")]


class MoEGrads(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("dx", "dw_router", "db_router", "dw1", "db1", "dw3", "dw2", "db2",
                                          "shared_dw1", "shared_dw3", "shared_dw2")]


class MoEECIO(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("logits", "row_token", "tok_row", "tok_gate", "offsets",
                                          "stage_events")]


MOE_BWD_STAGE_EVENTS = 9


class MoEBackwardOpts(C.Structure):
    _fields_ = [("aux_coef", C.c_float), ("z_coef", C.c_float), ("stage_events", C.c_void_p)]


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None

P = C.c_void_p
_SIGS = {
    "moe_version": ([], C.c_int32),
    "moe_last_error": ([C.c_char_p, C.c_size_t], None),
    "moe_workspace_size": ([P, C.c_int32, C.POINTER(C.c_size_t)], C.c_int),
    "moe_route": ([P] * 11 + [P, C.c_size_t, P], C.c_int),
    "moe_route_from_logits": ([P] * 8 + [P, C.c_size_t, P], C.c_int),
    "moe_permute": ([P] * 9 + [P, C.c_size_t, P], C.c_int),
    "moe_permute_noalloc": ([P] * 9 + [P], C.c_int),
    "moe_expert_ffn": ([P] * 9 + [P, C.c_size_t, P], C.c_int),
    "moe_shared_ffn": ([P] * 6 + [P, C.c_size_t, P], C.c_int),
    "moe_combine": ([P] * 7 + [P], C.c_int),
    "moe_stats": ([P] * 7 + [P], C.c_int),
    "moe_bias_update": ([P, P, P, C.c_float, P], C.c_int),
    "moe_forward": ([P] * 6 + [P, C.c_size_t, P], C.c_int),
    "moe_forward_from_routing": ([P] * 7 + [P, C.c_size_t, P], C.c_int),
    "moe_route_hash": ([P] * 4 + [P], C.c_int),
    "moe_ec_capacity": ([P, C.POINTER(C.c_int64)], C.c_int),
    "moe_backward": ([P] * 8 + [C.c_size_t, P], C.c_int),
    "moe_route_expert_choice": ([P] * 6 + [P], C.c_int),
    "moe_forward_expert_choice": ([P] * 5 + [P, C.c_size_t, P], C.c_int),
    "moe_check_device_error": ([C.POINTER(C.c_int32)], C.c_int),
    "moe_set_option": ([C.c_int32, C.c_int64], C.c_int),
    "moe_get_option": ([C.c_int32, C.POINTER(C.c_int64)], C.c_int),
}


def lib():
    """The loaded CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is not built; run `python -m sparse_mixture_experts_60_b300.build` "
                    "(there is no fallback implementation)")
            L = C.CDLL(LIB_PATH)
            for name, (args, res) in _SIGS.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def last_error() -> str:
    buf = C.create_string_buffer(512)
    lib().moe_last_error(buf, len(buf))
    return buf.value.decode(errors="replace")


def check(status: int) -> None:
    if status != MOE_OK:
        raise MoEError(status, last_error())
