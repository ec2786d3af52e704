"""ctypes binding of libbre (include/bre.h).  Argument marshalling only: every step runs
in the library's CUDA kernels.  Importing works without a GPU; calling needs one."""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

_lib = None

BRE_OK, BRE_ERR_ARG, BRE_ERR_UNSUPPORTED, BRE_ERR_CUDA, BRE_ERR_WORKSPACE = range(5)
BRE_DEVERR_EXPERT_ID, BRE_DEVERR_ROW_ID, BRE_DEVERR_TIMEOUT = 1, 2, 4
BRE_FMT_Q2_K, BRE_FMT_Q8_0, BRE_FMT_Q2_K_R16 = 1, 2, 3

# exported symbol -> (restype, argtypes)
_P, _I, _I64, _SZ, _F = C.c_void_p, C.c_int, C.c_int64, C.c_size_t, C.c_float
SIGNATURES = {
    "bre_status_string": (C.c_char_p, [_I]),
    "moe_route_workspace": (_SZ, [_I, _I]),
    "moe_route": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _SZ, _P]),
    "engram_inject_workspace": (_SZ, [_I, _I, _I]),
    "engram_inject": (_I, [_P, _I64, _P, _I, _P, _I, _P, _P, _P, _P, _I, _F, _P, _P, _P, _P, _SZ, _P]),
    "moe_route_ex": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _I, _P, _P, _P, _P, _SZ, _P]),
    "moe_route_static": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "moe_permute": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_route_permute": (_I, [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "moe_expert_ffn_workspace": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_expert_ffn": (_I, [_P, _P, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "moe_combine": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _P, _P, _P]),
    "moe_residual_norm": (_I, [_P, _P, _I, _I, _F, _F, _P, _P, _P]),
    "engram_gather_decode": (_I, [_P, _P, _I, _P, _I, _I, _P, _P, _P]),
    "bre_dequant": (_I, [_I, _P, _I64, _P, _P]),
    "bre_repack_q2k_r16": (_I, [_P, _P, _I, _I, _I, _I64, _I64, _P]),
    "bre_set_ffn_wait_limit": (_I, [_I64]),
}


class BreWeights(C.Structure):
    _fields_ = [("gate", C.c_void_p), ("up", C.c_void_p), ("down", C.c_void_p), ("fmt", C.c_int32),
                ("n_experts", C.c_int32), ("d", C.c_int32), ("d_ff", C.c_int32),
                ("expert_stride_gate", C.c_int64), ("expert_stride_up", C.c_int64),
                ("expert_stride_down", C.c_int64)]


class BreError(RuntimeError):
    pass


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libbre.so; raises if it is missing and cannot be built (there is no fallback)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise ImportError(f"libbre.so not built ({path}); run bit_routed_expert_gb300.build.build()")
            path = _build.build()
        L = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def check(rc: int, what: str):
    if rc != BRE_OK:
        msg = load().bre_status_string(rc).decode()
        raise BreError(f"{what}: {msg} (status {rc})")


def ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def stream_handle(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)
