"""CPU oracle for the routed-expert MoE layer and the Engram gather (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline leg.  The product path never imports it.  The C source
(``oracle.c``) is single-threaded, has its own format decoders, and shares no
code with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None

FMT_Q2_K = 1
FMT_Q8_0 = 2


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, no fast-math, no FMA contraction)."""
    src = os.path.join(_HERE, "oracle.c")
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
            os.path.getmtime(src), os.path.getmtime(os.path.join(_HERE, "oracle.h"))):
        tmp = _SO + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-Wall", "-Wextra", "-Wno-unused-parameter",
                               "-o", tmp, src, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_SO)
        P = C.c_void_p
        i32, i64 = C.c_int, C.c_int64
        L.or_f16_to_f32.restype = C.c_float
        L.or_f16_to_f32.argtypes = [C.c_uint16]
        L.or_bf16_to_f32.restype = C.c_float
        L.or_bf16_to_f32.argtypes = [C.c_uint16]
        L.or_bf16_rne.restype = C.c_uint16
        L.or_bf16_rne.argtypes = [C.c_float]
        L.or_bf16_rne_f64.restype = C.c_uint16
        L.or_bf16_rne_f64.argtypes = [C.c_double]
        L.or_e4m3_to_f32.restype = C.c_float
        L.or_e4m3_to_f32.argtypes = [C.c_uint8]
        L.or_e8m0_to_f32.restype = C.c_float
        L.or_e8m0_to_f32.argtypes = [C.c_uint8]
        L.or_sigmoid.restype = C.c_float
        L.or_sigmoid.argtypes = [C.c_float]
        L.or_dequant_q2k.argtypes = [P, i64, P]
        L.or_dequant_q8_0.argtypes = [P, i64, P]
        L.or_engram_gather.argtypes = [P, P, i32, P, i32, i32, P, P]
        L.or_route.argtypes = [P, P, P, i32, i32, i32, i32, P, P, P, P]
        L.or_sqrt_softplus.restype = C.c_float
        L.or_sqrt_softplus.argtypes = [C.c_float]
        L.or_route_ex.argtypes = [P, P, P, i32, i32, i32, i32, i32, P, P, P, P, i32, P, P, P]
        L.or_permute.argtypes = [P, i32, i32, i32, P, P, P, P, P, P]
        L.or_engram_kv.argtypes = [P, P, i32, i32, i32, P]
        L.or_engram_gate.argtypes = [P, P, P, P, P, i32, i32, C.c_double, P]
        L.or_expert_ffn.argtypes = [i32, P, P, P, i32, i32, P, i32, P]
        L.or_moe_layer.restype = C.c_int
        L.or_moe_layer.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P, P, i32, P, P, P, P]
        L.or_residual.argtypes = [P, P, i32, i32, C.c_float, P]
        L.or_rmsnorm.argtypes = [P, i32, i32, C.c_float, P]
        _lib = L
    return _lib


def _np(a, dtype=None):
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu()
        if a.dtype == torch.bfloat16:
            a = a.view(torch.int16)
        a = a.numpy()
    a = np.ascontiguousarray(a)
    if dtype is not None:
        a = a.view(dtype) if a.dtype.itemsize == np.dtype(dtype).itemsize else a.astype(dtype)
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def bf16_bits(x) -> np.ndarray:
    """BF16 tensor -> uint16 numpy bit patterns."""
    return _np(x, np.uint16)


# --------------------------------------------------------------------------- #

def dequant_q2k(blocks) -> np.ndarray:
    b = _np(blocks, np.uint8).reshape(-1)
    n = b.size // 84
    out = np.empty(n * 256, dtype=np.float32)
    lib().or_dequant_q2k(_p(b), n, _p(out))
    return out


def dequant_q8_0(blocks) -> np.ndarray:
    b = _np(blocks, np.uint8).reshape(-1)
    n = b.size // 34
    out = np.empty(n * 32, dtype=np.float32)
    lib().or_dequant_q8_0(_p(b), n, _p(out))
    return out


def engram_gather(tables, ids) -> tuple[np.ndarray, int]:
    """tables: list of uint8 [n_rows, 264]; ids int64 [T, n_tables, H] -> (uint16 [T, n_tables*256], err)."""
    tabs = [_np(t, np.uint8) for t in tables]
    ids = _np(ids, np.int64)
    T, nt, H = ids.shape
    assert nt == len(tabs)
    ptrs = (C.c_void_p * nt)(*[t.ctypes.data for t in tabs])
    nrows = np.array([t.shape[0] for t in tabs], dtype=np.int64)
    out = np.empty((T, nt * 256), dtype=np.uint16)
    err = np.zeros(1, dtype=np.int32)
    lib().or_engram_gather(C.cast(ptrs, C.c_void_p), _p(nrows), nt, _p(ids), T, H, _p(out), _p(err))
    return out, int(err[0])


def route(x, w_r, bias, k: int, want_scores: bool = False):
    xb = bf16_bits(x)
    T, d = xb.shape
    wr = _np(w_r, np.float32)
    E = wr.shape[1]
    b = None if bias is None else _np(bias, np.float32)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    z = np.empty((T, E), dtype=np.float32) if want_scores else None
    s = np.empty((T, E), dtype=np.float32) if want_scores else None
    lib().or_route(_p(xb), _p(wr), _p(b), T, d, E, k, _p(ids), _p(w), _p(z), _p(s))
    if want_scores:
        return ids, w, z, s
    return ids, w


def route_ex(x, w_r, bias, k: int, score: int = 0, vision_bias=None, is_media=None, tid2eid=None,
             token_ids=None):
    """Router with the per-row rule of the device router notes: score 0 sigmoid, 1 sqrt(softplus);
    media rows take vision_bias; on a hash layer (tid2eid given) text rows take tid2eid[token].
    Returns ids, weights, error word."""
    xb = bf16_bits(x)
    T, d = xb.shape
    wr = _np(w_r, np.float32)
    E = wr.shape[1]
    b = None if bias is None else _np(bias, np.float32)
    vb = None if vision_bias is None else _np(vision_bias, np.float32)
    md = None if is_media is None else np.ascontiguousarray(_np(is_media).astype(np.uint8))
    tb = None if tid2eid is None else _np(tid2eid, np.int32)
    tk = None if token_ids is None else _np(token_ids, np.int32)
    vocab = 0 if tb is None else tb.shape[0]
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    err = np.zeros(1, dtype=np.int32)
    lib().or_route_ex(_p(xb), _p(wr), _p(b), T, d, E, k, score, _p(vb), _p(md), _p(tb), _p(tk), vocab,
                      _p(ids), _p(w), _p(err))
    return ids, w, int(err[0])


def engram_kv(rows, w_kv) -> np.ndarray:
    """FP64 product of the gathered rows [T][K] (BF16) and engram_kv.weight [N][K] (BF16)."""
    rb = bf16_bits(rows)
    wb = bf16_bits(w_kv)
    T, K = rb.shape
    N = wb.shape[0]
    kv = np.empty((T, N), dtype=np.float64)
    lib().or_engram_kv(_p(rb), _p(wb), T, K, N, _p(kv))
    return kv


def engram_gate(kv, resid, q_norm, k_norm, mask=None, eps: float = 1e-6):
    """Gate and residual injection on four hyper-connection branches: returns (new residual
    [T][4][W] as BF16 bits, gates [T][4] in FP64)."""
    kv = np.ascontiguousarray(np.asarray(kv, dtype=np.float64))
    r = bf16_bits(resid).copy()
    T = r.shape[0]
    W = r.shape[-1]
    qn = _np(q_norm, np.float32)
    kn = _np(k_norm, np.float32)
    m = None if mask is None else np.ascontiguousarray(_np(mask).astype(np.uint8))
    g = np.empty((T, 4), dtype=np.float64)
    lib().or_engram_gate(_p(kv), _p(r), _p(qn), _p(kn), _p(m), T, W, eps, _p(g))
    return r, g


def permute(ids, E: int):
    ids = _np(ids, np.int32)
    T, k = ids.shape
    P = T * k
    offsets = np.empty(E + 1, dtype=np.int32)
    perm = np.empty(P, dtype=np.int32)
    inv = np.empty(P, dtype=np.int32)
    active = np.empty(E, dtype=np.int32)
    n_active = np.zeros(1, dtype=np.int32)
    err = np.zeros(1, dtype=np.int32)
    lib().or_permute(_p(ids), T, k, E, _p(offsets), _p(perm), _p(inv), _p(active), _p(n_active), _p(err))
    return dict(offsets=offsets, perm=perm, inv=inv, active=active[:n_active[0]], n_active=int(n_active[0]),
                err=int(err[0]))


def expert_ffn(fmt: int, gate, up, down, d: int, F: int, xs) -> np.ndarray:
    g, u, dn = (_np(a, np.uint8) for a in (gate, up, down))
    xb = bf16_bits(xs).reshape(-1, d)
    n = xb.shape[0]
    y = np.empty((n, d), dtype=np.float64)
    lib().or_expert_ffn(fmt, _p(g), _p(u), _p(dn), d, F, _p(xb), n, _p(y))
    return y


def moe_layer(x, w_r, bias, k: int, F: int, gate_e, up_e, down_e, sh_gate=None, sh_up=None, sh_down=None,
              F_shared: int = 0):
    """One MoE layer.  gate_e/up_e/down_e: sequence of E per-expert byte arrays (None if unused).

    Returns dict(out=uint16 [T,d] bf16 bits, out_f64=[T,d], ids, w)."""
    xb = bf16_bits(x)
    T, d = xb.shape
    wr = _np(w_r, np.float32)
    E = wr.shape[1]
    b = None if bias is None else _np(bias, np.float32)
    keep = []

    def ptrs(seq):
        arr = (C.c_void_p * E)()
        for e, a in enumerate(seq):
            if a is not None:
                a = _np(a, np.uint8)
                keep.append(a)
                arr[e] = a.ctypes.data
        keep.append(arr)
        return C.cast(arr, C.c_void_p)

    sg = su = sd = None
    if F_shared:
        sg, su, sd = (_np(a, np.uint8) for a in (sh_gate, sh_up, sh_down))
    out = np.empty((T, d), dtype=np.uint16)
    out64 = np.empty((T, d), dtype=np.float64)
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float32)
    rc = lib().or_moe_layer(_p(xb), T, d, E, k, F, _p(wr), _p(b), ptrs(gate_e), ptrs(up_e), ptrs(down_e),
                            _p(sg), _p(su), _p(sd), F_shared, _p(out), _p(out64), _p(ids), _p(w))
    if rc != 0:
        raise ValueError("oracle: a selected expert's weights were not supplied")
    return dict(out=out, out_f64=out64, ids=ids, w=w)


def residual(x, moe, scale: float) -> np.ndarray:
    xb, mb = bf16_bits(x), bf16_bits(moe)
    T, d = xb.shape
    out = np.empty((T, d), dtype=np.uint16)
    lib().or_residual(_p(xb), _p(mb), T, d, scale, _p(out))
    return out


def rmsnorm(x, eps: float = 1e-6) -> np.ndarray:
    xb = bf16_bits(x)
    T, d = xb.shape
    out = np.empty((T, d), dtype=np.uint16)
    lib().or_rmsnorm(_p(xb), T, d, eps, _p(out))
    return out
