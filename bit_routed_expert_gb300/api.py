"""Python face of libbre: the C entry points under the same names, taking torch CUDA tensors.

Marshalling only (pointers, sizes, the current stream, output allocation); all
arithmetic runs in the library.  BF16 tensors may be passed as torch.bfloat16 or as
int16/uint16 bit patterns.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import BRE_FMT_Q2_K, BRE_FMT_Q2_K_R16, BRE_FMT_Q8_0, BreWeights, check, ptr, stream_handle


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


@dataclass
class FfnWeights:
    """Quantised FFN weights resident on the device: gate/up [n, F, row] and down [n, d, row] uint8."""
    gate: torch.Tensor
    up: torch.Tensor
    down: torch.Tensor
    fmt: int
    d: int
    d_ff: int

    @property
    def n_experts(self) -> int:
        return 1 if self.gate.dim() == 2 else self.gate.shape[0]

    def struct(self) -> BreWeights:
        n = self.n_experts
        return BreWeights(self.gate.data_ptr(), self.up.data_ptr(), self.down.data_ptr(), self.fmt, n, self.d,
                          self.d_ff, self.gate[0].numel() if n > 1 else 0, self.up[0].numel() if n > 1 else 0,
                          self.down[0].numel() if n > 1 else 0)


def repack_q2k_r16(blocks, stream=None):
    """Q2_K matrices, uint8 [n, rows, row_bytes] or [rows, row_bytes] on the device -> a new tensor of
    the same shape holding the Q2_K_R16 layout the expert FFN reads (bre_repack_q2k_r16)."""
    L = _lib.load()
    t = _dev(blocks, "blocks")
    n, rows, rb = (1, t.shape[0], t.shape[1]) if t.dim() == 2 else tuple(t.shape)
    out = torch.empty_like(t)
    stride = rows * rb
    check(L.bre_repack_q2k_r16(ptr(t), ptr(out), n, rows, (rb // 84) * 256, stride, stride, stream_handle(stream)),
          "bre_repack_q2k_r16")
    return out


def routed_weights(gate, up, down, d: int, d_ff: int) -> FfnWeights:
    """Routed experts given as Q2_K matrices (gate/up [E, d_ff, d/256*84], down [E, d, d_ff/256*84],
    uint8 on the device), regrouped once into the Q2_K_R16 layout moe_expert_ffn takes."""
    return FfnWeights(repack_q2k_r16(gate), repack_q2k_r16(up), repack_q2k_r16(down), BRE_FMT_Q2_K_R16, d, d_ff)


def moe_route_workspace(T: int, E: int) -> int:
    return _lib.load().moe_route_workspace(T, E)


def moe_route(x, w_r, bias, k: int, ws=None, stream=None, ids=None, w=None):
    L = _lib.load()
    T, d = x.shape
    E = w_r.shape[1]
    _dev(x, "x"), _dev(w_r, "w_r")
    if ws is None:
        ws = torch.zeros(L.moe_route_workspace(T, E), dtype=torch.uint8, device=x.device)
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    check(L.moe_route(ptr(x), ptr(w_r), ptr(bias), T, d, E, k, ptr(ids), ptr(w), ptr(ws), ws.numel(),
                      stream_handle(stream)), "moe_route")
    return ids, w


SCORE_SIGMOID = 0
SCORE_SQRT_SOFTPLUS = 1


def moe_route_ex(x, w_r, bias, k: int, score: int = SCORE_SIGMOID, vision_bias=None, is_media=None,
                 tid2eid=None, token_ids=None, ws=None, dev_err=None, stream=None, ids=None, w=None):
    """moe_route with the per-row rule of the device router notes: score, media rows with a
    vision bias, hash layers (tid2eid [vocab][k], token_ids [T]).  Returns (ids, w)."""
    L = _lib.load()
    T, d = x.shape
    E = w_r.shape[1]
    _dev(x, "x"), _dev(w_r, "w_r")
    if ws is None:
        ws = torch.zeros(L.moe_route_workspace(T, E), dtype=torch.uint8, device=x.device)
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=x.device)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=x.device)
    vocab = 0 if tid2eid is None else tid2eid.shape[0]
    check(L.moe_route_ex(ptr(x), ptr(w_r), ptr(bias), T, d, E, k, score, ptr(vision_bias), ptr(is_media),
                         ptr(tid2eid), ptr(token_ids), vocab, ptr(ids), ptr(w), ptr(dev_err), ptr(ws), ws.numel(),
                         stream_handle(stream)), "moe_route_ex")
    return ids, w


def moe_permute(ids, E: int, dev_err=None, stream=None, out=None):
    """out: optional dict of preallocated offsets [E+1], perm/inv [T*k], active [E], n_active [1]."""
    L = _lib.load()
    T, k = ids.shape
    dv = ids.device
    if out is None:
        out = dict(offsets=torch.empty(E + 1, dtype=torch.int32, device=dv),
                   perm=torch.empty(T * k, dtype=torch.int32, device=dv),
                   inv=torch.empty(T * k, dtype=torch.int32, device=dv),
                   active=torch.empty(E, dtype=torch.int32, device=dv),
                   n_active=torch.empty(1, dtype=torch.int32, device=dv))
    check(L.moe_permute(ptr(_dev(ids, "ids")), T, k, E, ptr(out["offsets"]), ptr(out["perm"]), ptr(out["inv"]),
                        ptr(out["active"]), ptr(out["n_active"]), ptr(dev_err), stream_handle(stream)), "moe_permute")
    return out


def moe_route_permute(x, w_r, bias, k: int, ws=None, dev_err=None, stream=None, ids=None, w=None, out=None):
    """moe_route then moe_permute as one call; returns (ids, w, perm dict)."""
    L = _lib.load()
    T, d = x.shape
    E = w_r.shape[1]
    _dev(x, "x"), _dev(w_r, "w_r")
    dv = x.device
    if ws is None:
        ws = torch.zeros(L.moe_route_workspace(T, E), dtype=torch.uint8, device=dv)
    if ids is None:
        ids = torch.empty((T, k), dtype=torch.int32, device=dv)
    if w is None:
        w = torch.empty((T, k), dtype=torch.float32, device=dv)
    if out is None:
        out = dict(offsets=torch.empty(E + 1, dtype=torch.int32, device=dv),
                   perm=torch.empty(T * k, dtype=torch.int32, device=dv),
                   inv=torch.empty(T * k, dtype=torch.int32, device=dv),
                   active=torch.empty(E, dtype=torch.int32, device=dv),
                   n_active=torch.empty(1, dtype=torch.int32, device=dv))
    check(L.moe_route_permute(ptr(x), ptr(w_r), ptr(bias), T, d, E, k, ptr(ids), ptr(w), ptr(out["offsets"]),
                              ptr(out["perm"]), ptr(out["inv"]), ptr(out["active"]), ptr(out["n_active"]),
                              ptr(dev_err), ptr(ws), ws.numel(), stream_handle(stream)), "moe_route_permute")
    return ids, w, out


def moe_expert_ffn_workspace(T: int, k: int, E: int, d: int, d_ff: int, d_ff_shared: int) -> int:
    return _lib.load().moe_expert_ffn_workspace(T, k, E, d, d_ff, d_ff_shared)


def moe_expert_ffn(routed: FfnWeights, shared: FfnWeights | None, x, k: int, perm: dict, ws=None, dev_err=None,
                   y_pairs=None, y_shared=None, stream=None):
    L = _lib.load()
    T, d = x.shape
    dv = x.device
    Fs = shared.d_ff if shared is not None else 0
    if ws is None:
        ws = torch.zeros(L.moe_expert_ffn_workspace(T, k, routed.n_experts, d, routed.d_ff, Fs), dtype=torch.uint8,
                         device=dv)
    if y_pairs is None:
        y_pairs = torch.zeros((T * k, d), dtype=torch.float32, device=dv)
    if shared is not None and y_shared is None:
        y_shared = torch.empty((T, d), dtype=torch.float32, device=dv)
    rs = routed.struct()
    ss = shared.struct() if shared is not None else None
    check(L.moe_expert_ffn(C.byref(rs), C.byref(ss) if ss is not None else None, ptr(_dev(x, "x")), T, k,
                           ptr(perm["offsets"]), ptr(perm["perm"]), ptr(perm["active"]), ptr(perm["n_active"]),
                           ptr(y_pairs), ptr(y_shared), ptr(ws), ws.numel(), ptr(dev_err), stream_handle(stream)),
          "moe_expert_ffn")
    return y_pairs, y_shared


def moe_combine(y_pairs, topk_w, inv, offsets, E: int, y_shared, k: int, out=None, out_f32=None, stream=None):
    """Returns the BF16 layer output; also fills out_f32 (the value before rounding) when given."""
    L = _lib.load()
    P, d = y_pairs.shape
    T = P // k
    if out is None:
        out = torch.empty((T, d), dtype=torch.bfloat16, device=y_pairs.device)
    check(L.moe_combine(ptr(y_pairs), ptr(topk_w), ptr(inv), ptr(offsets), E, ptr(y_shared), T, k, d, ptr(out),
                        ptr(out_f32), stream_handle(stream)), "moe_combine")
    return out


def moe_residual_norm(x, moe, scale: float, eps: float = 1e-6, want_norm: bool = True, stream=None):
    L = _lib.load()
    T, d = x.shape
    x_out = torch.empty_like(x)
    u_out = torch.empty_like(x) if want_norm else None
    check(L.moe_residual_norm(ptr(x), ptr(moe), T, d, scale, eps, ptr(x_out), ptr(u_out), stream_handle(stream)),
          "moe_residual_norm")
    return x_out, u_out


def engram_gather_decode(tables, ids, dev_err=None, out=None, stream=None):
    """tables: list of uint8 [n_rows, 264] CUDA tensors; ids int64 [T, n_tables, H] -> bf16 [T, n_tables*256]."""
    L = _lib.load()
    T, nt, H = ids.shape
    arr = (C.c_void_p * nt)(*[t.data_ptr() for t in tables])
    nrows = (C.c_int64 * nt)(*[t.shape[0] for t in tables])
    if out is None:
        out = torch.empty((T, nt * 256), dtype=torch.bfloat16, device=ids.device)
    check(L.engram_gather_decode(C.cast(arr, C.c_void_p), C.cast(nrows, C.c_void_p), nt, ptr(_dev(ids, "ids")), T,
                                 H, ptr(out), ptr(dev_err), stream_handle(stream)), "engram_gather_decode")
    return out


def engram_inject_workspace(T: int, R: int, W: int) -> int:
    return _lib.load().engram_inject_workspace(T, R, W)


def engram_inject(table, row_ids, w_kv, resid, q_norm, k_norm, mask=None, eps: float = 1e-6, kv_out=None,
                  gate_out=None, dev_err=None, ws=None, stream=None):
    """Engram gate and residual injection for one layer: table uint8 [n_rows, 264]; row_ids int64
    [T, R]; w_kv bf16 [5W, R*256]; resid bf16 [T, 4, W] (updated in place and returned); q_norm,
    k_norm float32 [4, W]; mask uint8 [T] or None; kv_out float32 [T, 5W] / gate_out float32
    [T, 4] optional outputs."""
    L = _lib.load()
    T, R = row_ids.shape
    W = resid.shape[-1]
    if ws is None:
        ws = torch.zeros(L.engram_inject_workspace(T, R, W), dtype=torch.uint8, device=resid.device)
    check(L.engram_inject(ptr(_dev(table, "table")), table.shape[0], ptr(_dev(row_ids, "row_ids")), R,
                          ptr(_dev(w_kv, "w_kv")), W, ptr(_dev(resid, "resid")), ptr(q_norm), ptr(k_norm), ptr(mask), T,
                          float(eps), ptr(kv_out), ptr(gate_out), ptr(dev_err), ptr(ws), ws.numel(),
                          stream_handle(stream)), "engram_inject")
    return resid


def bre_dequant(fmt: int, blocks, stream=None):
    L = _lib.load()
    bb = 84 if fmt == BRE_FMT_Q2_K else 34
    n = blocks.numel() // bb
    out = torch.empty(n * (256 if fmt == BRE_FMT_Q2_K else 32), dtype=torch.float32, device=blocks.device)
    check(L.bre_dequant(fmt, ptr(_dev(blocks, "blocks")), n, ptr(out), stream_handle(stream)), "bre_dequant")
    return out


class MoeLayer:
    """One MoE layer resident on the device, with its workspaces; forward() runs
    route + permute (one call) -> expert FFN (routed + shared) -> combine."""

    def __init__(self, w_r, bias, routed: FfnWeights, shared: FfnWeights | None, k: int, T_max: int):
        self.w_r, self.bias, self.routed, self.shared, self.k = w_r, bias, routed, shared, k
        self.E = w_r.shape[1]
        self.d = w_r.shape[0]
        dv = w_r.device
        self.T_max = T_max
        Fs = shared.d_ff if shared is not None else 0
        self.route_ws = torch.zeros(moe_route_workspace(T_max, self.E), dtype=torch.uint8, device=dv)
        self.ffn_ws = torch.zeros(moe_expert_ffn_workspace(T_max, k, self.E, self.d, routed.d_ff, Fs),
                                  dtype=torch.uint8, device=dv)
        self.y_pairs = torch.zeros((T_max * k, self.d), dtype=torch.float32, device=dv)
        self.y_shared = torch.zeros((T_max, self.d), dtype=torch.float32, device=dv) if shared is not None else None
        self.dev_err = torch.zeros(1, dtype=torch.int32, device=dv)
        # per-call outputs, preallocated so that a forward can be captured in a CUDA graph
        self.ids = torch.empty((T_max, k), dtype=torch.int32, device=dv)
        self.w = torch.empty((T_max, k), dtype=torch.float32, device=dv)
        self.perm_buf = dict(offsets=torch.empty(self.E + 1, dtype=torch.int32, device=dv),
                             perm=torch.empty(T_max * k, dtype=torch.int32, device=dv),
                             inv=torch.empty(T_max * k, dtype=torch.int32, device=dv),
                             active=torch.empty(self.E, dtype=torch.int32, device=dv),
                             n_active=torch.empty(1, dtype=torch.int32, device=dv))

    def forward(self, x, out=None, stream=None, ffn_events=None, out_f32=None):
        """ffn_events: optional (start, end) CUDA events recorded around the expert FFN call;
        out_f32: optional [T, d] FP32 tensor for the layer output before BF16 rounding."""
        T = x.shape[0]
        pb = self.perm_buf
        ids, w, perm = moe_route_permute(x, self.w_r, self.bias, self.k, ws=self.route_ws, dev_err=self.dev_err,
                                         stream=stream, ids=self.ids[:T], w=self.w[:T],
                                         out=dict(offsets=pb["offsets"], perm=pb["perm"][:T * self.k],
                                                  inv=pb["inv"][:T * self.k], active=pb["active"],
                                                  n_active=pb["n_active"]))
        s = stream if stream is not None else torch.cuda.current_stream()
        if ffn_events is not None:
            ffn_events[0].record(s)
        y_pairs, y_shared = moe_expert_ffn(self.routed, self.shared, x, self.k, perm, ws=self.ffn_ws,
                                           dev_err=self.dev_err, y_pairs=self.y_pairs[:T * self.k],
                                           y_shared=None if self.y_shared is None else self.y_shared[:T],
                                           stream=stream)
        if ffn_events is not None:
            ffn_events[1].record(s)
        out = moe_combine(y_pairs, w, perm["inv"], perm["offsets"], self.E, y_shared, self.k, out=out,
                          out_f32=out_f32, stream=stream)
        return out, dict(ids=ids, w=w, **perm)


class MoeStack:
    """A stack of MoE layers with no attention (the speculative-verify batch): per layer
    u = norm(x), x <- bf16(x + moe(u) * scale) with scale = 1/sqrt(2); the norm of the
    next layer's input is fused into the residual update (moe_residual_norm)."""

    def __init__(self, layers, scale: float | None = None, eps: float = 1e-6):
        import math
        self.layers = layers
        self.scale = float(torch.tensor(1.0 / math.sqrt(2.0), dtype=torch.float32)) if scale is None else scale
        self.eps = eps
        L0 = layers[0]
        self.zero = torch.zeros((L0.T_max, L0.d), dtype=torch.bfloat16, device=L0.w_r.device)
        self.out = torch.empty((L0.T_max, L0.d), dtype=torch.bfloat16, device=L0.w_r.device)

    def forward(self, x, trace=None, stream=None):
        """Returns the final hidden state; `trace` (a list) receives per-layer (x, u, out, info)."""
        T = x.shape[0]
        x, u = moe_residual_norm(x, self.zero[:T], 0.0, self.eps, stream=stream)
        for layer in self.layers:
            out_f32 = None
            if trace is not None:
                out_f32 = torch.empty((T, layer.d), dtype=torch.float32, device=x.device)
            out, info = layer.forward(u, out=self.out[:T], stream=stream, out_f32=out_f32)
            if trace is not None:
                trace.append((x, u, out.clone(), out_f32, info))
            x, u = moe_residual_norm(x, out, self.scale, self.eps, stream=stream)
        return x


class StepGraph:
    """A sequence of library calls captured once as a CUDA graph and replayed.

    `fn` issues the calls on the current stream (every call above does); buffers it
    touches must stay allocated while the graph is used.  Decode-size steps are a few
    tens of microseconds of GPU work, so launching them one by one from the host would
    dominate; a replay launches the whole step at once."""

    def __init__(self, fn, warmup: int = 2):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(warmup):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            fn()

    def replay(self):
        self.graph.replay()
