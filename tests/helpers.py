"""Shared test helpers: device-resident synthetic layers and the oracle on the same bytes."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bit_routed_expert_gb300 import api, synth
from bit_routed_expert_gb300.api import BRE_FMT_Q8_0, FfnWeights, MoeLayer


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(u16: np.ndarray) -> np.ndarray:
    return torch.from_numpy(u16.astype(np.uint16).view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def device_layer(seed: int, layer: int, shape: synth.MoeShape, T_max: int, dev, with_shared: bool = True) -> MoeLayer:
    lw = synth.layer_weights(seed, layer, shape, device=dev)
    routed = api.routed_weights(lw.gate, lw.up, lw.down, shape.d, shape.F)
    shared = None
    if with_shared and shape.F_shared:
        shared = FfnWeights(lw.sh_gate, lw.sh_up, lw.sh_down, BRE_FMT_Q8_0, shape.d, shape.F_shared)
    return MoeLayer(lw.w_r.to(dev), lw.bias.to(dev), routed, shared, shape.k, T_max)


def oracle_layer(seed: int, layer: int, shape: synth.MoeShape, x: torch.Tensor, with_shared: bool = True,
                 ids_hint=None, bias=None, threads: int = 1):
    """Oracle MoE layer on CPU; experts are generated only for the experts the oracle's router selects.
    bias: overrides the shape's route bias.  threads > 1 splits the tokens into that many chunks run
    on threads (the oracle is plain C without shared state, and ctypes releases the GIL; each token's
    output depends on that token alone)."""
    w_r = synth.router_weight(seed, layer, shape.d, shape.E)
    if bias is None:
        bias = synth.route_bias(seed, layer, shape.E, shape.bias_half_width, shape.zipf)
    ids, _ = oracle.route(x, w_r, bias, shape.k)
    need = sorted(set(int(e) for e in ids.reshape(-1)))
    gate, up, down = [None] * shape.E, [None] * shape.E, [None] * shape.E
    for e in need:
        gate[e] = synth.expert_matrix(seed, layer, synth.S_GATE, shape, e, 1)[0].numpy()
        up[e] = synth.expert_matrix(seed, layer, synth.S_UP, shape, e, 1)[0].numpy()
        down[e] = synth.expert_matrix(seed, layer, synth.S_DOWN, shape, e, 1)[0].numpy()
    sg = su = sd = None
    Fs = 0
    if with_shared and shape.F_shared:
        sg = synth.shared_matrix(seed, layer, synth.S_SGATE, shape).numpy()
        su = synth.shared_matrix(seed, layer, synth.S_SUP, shape).numpy()
        sd = synth.shared_matrix(seed, layer, synth.S_SDOWN, shape).numpy()
        Fs = shape.F_shared
    x = x.cpu()
    T = x.shape[0]
    if threads <= 1 or T < 2:
        return oracle.moe_layer(x, w_r, bias, shape.k, shape.F, gate, up, down, sg, su, sd, Fs)
    import concurrent.futures as cf
    bounds = np.linspace(0, T, min(threads, T) + 1).astype(int)
    parts = [(int(a), int(b)) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]
    with cf.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        res = list(ex.map(lambda ab: oracle.moe_layer(x[ab[0]:ab[1]].contiguous(), w_r, bias, shape.k, shape.F, gate,
                                                      up, down, sg, su, sd, Fs), parts))
    return {key: np.concatenate([r[key] for r in res]) for key in res[0]}


def run_layer(layer: MoeLayer, x: torch.Tensor):
    """Layer forward on the device; returns (BF16 output, FP32 output before rounding, routing info)."""
    out_f32 = torch.empty((x.shape[0], layer.d), dtype=torch.float32, device=x.device)
    out, info = layer.forward(x, out_f32=out_f32)
    return out, out_f32, info


def assert_layer_close(out_bf16: torch.Tensor, out_f32: torch.Tensor, ref: dict, tol: float = 1e-2):
    """The FP32 layer output (before the final BF16 rounding) is within max|err| <= tol * rms(ref)
    of the oracle's FP64 value over the whole [T, d] output, and the BF16 output is exactly the
    round-to-nearest-even of that FP32 value."""
    r = ref["out_f64"]
    f = out_f32.detach().cpu().double().numpy()
    assert np.all(np.isfinite(f)), "non-finite GPU output"
    rms = float(np.sqrt(np.mean(r * r)))
    err = float(np.max(np.abs(f - r)))
    assert err <= tol * rms, f"max|err| {err:.4g} > {tol} * rms {rms:.4g}"
    rne = out_f32.detach().cpu().to(torch.bfloat16)
    assert torch.equal(out_bf16.detach().cpu().view(torch.int16), rne.view(torch.int16)), \
        "BF16 output is not the rounding of the FP32 output"
    log_error(err / rms, r.shape)
    return err / rms


def log_error(ratio: float, shape):
    """Record the achieved max|err|/rms of a layer comparison (evidence for the design notes)."""
    import inspect
    import os
    out = os.environ.get("BRE_OUT_DIR", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "out"))
    if os.path.isdir(out):
        caller = inspect.stack()[2].function
        with open(os.path.join(out, "parity_errors.txt"), "a") as f:
            f.write(f"{caller} shape={tuple(shape)} max_err/rms={ratio:.3e}\n")
