"""Seeded synthetic inputs for the routed-expert MoE layer and the Engram gather.

This module holds no arithmetic of the method itself: it only draws random
numbers and lays them out in the byte formats the kernels and the oracle
consume.  Both sides read the bytes it produces; neither side calls the other.

Generator
---------
Every draw is ``splitmix64`` in counter mode: the 64-bit word number ``i`` of
stream ``s`` under seed ``seed`` is ``mix64(key(seed, s) + (i + 1) * GAMMA)``
with ``key(seed, s) = mix64(seed ^ (s * GAMMA))``.  Any word can therefore be
regenerated on its own, so expert blocks or Engram rows can be produced for one
expert or one id list without materialising a whole table.  The integer-only
parts run with identical results on the CPU and on a CUDA device (torch int64
arithmetic wraps modulo 2**64); floating draws that use ``log``/``cos``
(normals) are produced on the CPU only.

Byte layouts produced here
--------------------------
* Q2_K block, 84 B per 256 weights: ``scales[16]`` (low nibble = scale, high
  nibble = min), ``qs[64]`` (2-bit codes), fp16 ``d``, fp16 ``dmin``.  Field
  order and distributions follow the MoE configuration text (codes and nibbles
  uniform, ``d ~ U(0.001, 0.01)``, ``dmin ~ U(0, 0.005)``).  Total size agrees
  with the Q2_K down-projection bytes of the strix-llama.cpp issue
  ("Published-GGUF header-only capacity result": 3,870,720 B = 46,080 x 84 B).
* Q8_0 block, 34 B per 32 weights: fp16 ``d`` then ``int8 q[32]``; ``q`` uniform
  in [-127, 127], ``d ~ U(0.0005, 0.0015)`` (the shared expert's distribution is
  not given anywhere; this is a stated reading).
* Engram row, 264 B: 256 E4M3 bytes uniform over the 254 finite codes, then 8
  E8M0 scale bytes uniform in 120..134 (strix-llama.cpp issue, "Feature
  Description": 256 native E4M3 values plus 8 E8M0 scales).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

GAMMA = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1

Q2K_BLOCK_BYTES = 84
Q8_0_BLOCK_BYTES = 34
ENGRAM_ROW_BYTES = 264
Q2K_WORDS = 12      # 10 words of scale/code bytes, 1 for d, 1 for dmin
Q8_0_WORDS = 9      # 8 words of 16-bit lanes for q, 1 for d
ENGRAM_WORDS = 66   # 264 16-bit lanes

# stream ids (tensor kinds); layer and set numbers are folded in by stream()
S_X, S_WR, S_BIAS, S_GATE, S_UP, S_DOWN, S_SGATE, S_SUP, S_SDOWN = range(1, 10)
S_ENGRAM_TABLE, S_ENGRAM_IDS, S_TOKENS, S_ZIPF_PERM = 16, 24, 25, 26
S_EKV, S_ENORM, S_ERESID = 27, 28, 29


def stream(kind: int, layer: int = 0, sub: int = 0) -> int:
    """Stream number for tensor ``kind`` of ``layer`` (``sub`` = token set or table)."""
    return (kind & 0xFF) | ((layer & 0xFFFF) << 8) | ((sub & 0xFFFF) << 24)


def _s64(c: int) -> int:
    c &= MASK64
    return c - (1 << 64) if c >= (1 << 63) else c


def _mix64_int(z: int) -> int:
    z &= MASK64
    z ^= z >> 30
    z = (z * M1) & MASK64
    z ^= z >> 27
    z = (z * M2) & MASK64
    z ^= z >> 31
    return z


def _key(seed: int, s: int) -> int:
    return _mix64_int((seed ^ ((s * GAMMA) & MASK64)) & MASK64)


def u64_py(seed: int, s: int, i: int) -> int:
    """Pure-Python reference of word ``i`` of stream ``s`` (used to check the torch path)."""
    return _mix64_int((_key(seed, s) + (i + 1) * GAMMA) & MASK64)


def _shr(z: torch.Tensor, n: int) -> torch.Tensor:
    # logical right shift on int64
    return (z >> n) & ((1 << (64 - n)) - 1)


def _mix64_t(z: torch.Tensor) -> torch.Tensor:
    z = z ^ _shr(z, 30)
    z = z * _s64(M1)
    z = z ^ _shr(z, 27)
    z = z * _s64(M2)
    z = z ^ _shr(z, 31)
    return z


def u64_at(seed: int, s: int, idx: torch.Tensor) -> torch.Tensor:
    """Words ``idx`` (int64 tensor, any device) of stream ``s``; returns int64 bit patterns."""
    k = _key(seed, s)
    z = (idx + 1) * _s64(GAMMA) + _s64(k)
    return _mix64_t(z)


def u64(seed: int, s: int, start: int, count: int, device="cpu") -> torch.Tensor:
    idx = torch.arange(start, start + count, dtype=torch.int64, device=device)
    return u64_at(seed, s, idx)


def _unit_double(w: torch.Tensor) -> torch.Tensor:
    """Top 53 bits as a double in [0, 1): exact, no library math."""
    return _shr(w, 11).to(torch.float64) * (2.0 ** -53)


def _lanes16(w: torch.Tensor) -> torch.Tensor:
    """Split int64 words [..., n] into 16-bit lanes [..., 4n] (little-endian order), as int64."""
    parts = [(_shr(w, 16 * j) & 0xFFFF) for j in range(4)]
    return torch.stack(parts, dim=-1).reshape(*w.shape[:-1], w.shape[-1] * 4)


def _f16_bits(v: torch.Tensor) -> torch.Tensor:
    """fp16 (RNE) bit pattern of a float64 tensor, as uint8 [..., 2] little-endian."""
    return v.to(torch.float16).view(torch.uint8).reshape(*v.shape, 2)


# --------------------------------------------------------------------------- #
# quantised expert blocks
# --------------------------------------------------------------------------- #

def q2k_blocks(seed: int, s: int, block_start: int, nblocks: int, device="cpu",
               chunk: int = 1 << 22) -> torch.Tensor:
    """Q2_K blocks ``block_start .. block_start+nblocks`` of stream ``s`` -> uint8 [nblocks, 84]."""
    out = torch.empty((nblocks, Q2K_BLOCK_BYTES), dtype=torch.uint8, device=device)
    for c0 in range(0, nblocks, chunk):
        n = min(chunk, nblocks - c0)
        w = u64(seed, s, (block_start + c0) * Q2K_WORDS, n * Q2K_WORDS, device).view(n, Q2K_WORDS)
        out[c0:c0 + n, :80] = w[:, :10].contiguous().view(torch.uint8).view(n, 80)
        d = 0.001 + 0.009 * _unit_double(w[:, 10])
        dmin = 0.005 * _unit_double(w[:, 11])
        out[c0:c0 + n, 80:82] = _f16_bits(d)
        out[c0:c0 + n, 82:84] = _f16_bits(dmin)
    return out


def q8_0_blocks(seed: int, s: int, block_start: int, nblocks: int, device="cpu",
                chunk: int = 1 << 22) -> torch.Tensor:
    """Q8_0 blocks of stream ``s`` -> uint8 [nblocks, 34] (fp16 d, then int8 q[32])."""
    out = torch.empty((nblocks, Q8_0_BLOCK_BYTES), dtype=torch.uint8, device=device)
    for c0 in range(0, nblocks, chunk):
        n = min(chunk, nblocks - c0)
        w = u64(seed, s, (block_start + c0) * Q8_0_WORDS, n * Q8_0_WORDS, device).view(n, Q8_0_WORDS)
        q = (_lanes16(w[:, :8]) % 255) - 127                       # [n, 32] in [-127, 127]
        d = 0.0005 + 0.001 * _unit_double(w[:, 8])
        out[c0:c0 + n, 0:2] = _f16_bits(d)
        out[c0:c0 + n, 2:34] = q.to(torch.int8).view(torch.uint8)
    return out


_FINITE_E4M3 = torch.tensor([b for b in range(256) if (b & 0x7F) != 0x7F], dtype=torch.int64)


def engram_rows_at(seed: int, s: int, rows: torch.Tensor) -> torch.Tensor:
    """Engram rows with the given row numbers (int64 tensor) -> uint8 [len, 264]."""
    dev = rows.device
    w = u64_at(seed, s, rows.reshape(-1, 1) * ENGRAM_WORDS
               + torch.arange(ENGRAM_WORDS, dtype=torch.int64, device=dev))
    lanes = _lanes16(w)                                            # [n, 264]
    fin = _FINITE_E4M3.to(dev)
    vals = fin[lanes[:, :256] % 254]
    scl = 120 + lanes[:, 256:] % 15
    return torch.cat([vals, scl], dim=1).to(torch.uint8)


def engram_table(seed: int, s: int, nrows: int, device="cpu", chunk: int = 1 << 20) -> torch.Tensor:
    out = torch.empty((nrows, ENGRAM_ROW_BYTES), dtype=torch.uint8, device=device)
    for r0 in range(0, nrows, chunk):
        n = min(chunk, nrows - r0)
        out[r0:r0 + n] = engram_rows_at(seed, s, torch.arange(r0, r0 + n, dtype=torch.int64, device=device))
    return out


# --------------------------------------------------------------------------- #
# floating draws (CPU)
# --------------------------------------------------------------------------- #

def uniform(seed: int, s: int, n: int, lo: float, hi: float, start: int = 0) -> torch.Tensor:
    """float64 uniforms in [lo, hi) (CPU)."""
    return lo + (hi - lo) * _unit_double(u64(seed, s, start, n))


def normal(seed: int, s: int, n: int, std: float = 1.0, start: int = 0) -> torch.Tensor:
    """float64 N(0, std^2) by Box-Muller in double (CPU), words 2i and 2i+1 per value."""
    w = u64(seed, s, 2 * start, 2 * n).view(n, 2)
    u1 = (_shr(w[:, 0], 11).to(torch.float64) + 1.0) * (2.0 ** -53)     # (0, 1]
    u2 = _unit_double(w[:, 1])
    return std * torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(2.0 * math.pi * u2)


def x_bf16(seed: int, layer: int, tset: int, T: int, d: int) -> torch.Tensor:
    """Activations x ~ N(0, 1) rounded to BF16 (RNE), [T, d]."""
    return normal(seed, stream(S_X, layer, tset), T * d).to(torch.float32).to(torch.bfloat16).view(T, d)


def engram_kv_weight(seed: int, layer: int, N: int, K: int, std: float = 1e-5, device="cpu") -> torch.Tensor:
    """engram_kv.weight ~ N(0, std^2) rounded to BF16, [N = 5 W outputs][K = R * 256 inputs].  The
    decoded Engram rows reach magnitudes of ~1e4 (e4m3 up to 448 times scales up to 2^7), so a
    small std keeps the keys and the value near unit size."""
    return normal(seed, stream(S_EKV, layer), N * K, std).to(torch.float32).to(torch.bfloat16).view(N, K).to(device)


def engram_norm_weights(seed: int, layer: int, which: int, W: int) -> torch.Tensor:
    """q_norm (which = 0) / k_norm (1) of the four hyper-connection branches: 1 + N(0, 0.1^2), FP32 [4, W]."""
    return (1.0 + normal(seed, stream(S_ENORM, layer, which), 4 * W, 0.1)).to(torch.float32).view(4, W)


def engram_residual(seed: int, layer: int, tset: int, T: int, W: int) -> torch.Tensor:
    """The four hyper-connection residual branches ~ N(0, 1) rounded to BF16, [T, 4, W]."""
    return normal(seed, stream(S_ERESID, layer, tset), T * 4 * W).to(torch.float32).to(torch.bfloat16).view(T, 4, W)


def router_weight(seed: int, layer: int, d: int, E: int) -> torch.Tensor:
    """W_r ~ N(0, 0.02^2), FP32, [d, E] row-major."""
    return normal(seed, stream(S_WR, layer), d * E, 0.02).to(torch.float32).view(d, E)


def zipf_log_popularity(seed: int, layer: int, E: int, s_exp: float = 1.1) -> torch.Tensor:
    """ln p_e with p_e = r_e^-s / sum_r r^-s and r_e = 1 + (position of e in a seeded permutation)."""
    keys = _shr(u64(seed, stream(S_ZIPF_PERM, layer), 0, E), 11)
    perm = torch.argsort(keys, stable=True)                      # perm[r] = expert at rank r+1
    rank = torch.empty(E, dtype=torch.int64)
    rank[perm] = torch.arange(E)
    r = (rank + 1).to(torch.float64)
    norm = torch.sum(torch.arange(1, E + 1, dtype=torch.float64) ** (-s_exp))
    return (-s_exp) * torch.log(r) - torch.log(norm)


def route_bias(seed: int, layer: int, E: int, half_width: float, zipf: float | None = None) -> torch.Tensor:
    """b ~ U(-w, w) (+ ln p_e for the Zipf-skewed prefill), FP32 [E]."""
    b = uniform(seed, stream(S_BIAS, layer), E, -half_width, half_width)
    if zipf is not None:
        b = b + zipf_log_popularity(seed, layer, E, zipf)
    return b.to(torch.float32)


# --------------------------------------------------------------------------- #
# Engram row ids
# --------------------------------------------------------------------------- #

ENGRAM_VOCAB = 129280     # token ids uniform in [0, 129280); the same value is the pad token
ENGRAM_PAD = 129280


def engram_ids_uniform(seed: int, n: int, n_rows: int) -> torch.Tensor:
    w = u64(seed, stream(S_ENGRAM_IDS), 0, n)
    return (_shr(w, 1) % n_rows).to(torch.int64)


def engram_ids_ngram(seed: int, T: int, n_tables: int, H: int, n_rows: int) -> np.ndarray:
    """Row ids [T, n_tables, H] from a seeded 64-bit multiplicative hash of token n-grams.

    The pages do not give the Engram hash.  Stand-in: tokens uniform in
    [0, 129280); head h uses n = 2 for h < H/2, else 3; positions before the
    start read the pad token; x = mix64(seed ^ (tau*H + h)); per gram token,
    oldest first, x = (x ^ tok) * GAMMA mod 2**64; row = (x >> 32) mod n_rows.
    """
    w = u64(seed, stream(S_TOKENS), 0, T).numpy().view(np.uint64)
    tok = (w % np.uint64(ENGRAM_VOCAB)).astype(np.uint64)
    pad = np.uint64(ENGRAM_PAD)
    ids = np.empty((T, n_tables, H), dtype=np.int64)
    g = np.uint64(GAMMA)
    with np.errstate(over="ignore"):
        for tau in range(n_tables):
            for h in range(H):
                n = 2 if h < H // 2 else 3
                x = np.full(T, np.uint64(_mix64_int(seed ^ (tau * H + h))), dtype=np.uint64)
                for back in range(n - 1, -1, -1):           # oldest token first
                    src = np.full(T, pad, dtype=np.uint64)
                    src[back:] = tok[:T - back] if back else tok
                    x = (x ^ src) * g
                ids[:, tau, h] = ((x >> np.uint64(32)) % np.uint64(n_rows)).astype(np.int64)
    return ids


# --------------------------------------------------------------------------- #
# workload descriptions
# --------------------------------------------------------------------------- #

@dataclass
class MoeShape:
    d: int
    E: int
    k: int
    F: int
    F_shared: int
    bias_half_width: float
    zipf: float | None = None

    @property
    def gate_row_bytes(self) -> int:
        return (self.d // 256) * Q2K_BLOCK_BYTES

    @property
    def down_row_bytes(self) -> int:
        return (self.F // 256) * Q2K_BLOCK_BYTES

    @property
    def expert_gate_bytes(self) -> int:
        return self.F * self.gate_row_bytes

    @property
    def expert_down_bytes(self) -> int:
        return self.d * self.down_row_bytes

    @property
    def expert_bytes(self) -> int:
        return 2 * self.expert_gate_bytes + self.expert_down_bytes

    @property
    def shared_bytes(self) -> int:
        if not self.F_shared:
            return 0
        return 2 * self.F_shared * (self.d // 32) * Q8_0_BLOCK_BYTES + self.d * (self.F_shared // 32) * Q8_0_BLOCK_BYTES


TINY = MoeShape(d=512, E=32, k=6, F=256, F_shared=256, bias_half_width=0.1)
V41 = MoeShape(d=4096, E=384, k=6, F=2048, F_shared=2048, bias_half_width=0.5)
V41_PREFILL = MoeShape(d=4096, E=384, k=6, F=2048, F_shared=2048, bias_half_width=0.5, zipf=1.1)


@dataclass
class LayerWeights:
    """One MoE layer's inputs; ``gate``/``up``/``down`` are [E, rows, row_bytes] uint8."""
    shape: MoeShape
    layer: int
    w_r: torch.Tensor
    bias: torch.Tensor
    gate: torch.Tensor | None = None
    up: torch.Tensor | None = None
    down: torch.Tensor | None = None
    sh_gate: torch.Tensor | None = None
    sh_up: torch.Tensor | None = None
    sh_down: torch.Tensor | None = None
    extra: dict = field(default_factory=dict)


def expert_matrix(seed: int, layer: int, kind: int, shape: MoeShape, e0: int, ne: int, device="cpu") -> torch.Tensor:
    """Q2_K bytes of experts e0..e0+ne of one routed matrix (kind S_GATE/S_UP/S_DOWN) -> [ne, rows, row_bytes]."""
    if kind == S_DOWN:
        rows, nb = shape.d, shape.F // 256
    else:
        rows, nb = shape.F, shape.d // 256
    blocks_per_expert = rows * nb
    b = q2k_blocks(seed, stream(kind, layer), e0 * blocks_per_expert, ne * blocks_per_expert, device)
    return b.view(ne, rows, nb * Q2K_BLOCK_BYTES)


def shared_matrix(seed: int, layer: int, kind: int, shape: MoeShape, device="cpu") -> torch.Tensor:
    """Q8_0 bytes of one shared-expert matrix (kind S_SGATE/S_SUP/S_SDOWN) -> [rows, row_bytes]."""
    if kind == S_SDOWN:
        rows, nb = shape.d, shape.F_shared // 32
    else:
        rows, nb = shape.F_shared, shape.d // 32
    b = q8_0_blocks(seed, stream(kind, layer), 0, rows * nb, device)
    return b.view(rows, nb * Q8_0_BLOCK_BYTES)


def layer_weights(seed: int, layer: int, shape: MoeShape, device="cpu", experts: bool = True) -> LayerWeights:
    lw = LayerWeights(shape=shape, layer=layer,
                      w_r=router_weight(seed, layer, shape.d, shape.E),
                      bias=route_bias(seed, layer, shape.E, shape.bias_half_width, shape.zipf))
    if experts:
        lw.gate = expert_matrix(seed, layer, S_GATE, shape, 0, shape.E, device)
        lw.up = expert_matrix(seed, layer, S_UP, shape, 0, shape.E, device)
        lw.down = expert_matrix(seed, layer, S_DOWN, shape, 0, shape.E, device)
    if shape.F_shared:
        lw.sh_gate = shared_matrix(seed, layer, S_SGATE, shape, device)
        lw.sh_up = shared_matrix(seed, layer, S_SUP, shape, device)
        lw.sh_down = shared_matrix(seed, layer, S_SDOWN, shape, device)
    return lw
