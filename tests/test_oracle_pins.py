"""Pins of the CPU oracle against sources other than itself (no GPU needed).

Each test checks the oracle against something independent of its code:
library decoders (numpy float16, torch float8), exact rational arithmetic,
brute force on tiny inputs, closed forms and invariants, and the byte counts
printed on the pages (tests/golden/page_sizes.json).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from bit_routed_expert_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
L = oracle.lib()


# --------------------------------------------------------------------------- #
# independent helpers (test side)
# --------------------------------------------------------------------------- #

def f32_bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def round_f32(fr: Fraction) -> float:
    """Exact round-to-nearest-even of a rational to binary32 (finite range)."""
    if fr == 0:
        return 0.0
    sign = -1.0 if fr < 0 else 1.0
    a = abs(fr)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = max(e - 23, -149)
    sc = a / (Fraction(2) ** q)
    n = sc.numerator // sc.denominator
    rem = sc - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * float(Fraction(n) * (Fraction(2) ** q))


def np_dequant_q2k(blocks: np.ndarray) -> np.ndarray:
    """Vectorised Q2_K decode written independently of the oracle (numpy float16 for d, dmin)."""
    b = blocks.reshape(-1, 84)
    sc = (b[:, :16] & 15).astype(np.float32)
    m = (b[:, :16] >> 4).astype(np.float32)
    qs = b[:, 16:80]
    codes = np.stack([(qs >> s) & 3 for s in (0, 2, 4, 6)], axis=-1).reshape(-1, 256).astype(np.float32)
    d = b[:, 80:82].copy().view(np.float16).astype(np.float32)           # [n, 1]
    dmin = b[:, 82:84].copy().view(np.float16).astype(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        dsc = np.repeat(d * sc, 16, axis=1).astype(np.float32)
        dmm = np.repeat(dmin * m, 16, axis=1).astype(np.float32)
        return (dsc * codes - dmm).astype(np.float32).reshape(-1)


def np_dequant_q8_0(blocks: np.ndarray) -> np.ndarray:
    b = blocks.reshape(-1, 34)
    d = b[:, 0:2].copy().view(np.float16).astype(np.float32)
    q = b[:, 2:].view(np.int8).astype(np.float32)
    with np.errstate(invalid="ignore", over="ignore"):
        return (d * q).astype(np.float32).reshape(-1)


def same_f32(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    return np.all(both_nan | (f32_bits(a) == f32_bits(b)))


# --------------------------------------------------------------------------- #
# page-printed sizes
# --------------------------------------------------------------------------- #

def test_page_sizes_match_formats():
    g = json.load(open(os.path.join(GOLDEN, "page_sizes.json")))
    assert g["engram_row_bytes"] == synth.ENGRAM_ROW_BYTES == g["engram_values_per_row"] + g["engram_scales_per_row"]
    # 256 E4M3 values share 8 E8M0 scales: one scale per 32 values
    assert g["engram_values_per_row"] // g["engram_scales_per_row"] == 32
    # Q2_K down projection: the published byte count divides into 84-byte blocks of 256 weights,
    # and the IQ2_XXS gate/up tensors of the same weight count into 66-byte blocks
    nblk = g["down_bytes_per_expert_layer"] // synth.Q2K_BLOCK_BYTES
    assert nblk * synth.Q2K_BLOCK_BYTES == g["down_bytes_per_expert_layer"]
    assert g["gate_bytes_per_expert_layer"] == nblk * 66
    assert g["slot_bytes_all_layers"] == g["layers"] * (
        g["gate_bytes_per_expert_layer"] + g["up_bytes_per_expert_layer"] + g["down_bytes_per_expert_layer"])
    blk = synth.q2k_blocks(1, 5, 0, 3)
    assert blk.shape == (3, 84)
    assert oracle.dequant_q2k(blk).size == 3 * g["q2k_block_weights"]


# --------------------------------------------------------------------------- #
# scalar formats
# --------------------------------------------------------------------------- #

def test_fp16_decode_exhaustive():
    allh = np.arange(65536, dtype=np.uint16)
    ref = allh.view(np.float16).astype(np.float32)
    got = np.array([L.or_f16_to_f32(int(h)) for h in allh], dtype=np.float32)
    assert same_f32(got, ref)


def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32)
    edge = np.array([0, 0x80000000, 0x7F7FFFFF, 0x7F7F8000, 0x7F7F7FFF, 0x00000001, 0x00008000, 0x00018000,
                     0x3F808000, 0x3F818000, 0x3F807FFF, 0x7F800000, 0xFF800000], dtype=np.uint32)
    bits = np.concatenate([bits, edge])
    f = bits.view(np.float32)
    finite = ~np.isnan(f)
    ref = torch.from_numpy(f[finite].copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([L.or_bf16_rne(float(v)) for v in f[finite]], dtype=np.uint16)
    assert np.array_equal(got, ref)
    for v in f[~finite][:50]:
        assert L.or_bf16_rne(float(v)) == 0x7FC0


def _bf16_nearest_exact(x: float) -> int:
    """Nearest-even bf16 of a double by exact rational comparison of the two neighbours."""
    fx = Fraction(x)
    f32 = np.float32(x)                      # some float near x
    hi16 = int(f32_bits(f32)) >> 16
    cands = []
    for h in range(max(hi16 - 2, 0), hi16 + 3):
        for s in (0, 0x8000):
            hb = (h & 0x7FFF) | s
            v = np.uint32(hb << 16).view(np.float32)
            if np.isfinite(v):
                cands.append((abs(Fraction(float(v)) - fx), hb & 1, hb))
    cands.sort()
    best = [c for c in cands if c[0] == cands[0][0]]
    best.sort(key=lambda c: c[1])             # ties: even mantissa
    return best[0][2]


def test_bf16_rne_from_double_single_rounding():
    rng = np.random.default_rng(4)
    xs = list(rng.standard_normal(3000) * 10.0 ** rng.integers(-6, 6, 3000))
    # halfway between two bf16 values, then one double ulp above / below: a double->float->bf16
    # chain rounds these wrongly; a single rounding must not
    for b in (0x3F80, 0x4123, 0xC0F1, 0x3A01):
        lo = float(np.uint32(b << 16).view(np.float32))
        hi = float(np.uint32((b + 1) << 16).view(np.float32))
        mid = (lo + hi) / 2
        xs += [mid, math.nextafter(mid, math.inf), math.nextafter(mid, -math.inf)]
        f = float(np.float32(mid))
        xs += [math.nextafter(f, math.inf), math.nextafter(f, -math.inf)]
    for x in xs:
        assert L.or_bf16_rne_f64(x) == _bf16_nearest_exact(x), x


def test_e4m3_exhaustive_vs_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float().numpy()
    got = np.array([L.or_e4m3_to_f32(int(c)) for c in range(256)], dtype=np.float32)
    assert same_f32(got, ref)
    # closed-form anchors of OCP E4M3
    assert L.or_e4m3_to_f32(0x7E) == 448.0 and L.or_e4m3_to_f32(0x01) == 2.0 ** -9
    assert L.or_e4m3_to_f32(0x08) == 2.0 ** -6 and L.or_e4m3_to_f32(0x38) == 1.0
    assert math.isnan(L.or_e4m3_to_f32(0x7F)) and math.isnan(L.or_e4m3_to_f32(0xFF))
    assert math.copysign(1.0, L.or_e4m3_to_f32(0x80)) == -1.0


def test_e8m0_exhaustive():
    for e in range(255):
        assert L.or_e8m0_to_f32(e) == math.ldexp(1.0, e - 127)
    assert math.isnan(L.or_e8m0_to_f32(255))
    if hasattr(torch, "float8_e8m0fnu"):
        ref = torch.arange(255, dtype=torch.uint8).view(torch.float8_e8m0fnu).float().numpy()
        got = np.array([L.or_e8m0_to_f32(e) for e in range(255)], dtype=np.float32)
        assert same_f32(got, ref)


# --------------------------------------------------------------------------- #
# Engram rows
# --------------------------------------------------------------------------- #

def _all_pairs_table():
    """256 rows covering every (E4M3 code, E8M0 byte) pair once per 32-value slice."""
    rows = np.zeros((256, 264), dtype=np.uint8)
    for r in range(32):
        for rot in range(8):
            i = r * 8 + rot
            rows[i, :256] = (np.arange(256) + 32 * rot) % 256
            rows[i, 256:] = np.arange(8 * r, 8 * r + 8)
    return rows


def test_engram_decode_exhaustive_pairs():
    tab = _all_pairs_table()
    ids = np.arange(256, dtype=np.int64).reshape(256, 1, 1)
    out, err = oracle.engram_gather([tab], ids)
    assert err == 0
    v = torch.from_numpy(tab[:, :256].copy()).view(torch.float8_e4m3fn).float().numpy()
    scl = np.array([[math.ldexp(1.0, int(e) - 127) if e < 255 else math.nan for e in row] for row in tab[:, 256:]],
                   dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        prod = (v.astype(np.float64) * np.repeat(scl, 32, axis=1)).astype(np.float32)
    # the product of a <=4-bit significand and a power of two is exact in float (or overflows)
    ref = torch.from_numpy(prod).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    ref[np.isnan(prod)] = 0x7FC0
    assert np.array_equal(out, ref)
    # every (code, scale) pair appears
    pairs = set()
    for i in range(256):
        for c in range(256):
            pairs.add((int(tab[i, c]), int(tab[i, 256 + c // 32])))
    assert len(pairs) == 65536


def test_engram_head_sum_order():
    # 8 heads of one table, values of very different magnitude so that the float
    # sum depends on its order
    rng = np.random.default_rng(7)
    tab = synth.engram_table(11, synth.stream(synth.S_ENGRAM_TABLE), 64).numpy()
    tab[:, 256:] = rng.integers(110, 145, (64, 8))
    ids = rng.integers(0, 64, (40, 1, 8)).astype(np.int64)
    out, err = oracle.engram_gather([tab], ids)
    assert err == 0
    dec = torch.from_numpy(tab[:, :256].copy()).view(torch.float8_e4m3fn).float().numpy() * \
        np.repeat(np.ldexp(1.0, tab[:, 256:].astype(np.int64) - 127), 32, axis=1).astype(np.float32)
    seq = dec[ids[:, 0, 0]].astype(np.float32)
    for h in range(1, 8):
        seq = (seq + dec[ids[:, 0, h]]).astype(np.float32)
    rev = dec[ids[:, 0, 7]].astype(np.float32)
    for h in range(6, -1, -1):
        rev = (rev + dec[ids[:, 0, h]]).astype(np.float32)
    ref = torch.from_numpy(seq).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    rref = torch.from_numpy(rev).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, ref)
    assert not np.array_equal(ref, rref), "inputs do not distinguish the summation order"


def test_engram_bad_ids_decode_as_zero():
    tab = synth.engram_table(5, synth.stream(synth.S_ENGRAM_TABLE), 16).numpy()
    ids = np.array([[[3]], [[16]], [[-1]]], dtype=np.int64)
    out, err = oracle.engram_gather([tab], ids)
    assert err & 2
    assert np.all(out[1:] == 0)
    good, e0 = oracle.engram_gather([tab], ids[:1])
    assert e0 == 0 and np.array_equal(out[0], good[0])


def test_engram_signed_zero_kept():
    tab = np.zeros((1, 264), dtype=np.uint8)
    tab[0, :256] = 0x80                   # -0.0
    tab[0, 256:] = 127
    out, _ = oracle.engram_gather([tab], np.zeros((1, 1, 3), dtype=np.int64))
    assert np.all(out == 0x8000)


# --------------------------------------------------------------------------- #
# block formats
# --------------------------------------------------------------------------- #

def test_q2k_decode_vs_independent_numpy():
    blk = synth.q2k_blocks(2, 9, 0, 4096).numpy()
    assert np.array_equal(f32_bits(oracle.dequant_q2k(blk)), f32_bits(np_dequant_q2k(blk)))


def test_q2k_decode_all_fp16_scales():
    # every fp16 bit pattern as d and as dmin, with random codes and nibbles
    rng = np.random.default_rng(5)
    n = 65536
    blk = rng.integers(0, 256, (n, 84), dtype=np.uint64).astype(np.uint8)
    blk[:, 80:82] = np.arange(n, dtype=np.uint16).view(np.uint8).reshape(n, 2)
    blk[:, 82:84] = np.roll(np.arange(n, dtype=np.uint16), 12345).view(np.uint8).reshape(n, 2)
    assert same_f32(oracle.dequant_q2k(blk), np_dequant_q2k(blk))


def test_q2k_field_positions():
    # one nonzero field at a time: which weights change tells the index mapping
    base = np.zeros(84, dtype=np.uint8)
    base[80:82] = np.array([0x3C00], dtype=np.uint16).view(np.uint8)    # d = 1
    base[82:84] = np.array([0x3800], dtype=np.uint16).view(np.uint8)    # dmin = 0.5
    for j in (0, 5, 15):
        b = base.copy()
        b[j] = 0x30                          # m_j = 3, sc_j = 0
        w = oracle.dequant_q2k(b)
        nz = np.nonzero(w)[0]
        assert list(nz) == list(range(16 * j, 16 * j + 16)) and np.all(w[nz] == -1.5)
    for i in (0, 1, 2, 3, 4, 17, 255):
        b = base.copy()
        b[i // 16] = 0x07                    # sc = 7 on the sub-block of weight i
        b[16 + i // 4] = 3 << (2 * (i % 4))  # code 3 at weight i
        w = oracle.dequant_q2k(b)
        assert list(np.nonzero(w)[0]) == [i] and w[i] == 21.0


def test_q8_0_decode():
    blk = synth.q8_0_blocks(2, 9, 0, 4096).numpy()
    assert np.array_equal(f32_bits(oracle.dequant_q8_0(blk)), f32_bits(np_dequant_q8_0(blk)))
    b = np.zeros(34, dtype=np.uint8)
    b[0:2] = np.array([0x4000], dtype=np.uint16).view(np.uint8)         # d = 2
    b[2 + 7] = 0xFF                                                     # q = -1
    b[2 + 31] = 0x7F                                                    # q = 127
    w = oracle.dequant_q8_0(b)
    assert w[7] == -2.0 and w[31] == 254.0 and np.count_nonzero(w) == 2


def test_synth_generator_reproducible():
    s = synth.stream(synth.S_GATE, 3)
    for i in (0, 1, 77, 123456):
        assert int(synth.u64(7, s, i, 1)[0]) & ((1 << 64) - 1) == synth.u64_py(7, s, i)
    a = synth.q2k_blocks(7, s, 100, 50)
    b = synth.q2k_blocks(7, s, 0, 200)[100:150]
    assert torch.equal(a, b)
    d = a[:, 80:82].contiguous().view(torch.float16).float()
    assert float(d.min()) >= 0.00099 and float(d.max()) <= 0.01001
    rows = synth.engram_rows_at(3, 16, torch.tensor([5, 1, 5]))
    assert torch.equal(rows[0], rows[2]) and not torch.equal(rows[0], rows[1])
    assert int(rows[:, 256:].min()) >= 120 and int(rows[:, 256:].max()) <= 134
    assert not bool(((rows[:, :256] & 0x7F) == 0x7F).any())


# --------------------------------------------------------------------------- #
# router
# --------------------------------------------------------------------------- #

def _tiny_router(seed=1, T=3, d=64, E=8):
    x = synth.x_bf16(seed, 0, 0, T, d)
    wr = synth.router_weight(seed, 0, d, E) * 10        # spread the scores
    b = synth.route_bias(seed, 0, E, 0.1)
    return x, wr, b


def test_router_lane32_exact_rational():
    x, wr, b = _tiny_router()
    T, d = x.shape
    E = wr.shape[1]
    _, _, z, _ = oracle.route(x, wr, b, 2, want_scores=True)
    xf = x.float().numpy()
    wf = wr.numpy()
    for t in range(T):
        for e in range(E):
            p = [0.0] * 32
            for j in range(32):
                for c in range(j, d, 32):
                    p[j] = round_f32(Fraction(float(xf[t, c])) * Fraction(float(wf[c, e])) + Fraction(p[j]))
            for o in (16, 8, 4, 2, 1):
                p = [round_f32(Fraction(p[j]) + Fraction(p[j ^ o])) for j in range(32)]
            assert np.float32(p[0]) == z[t, e]


def test_router_logits_within_fp32_bound():
    T, d, E = 4, 512, 32
    x = synth.x_bf16(3, 0, 0, T, d)
    wr = synth.router_weight(3, 0, d, E)
    _, _, z, _ = oracle.route(x, wr, None, 6, want_scores=True)
    xf = x.double().numpy()
    wf = wr.double().numpy()
    z64 = xf @ wf
    mag = np.abs(xf) @ np.abs(wf)
    gamma = (d // 32 + 6) * 2.0 ** -24 * 1.01
    assert np.all(np.abs(z - z64) <= gamma * mag)


def test_router_sigmoid_vs_high_precision():
    """R2: the float sigmoid is within 4 ulp of the exact value everywhere it is used, exact
    at 0, and 0 beyond the documented cut-off."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    zs = np.concatenate([np.linspace(-87.9, 60.0, 4001), np.random.default_rng(2).standard_normal(2000) * 8,
                         [0.0, -1e-30, 1e-30, 17.0, -17.0, 30.0, 31.0, -88.0]]).astype(np.float32)
    for z in zs:
        got = np.float32(L.or_sigmoid(float(z)))
        exact = 1 / (1 + mpmath.exp(-mpmath.mpf(float(z))))
        ref = np.float32(float(exact))
        ulp = float(np.spacing(ref))
        assert abs(Fraction(float(got)) - Fraction(str(mpmath.nstr(exact, 40)))) <= 4 * Fraction(ulp), float(z)
    assert L.or_sigmoid(0.0) == 0.5
    assert L.or_sigmoid(-88.5) == 0.0 and L.or_sigmoid(100.0) == 1.0
    x, wr, b = _tiny_router(T=4, d=64, E=16)
    _, _, z, s = oracle.route(x, wr, b, 2, want_scores=True)
    assert np.array_equal(s, np.array([[L.or_sigmoid(float(v)) for v in row] for row in z], dtype=np.float32))


def test_router_selection_brute_force():
    for seed in range(5):
        T, d, E, k = 4, 512, 32, 6
        x = synth.x_bf16(seed, 0, 0, T, d)
        wr = synth.router_weight(seed, 0, d, E)
        b = synth.route_bias(seed, 0, E, 0.1)
        ids, w, z, s = oracle.route(x, wr, b, k, want_scores=True)
        bn = b.numpy()
        for t in range(T):
            keys = (s[t] + bn).astype(np.float32)
            order = sorted(range(E), key=lambda e: (-float(keys[e]), e))
            assert list(ids[t]) == order[:k]
            sel = s[t, ids[t]]
            S = np.float32(0)
            for v in sel:
                S = np.float32(S + v)
            assert np.array_equal(w[t], (sel / S).astype(np.float32))
            assert abs(float(np.sum(w[t].astype(np.float64))) - 1.0) <= 6 * 2.0 ** -24


def test_router_zero_bias_is_topk_of_logits():
    T, d, E, k = 8, 512, 32, 6
    x = synth.x_bf16(9, 0, 0, T, d)
    wr = synth.router_weight(9, 0, d, E)
    ids, _ = oracle.route(x, wr, None, k)
    z64 = x.double().numpy() @ wr.double().numpy()
    for t in range(T):
        order = np.argsort(-z64[t], kind="stable")
        margin = z64[t, order[k - 1]] - z64[t, order[k]]
        if margin > 1e-6:
            assert set(ids[t]) == set(order[:k])
            assert list(ids[t]) == list(order[:k])


def test_router_ties_go_to_lower_id_and_bias_is_selection_only():
    d, E, k = 64, 16, 6
    x = synth.x_bf16(2, 0, 0, 2, d)
    wr = torch.zeros((d, E), dtype=torch.float32)       # every logit 0 -> every score 0.5
    ids, w = oracle.route(x, wr, None, k)
    assert np.all(ids == np.arange(k)) and np.all(w == np.float32(0.5) / np.float32(3.0))
    b = torch.zeros(E)
    b[9] = 0.25
    b[12] = 0.25
    ids, w = oracle.route(x, wr, b, k)
    assert list(ids[0]) == [9, 12, 0, 1, 2, 3]
    assert np.all(w == np.float32(0.5) / np.float32(3.0))   # weights from the unbiased scores


# --------------------------------------------------------------------------- #
# router variants (per-row rule of the device router notes)
# --------------------------------------------------------------------------- #

def test_sqrt_softplus_vs_high_precision():
    """R12: the float sqrt(softplus(z)) is within 2 ulp of the exact value on |z| <= 87, and
    its special values are those of the definition (or of the documented cut-off)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    zs = np.concatenate([np.linspace(-86.9, 86.9, 3001), np.random.default_rng(5).standard_normal(2000) * 6,
                         [0.0, -1e-30, 1e-30, 1.0, -1.0, 15.0, -15.0, 40.0, -40.0]]).astype(np.float32)
    for z in zs:
        got = np.float32(L.or_sqrt_softplus(float(z)))
        zz = mpmath.mpf(float(z))
        exact = mpmath.sqrt(mpmath.log(1 + mpmath.exp(zz)))
        ref = np.float32(float(exact))
        ulp = float(np.spacing(ref))
        assert abs(Fraction(float(got)) - Fraction(str(mpmath.nstr(exact, 40)))) <= 2 * Fraction(ulp), float(z)
    assert L.or_sqrt_softplus(-100.0) == 0.0                      # |z| > 87: exp term dropped
    assert L.or_sqrt_softplus(100.0) == np.float32(10.0)
    assert math.isinf(L.or_sqrt_softplus(float("inf"))) and L.or_sqrt_softplus(float("-inf")) == 0.0
    assert math.isnan(L.or_sqrt_softplus(float("nan")))
    # monotone non-decreasing (so, without a bias, it selects what the logits select)
    grid = np.linspace(-86.0, 86.0, 20001).astype(np.float32)
    vals = np.array([L.or_sqrt_softplus(float(z)) for z in grid], dtype=np.float32)
    assert np.all(np.diff(vals) >= 0)


def _variant_inputs(seed=4, T=6, d=256, E=40, k=6):
    x = synth.x_bf16(seed, 0, 0, T, d)
    wr = synth.router_weight(seed, 0, d, E)
    b = synth.route_bias(seed, 0, E, 0.3)
    vb = synth.route_bias(seed, 1, E, 0.3)
    return x, wr, b, vb


def test_route_ex_defaults_equal_route():
    x, wr, b, _ = _variant_inputs()
    ids0, w0 = oracle.route(x, wr, b, 6)
    ids1, w1, err = oracle.route_ex(x, wr, b, 6)
    assert err == 0 and np.array_equal(ids0, ids1) and same_f32(w0, w1)


def test_route_ex_media_rows_take_the_vision_bias():
    x, wr, b, vb = _variant_inputs()
    media = np.array([0, 1, 1, 0, 1, 0], dtype=np.uint8)
    ids, w, err = oracle.route_ex(x, wr, b, 6, vision_bias=vb, is_media=media)
    ids_t, w_t = oracle.route(x, wr, b, 6)
    ids_m, w_m = oracle.route(x, wr, vb, 6)
    assert err == 0
    for t in range(len(media)):
        ref_i, ref_w = (ids_m, w_m) if media[t] else (ids_t, w_t)
        assert np.array_equal(ids[t], ref_i[t]) and same_f32(w[t], ref_w[t])
    # without the vision bias nothing is media
    ids2, w2, _ = oracle.route_ex(x, wr, b, 6, is_media=media)
    assert np.array_equal(ids2, ids_t) and same_f32(w2, w_t)


def test_route_ex_hash_rows_take_the_table():
    x, wr, b, vb = _variant_inputs()
    T, k, E = 6, 6, 40
    rng = np.random.default_rng(11)
    vocab = 50
    table = np.stack([rng.permutation(E)[:k] for _ in range(vocab)]).astype(np.int32)
    tok = rng.integers(0, vocab, size=T).astype(np.int32)
    media = np.array([0, 0, 1, 0, 0, 1], dtype=np.uint8)
    ids, w, err = oracle.route_ex(x, wr, b, k, vision_bias=vb, is_media=media, tid2eid=table, token_ids=tok)
    _, _, _, s = oracle.route(x, wr, b, k, want_scores=True)     # unbiased sigmoid scores
    ids_m, w_m = oracle.route(x, wr, vb, k)
    assert err == 0
    for t in range(T):
        if media[t]:
            assert np.array_equal(ids[t], ids_m[t]) and same_f32(w[t], w_m[t])
            continue
        assert np.array_equal(ids[t], table[tok[t]])
        sel = s[t, table[tok[t]]]
        S = np.float32(0)
        for j, v in enumerate(sel):
            S = v if j == 0 else np.float32(S + v)
        assert same_f32(w[t], (sel / S).astype(np.float32))


def test_route_ex_sqrt_softplus_selects_what_the_logits_select():
    T, d, E, k = 8, 512, 32, 6
    x = synth.x_bf16(9, 0, 0, T, d)
    wr = synth.router_weight(9, 0, d, E)
    ids, w, err = oracle.route_ex(x, wr, None, k, score=1)
    _, _, z, _ = oracle.route(x, wr, None, k, want_scores=True)
    z64 = x.double().numpy() @ wr.double().numpy()
    assert err == 0
    for t in range(T):
        order = np.argsort(-z64[t], kind="stable")
        if z64[t, order[k - 1]] - z64[t, order[k]] > 1e-6:
            assert list(ids[t]) == list(order[:k])
        sel = np.array([L.or_sqrt_softplus(float(z[t, e])) for e in ids[t]], dtype=np.float32)
        S = np.float32(0)
        for j, v in enumerate(sel):
            S = v if j == 0 else np.float32(S + v)
        assert same_f32(w[t], (sel / S).astype(np.float32))


def test_route_ex_hash_errors():
    x, wr, b, _ = _variant_inputs(T=3)
    k, E = 6, 40
    table = np.array([[0, 1, 2, 3, 4, 5], [7, 99, 8, 9, 10, -2]], dtype=np.int32)
    tok = np.array([1, 5, 0], dtype=np.int32)          # row 1: token outside the table
    ids, w, err = oracle.route_ex(x, wr, b, k, tid2eid=table, token_ids=tok)
    assert err == 3
    assert list(ids[0]) == [7, 99, 8, 9, 10, -2]
    assert w[0, 1] == 0 and w[0, 5] == 0 and np.all(w[0, [0, 2, 3, 4]] > 0)
    assert np.all(ids[1] == -1) and np.all(w[1] == 0)
    assert list(ids[2]) == [0, 1, 2, 3, 4, 5]


# --------------------------------------------------------------------------- #
# permutation
# --------------------------------------------------------------------------- #

def test_permute_brute_force():
    rng = np.random.default_rng(1)
    for T, k, E in ((4, 6, 32), (64, 6, 32), (5, 6, 384), (1, 1, 1)):
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
        r = oracle.permute(ids, E)
        flat = ids.reshape(-1)
        order = sorted(range(T * k), key=lambda p: flat[p])       # Python's sort is stable
        assert list(r["perm"]) == order
        assert np.array_equal(np.sort(r["perm"]), np.arange(T * k))
        assert np.all(r["perm"][r["inv"]] == np.arange(T * k))
        counts = np.bincount(flat, minlength=E)
        assert np.array_equal(np.diff(r["offsets"]), counts) and r["offsets"][0] == 0
        assert list(r["active"]) == [e for e in range(E) if counts[e]]
        assert r["err"] == 0


def test_permute_bad_ids():
    ids = np.array([[0, 5], [40, 1]], dtype=np.int32)
    r = oracle.permute(ids, 8)
    assert r["err"] & 1
    assert r["offsets"][8] == 3 and r["perm"][3] == 2 and r["inv"][2] == 3


# --------------------------------------------------------------------------- #
# FFN and layer
# --------------------------------------------------------------------------- #

def _dense_expert(gate, up, down, d, F, fmt="q2k"):
    dec = np_dequant_q2k if fmt == "q2k" else np_dequant_q8_0
    G = dec(np.ascontiguousarray(gate)).reshape(F, d).astype(np.float64)
    U = dec(np.ascontiguousarray(up)).reshape(F, d).astype(np.float64)
    D = dec(np.ascontiguousarray(down)).reshape(d, F).astype(np.float64)
    return G, U, D


def _ffn64(G, U, D, x):
    g = x @ G.T
    u = x @ U.T
    return (g / (1 + np.exp(-g)) * u) @ D.T


def test_layer_dense_equivalent_tiny():
    sh = synth.TINY
    lw = synth.layer_weights(1, 0, sh)
    x = synth.x_bf16(1, 0, 0, 4, sh.d)
    r = oracle.moe_layer(x, lw.w_r, lw.bias, sh.k, sh.F, list(lw.gate.numpy()), list(lw.up.numpy()),
                         list(lw.down.numpy()), lw.sh_gate.numpy(), lw.sh_up.numpy(), lw.sh_down.numpy(), sh.F_shared)
    xf = x.double().numpy()
    ids, w = oracle.route(x, lw.w_r, lw.bias, sh.k)
    dense = _ffn64(*_dense_expert(lw.sh_gate.numpy(), lw.sh_up.numpy(), lw.sh_down.numpy(), sh.d, sh.F_shared, "q8"),
                   xf)
    for e in range(sh.E):
        # dense mixture over every expert with a 0/1 selection mask
        mask = np.array([float(w[t][list(ids[t]).index(e)]) if e in ids[t] else 0.0 for t in range(4)])
        ye = _ffn64(*_dense_expert(lw.gate[e].numpy(), lw.up[e].numpy(), lw.down[e].numpy(), sh.d, sh.F), xf)
        dense += mask[:, None] * ye
    assert np.array_equal(r["ids"], ids)
    assert np.max(np.abs(r["out_f64"] - dense)) <= 1e-12 * np.max(np.abs(dense))
    assert np.array_equal(r["out"], np.array([L.or_bf16_rne_f64(v) for v in r["out_f64"].reshape(-1)],
                                             dtype=np.uint16).reshape(r["out"].shape))


def test_layer_zero_codes_gives_shared_only():
    sh = synth.TINY
    lw = synth.layer_weights(2, 0, sh)
    zero = np.zeros((sh.F, (sh.d // 256) * 84), dtype=np.uint8)
    zero_d = np.zeros((sh.d, (sh.F // 256) * 84), dtype=np.uint8)
    x = synth.x_bf16(2, 0, 0, 4, sh.d)
    r = oracle.moe_layer(x, lw.w_r, lw.bias, sh.k, sh.F, [zero] * sh.E, [zero] * sh.E, [zero_d] * sh.E,
                         lw.sh_gate, lw.sh_up, lw.sh_down, sh.F_shared)
    ysh = oracle.expert_ffn(oracle.FMT_Q8_0, lw.sh_gate, lw.sh_up, lw.sh_down, sh.d, sh.F_shared, x)
    assert np.array_equal(r["out_f64"], ysh)


def test_layer_k_equals_E_uniform_mixture():
    sh = synth.MoeShape(d=256, E=4, k=4, F=256, F_shared=0, bias_half_width=0.0)
    lw = synth.layer_weights(4, 0, sh)
    x = synth.x_bf16(4, 0, 0, 2, sh.d)
    wr = torch.zeros((sh.d, sh.E))
    r = oracle.moe_layer(x, wr, None, sh.k, sh.F, list(lw.gate.numpy()), list(lw.up.numpy()), list(lw.down.numpy()))
    assert np.all(r["w"] == np.float32(0.25))
    xf = x.double().numpy()
    ref = sum(0.25 * _ffn64(*_dense_expert(lw.gate[e].numpy(), lw.up[e].numpy(), lw.down[e].numpy(), sh.d, sh.F), xf)
              for e in range(sh.E))
    assert np.max(np.abs(r["out_f64"] - ref)) <= 1e-12 * np.max(np.abs(ref))


def test_rmsnorm_and_residual():
    x = synth.x_bf16(5, 0, 0, 5, 4096)
    x = (x.float() * 37.0).to(torch.bfloat16)
    u = oracle.rmsnorm(x, 1e-6)
    xf = x.double().numpy()
    ref = xf / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + 1e-6)
    uf = torch.from_numpy(u.view(np.int16)).view(torch.bfloat16).double().numpy()
    # one bf16 rounding of a value within a few float ulps of the exact one
    assert np.all(np.abs(uf - ref) <= np.abs(ref) * (2.0 ** -8 + 2.0 ** -20))
    m = synth.x_bf16(6, 0, 0, 5, 4096)
    xn = oracle.residual(x, m, float(np.float32(1 / math.sqrt(2))))
    exp_ = (x.float().numpy() + (m.float().numpy() * np.float32(1 / math.sqrt(2))).astype(np.float32)).astype(np.float32)
    ref2 = torch.from_numpy(exp_).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(xn, ref2)


def test_verify_stack_literal_recurrence_overflows():
    """The layer-stack recurrence x <- x + moe(x)/sqrt(2) applied literally (no norm on the
    MoE input) overflows BF16 within a few layers, because h = silu(g)*u grows like |x|^2;
    this is why the stack normalises each layer's MoE input (a stated reading)."""
    sh = synth.TINY
    x = synth.x_bf16(1, 0, 0, 5, sh.d)
    s = float(np.float32(1 / math.sqrt(2)))
    finite_layers = 0
    for layer in range(6):
        lw = synth.layer_weights(1, layer, sh)
        r = oracle.moe_layer(x, lw.w_r, lw.bias, sh.k, sh.F, list(lw.gate.numpy()), list(lw.up.numpy()),
                             list(lw.down.numpy()), lw.sh_gate.numpy(), lw.sh_up.numpy(), lw.sh_down.numpy(),
                             sh.F_shared)
        x = torch.from_numpy(oracle.residual(x, torch.from_numpy(r["out"].view(np.int16)).view(torch.bfloat16), s)
                             .view(np.int16)).view(torch.bfloat16)
        if not bool(torch.isfinite(x.float()).all()):
            break
        finite_layers += 1
    assert finite_layers < 6


# --------------------------------------------------------------------------- #
# Engram gate and residual injection (closed forms and invariants)
# --------------------------------------------------------------------------- #

def _bf16(a):
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)


def _sig(x):
    return 1.0 / (1.0 + math.exp(-x))


def test_engram_kv_is_a_plain_product():
    """A selection matrix (one power of two per row) reproduces the chosen inputs exactly, and
    a product with integer entries is exact in FP64."""
    rng = np.random.default_rng(3)
    T, K, N = 3, 96, 40
    rows = _bf16(rng.standard_normal((T, K)))
    pick = rng.integers(0, K, N)
    w = np.zeros((N, K), dtype=np.float32)
    w[np.arange(N), pick] = 2.0 ** rng.integers(-3, 4, N)
    kv = oracle.engram_kv(rows, _bf16(w))
    assert np.array_equal(kv, rows.float().numpy()[:, pick] * w[np.arange(N), pick])
    ri = _bf16(rng.integers(-8, 9, (T, K)))
    wi = _bf16(rng.integers(-8, 9, (N, K)))
    assert np.array_equal(oracle.engram_kv(ri, wi), ri.double().numpy() @ wi.double().numpy().T)


def _gate_case(T=2, W=64, seed=0):
    rng = np.random.default_rng(seed)
    kv = rng.standard_normal((T, 5 * W))
    resid = _bf16(rng.standard_normal((T, 4, W)))
    qn = (1 + 0.1 * rng.standard_normal((4, W))).astype(np.float32)
    kn = (1 + 0.1 * rng.standard_normal((4, W))).astype(np.float32)
    return kv, resid, qn, kn


def test_engram_gate_known_dot():
    """r = 1, qn = kn = 1, key = a: dot = W a / sqrt(1 + eps) / sqrt(a^2 + eps) / sqrt(W); the
    update is bf16(1 + g * bf16(v)) for a constant value v."""
    T, W, eps = 1, 5120, 1e-6
    for a, v in ((0.75, 0.3), (-2.0, 1.5), (1e-3, -0.7)):
        kv = np.zeros((T, 5 * W))
        kv[:, :4 * W] = a
        kv[:, 4 * W:] = v
        resid = _bf16(np.ones((T, 4, W)))
        ones = np.ones((4, W), dtype=np.float32)
        out, g = oracle.engram_gate(kv, resid, ones, ones, eps=eps)
        dot = W * a / math.sqrt(1 + eps) / math.sqrt(a * a + eps) / math.sqrt(W)
        ref_g = _sig(math.copysign(math.sqrt(max(abs(dot), 1e-6)), dot))
        assert np.allclose(g, ref_g, rtol=0, atol=1e-12)
        vb = float(_bf16([v]).float()[0])
        ref = _bf16(np.full((T, 4, W), 1.0 + ref_g * vb))
        assert np.array_equal(out, ref.view(torch.int16).numpy().view(np.uint16))


def test_engram_gate_known_dot_with_norm_weights():
    """The q_norm and k_norm factors of the dot product (strix-llama.cpp issue, "Placement":
    dot = sum_i residual * q_norm * k_norm * key), pinned with weights that differ by branch and
    by index: r = 1, key = a, q_norm[h,i] = 2^((i+h) mod 3), k_norm[h,i] = 2^-((i+2h) mod 5).
    Then dot_h = a * S_h / sqrt(1 + eps) / sqrt(a^2 + eps) / sqrt(W) with S_h = sum_i
    q_norm[h,i] k_norm[h,i], an exact dyadic sum.  Dropping either factor, using one of them
    twice, or reading another branch's weights changes S_h (the four S_h differ, and differ from
    sum q_norm^2, sum k_norm^2 and W)."""
    from fractions import Fraction
    T, W, eps = 1, 64, 1e-6
    i = np.arange(W)
    qn = np.stack([2.0 ** ((i + h) % 3) for h in range(4)]).astype(np.float32)
    kn = np.stack([2.0 ** -((i + 2 * h) % 5) for h in range(4)]).astype(np.float32)
    S = [sum(Fraction(2) ** (((j + h) % 3) - ((j + 2 * h) % 5)) for j in range(W)) for h in range(4)]
    assert len(set(S)) == 4
    for h in range(4):
        others = {sum(Fraction(2) ** (2 * ((j + h) % 3)) for j in range(W)),
                  sum(Fraction(2) ** (-2 * ((j + 2 * h) % 5)) for j in range(W)), Fraction(W)}
        assert S[h] not in others
    for a, v in ((0.75, 0.3), (-2.0, 1.5)):
        kv = np.zeros((T, 5 * W))
        kv[:, :4 * W] = a
        kv[:, 4 * W:] = v
        resid = _bf16(np.ones((T, 4, W)))
        out, g = oracle.engram_gate(kv, resid, qn, kn, eps=eps)
        vb = float(_bf16([v]).float()[0])
        for h in range(4):
            dot = a * float(S[h]) / math.sqrt(1 + eps) / math.sqrt(a * a + eps) / math.sqrt(W)
            ref_g = _sig(math.copysign(math.sqrt(max(abs(dot), 1e-6)), dot))
            assert abs(g[0, h] - ref_g) <= 1e-12
            ref = _bf16(np.full(W, 1.0 + ref_g * vb))
            assert np.array_equal(out[0, h], ref.view(torch.int16).numpy().view(np.uint16))


def test_engram_gate_zero_key_floor_and_zero_value_identity():
    kv, resid, qn, kn = _gate_case()
    W = resid.shape[-1]
    kv0 = kv.copy()
    kv0[:, :4 * W] = 0.0                                  # dot = 0 -> gate = sigmoid(+1e-3)
    _, g = oracle.engram_gate(kv0, resid, qn, kn)
    assert np.allclose(g, _sig(1e-3), rtol=0, atol=1e-15)
    kv1 = kv.copy()
    kv1[:, 4 * W:] = 0.0                                  # no value: the residual is unchanged
    out, _ = oracle.engram_gate(kv1, resid, qn, kn)
    assert np.array_equal(out, resid.view(torch.int16).numpy().view(np.uint16))


def test_engram_gate_masked_rows_unchanged():
    kv, resid, qn, kn = _gate_case(T=3)
    mask = np.array([0, 1, 0], dtype=np.uint8)
    out, g = oracle.engram_gate(kv, resid, qn, kn, mask=mask)
    rb = resid.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out[1], rb[1]) and np.all(g[1] == 0)
    assert not np.array_equal(out[0], rb[0])


def test_engram_gate_invariances():
    """The gate does not change when a branch's residual or key is scaled (both norms divide the
    scale out; exact up to eps), and negating the residual gives 1 - gate."""
    kv, resid, qn, kn = _gate_case(T=2, W=256, seed=5)
    W = 256
    _, g = oracle.engram_gate(kv, resid, qn, kn)
    _, g2 = oracle.engram_gate(kv, _bf16(resid.float().numpy() * 4.0), qn, kn)
    # eps = 1e-6 against mean squares near 1 moves the gate by well under 1e-6
    assert np.allclose(g, g2, rtol=0, atol=1e-6)
    kvs = kv.copy()
    kvs[:, :4 * W] *= 4.0
    _, g3 = oracle.engram_gate(kvs, resid, qn, kn)
    assert np.allclose(g, g3, rtol=0, atol=1e-6)
    _, gn = oracle.engram_gate(kv, _bf16(-resid.float().numpy()), qn, kn)
    assert np.allclose(g + gn, 1.0, rtol=0, atol=1e-12)
    # the gate depends on the branch's own key only
    kvb = kv.copy()
    kvb[:, 1 * W:2 * W] = 3.0
    _, g4 = oracle.engram_gate(kvb, resid, qn, kn)
    assert np.array_equal(g4[:, [0, 2, 3]], g[:, [0, 2, 3]]) and not np.allclose(g4[:, 1], g[:, 1])
