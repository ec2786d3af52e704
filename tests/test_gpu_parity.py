"""Parity of the CUDA path (through the C-ABI) with the CPU oracle, on the same seeded inputs.

Bar: bit-exact for ids, permutation, dequantised values and Engram BF16 output;
max|out - ref| <= 1e-2 * rms(ref) for MoE layer outputs (ref in FP64).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from bit_routed_expert_gb300 import api, synth
from bit_routed_expert_gb300.api import BRE_FMT_Q2_K, BRE_FMT_Q8_0, FfnWeights, MoeLayer
from helpers import assert_layer_close, bf16_bits, device_layer, oracle_layer, run_layer

pytestmark = pytest.mark.gpu

SEED = 1


def _sync():
    torch.cuda.synchronize()


# --------------------------------------------------------------------------- #
# generator: identical bytes on CPU and GPU
# --------------------------------------------------------------------------- #

def test_generator_cpu_gpu_identical(cuda_dev):
    s = synth.stream(synth.S_GATE, 2)
    a = synth.q2k_blocks(SEED, s, 1000, 5000, device="cpu")
    b = synth.q2k_blocks(SEED, s, 1000, 5000, device=cuda_dev).cpu()
    assert torch.equal(a, b)
    a = synth.q8_0_blocks(SEED, s, 7, 3000, device="cpu")
    b = synth.q8_0_blocks(SEED, s, 7, 3000, device=cuda_dev).cpu()
    assert torch.equal(a, b)
    r = torch.tensor([0, 5, 4194303, 77777], dtype=torch.int64)
    assert torch.equal(synth.engram_rows_at(SEED, 16, r), synth.engram_rows_at(SEED, 16, r.to(cuda_dev)).cpu())


# --------------------------------------------------------------------------- #
# formats
# --------------------------------------------------------------------------- #

def test_dequant_q2k_bit_exact(cuda_dev):
    blk = synth.q2k_blocks(SEED, 99, 0, 20000)
    rng = np.random.default_rng(0)
    special = rng.integers(0, 256, (65536, 84), dtype=np.uint64).astype(np.uint8)
    special[:, 80:82] = np.arange(65536, dtype=np.uint16).view(np.uint8).reshape(-1, 2)
    special[:, 82:84] = np.roll(np.arange(65536, dtype=np.uint16), 999).view(np.uint8).reshape(-1, 2)
    allb = torch.cat([blk, torch.from_numpy(special)])
    got = api.bre_dequant(BRE_FMT_Q2_K, allb.to(cuda_dev)).cpu().numpy()
    ref = oracle.dequant_q2k(allb.numpy())
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _np_repack_r16(m: np.ndarray) -> np.ndarray:
    """The Q2_K_R16 layout restated from its definition (bre.h, bre_repack_q2k_r16): m uint8
    [rows, nb * 84] Q2_K blocks -> [rows / 16, nb, 1344]."""
    rows, nb = m.shape[0], m.shape[1] // 84
    blk = m.reshape(rows, nb, 84).astype(np.uint32)
    qs = blk[:, :, 16:80]
    codes = np.stack([(qs >> (2 * c)) & 3 for c in range(4)], axis=-1).reshape(rows, nb, 256)
    out = np.zeros((rows // 16, nb, 1344), dtype=np.uint8)
    for R in range(16):
        g, rr = R & 7, R >> 3
        rsel = np.arange(rows // 16) * 16 + R
        for t in range(4):
            L = 4 * g + t
            for p in range(2):
                for w in range(2):
                    word = np.zeros((rows // 16, nb), dtype=np.uint32)
                    for h in range(2):
                        j = 4 * t + 2 * p + h
                        for s_ in range(8):
                            word |= codes[rsel, :, 16 * j + 8 * w + s_] << (16 * h + 2 * s_)
                    o = rr * 512 + 16 * L + 4 * (2 * p + w)
                    out[:, :, o:o + 4] = word[..., None].view(np.uint8).reshape(rows // 16, nb, 4)
        out[:, :, 1280 + 8 * g + 4 * rr:1280 + 8 * g + 4 * rr + 4] = blk[rsel, :, 80:84].astype(np.uint8)
    for g in range(8):
        for t in range(4):
            L = 4 * g + t
            scw = np.zeros((rows // 16, nb), dtype=np.uint32)
            mw = np.zeros((rows // 16, nb), dtype=np.uint32)
            for rr in range(2):
                rsel = np.arange(rows // 16) * 16 + 8 * rr + g
                for p in range(2):
                    for h in range(2):
                        j = 4 * t + 2 * p + h
                        pos = 16 * h + 4 * (2 * rr + p)
                        scw |= (blk[rsel, :, j] & 15) << pos
                        mw |= (blk[rsel, :, j] >> 4) << pos
            out[:, :, 1024 + 8 * L:1024 + 8 * L + 4] = scw[..., None].view(np.uint8).reshape(rows // 16, nb, 4)
            out[:, :, 1028 + 8 * L:1028 + 8 * L + 4] = mw[..., None].view(np.uint8).reshape(rows // 16, nb, 4)
    return out


@pytest.mark.parametrize("n,rows,cols", [(3, 64, 1024), (1, 16, 256), (2, 48, 512)])
def test_repack_q2k_r16_layout(cuda_dev, n, rows, cols):
    """bre_repack_q2k_r16 against the layout's definition, byte for byte; the tiles hold exactly
    the blocks' bytes (same size, every code, nibble and d/dmin accounted for)."""
    shape = synth.MoeShape(d=cols, E=n, k=1, F=rows, F_shared=0, bias_half_width=0.1)
    m = synth.expert_matrix(SEED, 3, synth.S_GATE, shape, 0, n)           # [n, rows, cols/256*84]
    got = api.repack_q2k_r16(m.to(cuda_dev)).cpu().numpy()
    for e in range(n):
        ref = _np_repack_r16(m[e].numpy())
        assert np.array_equal(got[e].reshape(-1), ref.reshape(-1))


def test_dequant_q80_bit_exact(cuda_dev):
    blk = synth.q8_0_blocks(SEED, 98, 0, 20000)
    got = api.bre_dequant(BRE_FMT_Q8_0, blk.to(cuda_dev)).cpu().numpy()
    ref = oracle.dequant_q8_0(blk.numpy())
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------------------------- #
# Engram
# --------------------------------------------------------------------------- #

def _all_pairs_table():
    rows = np.zeros((256, 264), dtype=np.uint8)
    for r in range(32):
        for rot in range(8):
            i = r * 8 + rot
            rows[i, :256] = (np.arange(256) + 32 * rot) % 256
            rows[i, 256:] = np.arange(8 * r, 8 * r + 8)
    return rows


def test_engram_exhaustive_codes_and_scales(cuda_dev):
    tab = _all_pairs_table()
    ids = np.arange(256, dtype=np.int64).reshape(256, 1, 1)
    ref, err = oracle.engram_gather([tab], ids)
    got = api.engram_gather_decode([torch.from_numpy(tab).to(cuda_dev)], torch.from_numpy(ids).to(cuda_dev))
    assert np.array_equal(bf16_bits(got), ref)


def test_engram_eight_heads_all_pairs(cuda_dev):
    # the 8-head kernel: token t sums rows (t + 37 h) mod 256 of the all-pairs table over heads
    # h = 0..7, so every (code, scale) pair, NaN, infinite and subnormal scales included, enters
    # the head sum at every head position
    tab = _all_pairs_table()
    ids = ((np.arange(256)[:, None] + 37 * np.arange(8)[None, :]) % 256).astype(np.int64).reshape(256, 1, 8)
    ref, err = oracle.engram_gather([tab], ids)
    got = api.engram_gather_decode([torch.from_numpy(tab).to(cuda_dev)], torch.from_numpy(ids).to(cuda_dev))
    assert np.array_equal(bf16_bits(got), ref)


def test_engram_tiny_config(cuda_dev):
    tab = synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE), 1024)
    ids = synth.engram_ids_uniform(SEED, 64, 1024).view(64, 1, 1)
    ref, err = oracle.engram_gather([tab.numpy()], ids.numpy())
    dev_err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    got = api.engram_gather_decode([tab.to(cuda_dev)], ids.to(cuda_dev), dev_err=dev_err)
    assert np.array_equal(bf16_bits(got), ref) and err == 0 and int(dev_err) == 0


def test_engram_heads_and_bad_ids(cuda_dev):
    rng = np.random.default_rng(3)
    tabs = [synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, tau), 500 + 37 * tau) for tau in range(3)]
    for tb in tabs:
        tb[:, 256:] = torch.from_numpy(rng.integers(100, 160, (tb.shape[0], 8)).astype(np.uint8))
    for H in (1, 3, 8, 13):
        ids = np.stack([rng.integers(0, tb.shape[0], (37, H)) for tb in tabs], axis=1).astype(np.int64)
        ids[3, 0, 0] = -1                       # invalid ids: negative, = n_rows, far beyond
        ids[10, 1, H - 1] = tabs[1].shape[0]
        ids[36, 2, H // 2] = 1 << 40
        ref, err = oracle.engram_gather([t.numpy() for t in tabs], ids)
        dev_err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
        got = api.engram_gather_decode([t.to(cuda_dev) for t in tabs], torch.from_numpy(ids).to(cuda_dev),
                                       dev_err=dev_err)
        assert np.array_equal(bf16_bits(got), ref)
        assert int(dev_err) == err == 2


def test_engram_full_size_sampled(cuda_dev):
    n_rows, T, H = 4194304, 8192, 8
    tabs = [synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, tau), n_rows, device=cuda_dev)
            for tau in range(2)]
    ids = synth.engram_ids_ngram(SEED, T, 2, H, n_rows)
    got = api.engram_gather_decode(tabs, torch.from_numpy(ids).to(cuda_dev))
    sample = np.unique(np.concatenate([np.arange(8), np.random.default_rng(1).integers(0, T, 500), [T - 1]]))
    sub = ids[sample]
    # oracle on the rows those ids name, regenerated on the CPU
    small_tabs, remap = [], np.empty_like(sub)
    for tau in range(2):
        u, inv = np.unique(sub[:, tau, :], return_inverse=True)
        small_tabs.append(synth.engram_rows_at(SEED, synth.stream(synth.S_ENGRAM_TABLE, 0, tau),
                                               torch.from_numpy(u)).numpy())
        remap[:, tau, :] = inv.reshape(sub.shape[0], H)
    ref, err = oracle.engram_gather(small_tabs, remap)
    assert np.array_equal(bf16_bits(got)[sample], ref)


# --------------------------------------------------------------------------- #
# router and permutation
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("shape,T", [(synth.TINY, 4), (synth.V41, 1), (synth.V41, 2), (synth.V41, 4), (synth.V41, 8),
                                     (synth.V41, 5), (synth.V41, 17), (synth.V41, 32), (synth.TINY, 9),
                                     (synth.TINY, 33), (synth.TINY, 300)])
def test_route_bit_exact(cuda_dev, shape, T):
    for tset in range(2):
        x = synth.x_bf16(SEED, 0, tset, T, shape.d)
        w_r = synth.router_weight(SEED, 0, shape.d, shape.E)
        b = synth.route_bias(SEED, 0, shape.E, shape.bias_half_width)
        ids_ref, w_ref = oracle.route(x, w_r, b, shape.k)
        ids, w = api.moe_route(x.to(cuda_dev), w_r.to(cuda_dev), b.to(cuda_dev), shape.k)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        assert np.array_equal(w.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))


def test_route_prefill_zipf_sampled(cuda_dev):
    shape, T = synth.V41_PREFILL, 8192
    x = synth.x_bf16(SEED, 0, 0, T, shape.d)
    w_r = synth.router_weight(SEED, 0, shape.d, shape.E)
    b = synth.route_bias(SEED, 0, shape.E, shape.bias_half_width, shape.zipf)
    ids, w = api.moe_route(x.to(cuda_dev), w_r.to(cuda_dev), b.to(cuda_dev), shape.k)
    sample = np.concatenate([np.arange(0, T, 17), [T - 1]])
    ids_ref, w_ref = oracle.route(x[sample], w_r, b, shape.k)
    assert np.array_equal(ids.cpu().numpy()[sample], ids_ref)
    assert np.array_equal(w.cpu().numpy()[sample].view(np.uint32), w_ref.view(np.uint32))


@pytest.mark.parametrize("T,d,E,k", [(3, 96, 40, 32), (12, 64, 33, 7), (2, 32, 1, 1), (20, 160, 70, 9),
                                     (40, 96, 33, 7), (100, 224, 70, 9), (77, 4096, 384, 6)])
def test_route_odd_shapes(cuda_dev, T, d, E, k):
    """Expert counts that leave a partial block of 32, k up to 32, several token groups; above
    32 tokens the large-batch kernel, with rows not a multiple of its 128-row stage."""
    x = synth.x_bf16(SEED + d, 0, 0, T, d)
    w_r = synth.router_weight(SEED + E, 0, d, E)
    b = synth.route_bias(SEED + k, 0, E, 0.3)
    ids_ref, w_ref = oracle.route(x, w_r, b, k)
    ids, w = api.moe_route(x.to(cuda_dev), w_r.to(cuda_dev), b.to(cuda_dev), k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))


@pytest.mark.parametrize("shape,T", [(synth.TINY, 4), (synth.V41, 1), (synth.V41, 8), (synth.V41, 5),
                                     (synth.V41, 17), (synth.V41, 32), (synth.V41, 33), (synth.TINY, 300),
                                     (synth.TINY, 1000), (synth.TINY, 2731), (synth.V41, 700)])
def test_route_permute_fused(cuda_dev, shape, T):
    """moe_route_permute equals the oracle's route followed by its permutation (one launch up to
    32 tokens; above, the scores and top k, then a permutation that takes three grid-wide
    launches over chunks of 1,024 pairs once there are more than 1,024 pairs)."""
    x = synth.x_bf16(SEED, 0, 9, T, shape.d)
    w_r = synth.router_weight(SEED, 0, shape.d, shape.E)
    b = synth.route_bias(SEED, 0, shape.E, shape.bias_half_width)
    ids_ref, w_ref = oracle.route(x, w_r, b, shape.k)
    ref = oracle.permute(ids_ref, shape.E)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    ws = torch.zeros(api.moe_route_workspace(T, shape.E), dtype=torch.uint8, device=cuda_dev)
    for _ in range(2):   # the second call reuses the workspace (its counters must be back at zero)
        ids, w, got = api.moe_route_permute(x.to(cuda_dev), w_r.to(cuda_dev), b.to(cuda_dev), shape.k, ws=ws,
                                            dev_err=err)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        assert np.array_equal(w.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))
        for key in ("offsets", "perm", "inv"):
            assert np.array_equal(got[key].cpu().numpy(), ref[key]), key
        na = int(got["n_active"])
        assert na == ref["n_active"]
        assert np.array_equal(got["active"].cpu().numpy()[:na], ref["active"])
        assert np.all(got["active"].cpu().numpy()[na:] == -1)
    assert int(err) == 0


def _variant_case(T, d, E, k, seed):
    x = synth.x_bf16(seed, 0, 3, T, d)
    w_r = synth.router_weight(seed, 0, d, E)
    b = synth.route_bias(seed, 0, E, 0.3)
    vb = synth.route_bias(seed, 1, E, 0.3)
    rng = np.random.default_rng(seed)
    media = (rng.random(T) < 0.4).astype(np.uint8)
    vocab = 1000
    table = np.stack([rng.permutation(E)[:k] for _ in range(vocab)]).astype(np.int32)
    tok = rng.integers(0, vocab, T).astype(np.int32)
    return x, w_r, b, vb, media, table, tok


_VARIANT_MODES = {
    "softplus": dict(score=1),
    "media": dict(media=True),
    "hash": dict(hash=True),
    "hash_softplus_media": dict(score=1, media=True, hash=True),
}


@pytest.mark.parametrize("T,d,E,k", [(1, 4096, 384, 6), (8, 4096, 384, 6), (5, 256, 40, 6), (32, 512, 384, 6),
                                     (33, 256, 70, 9), (300, 512, 384, 6)])
@pytest.mark.parametrize("mode", list(_VARIANT_MODES))
def test_route_ex_bit_exact(cuda_dev, T, d, E, k, mode):
    """moe_route_ex equals the oracle bit for bit in every mode of the per-row rule, on both
    router kernels (T <= 32 and T > 32) and with partial expert blocks."""
    x, w_r, b, vb, media, table, tok = _variant_case(T, d, E, k, SEED + T + E)
    o = _VARIANT_MODES[mode]
    score = o.get("score", 0)
    kw_ref = dict(score=score)
    if o.get("media"):
        kw_ref.update(vision_bias=vb, is_media=media)
    if o.get("hash"):
        kw_ref.update(tid2eid=table, token_ids=tok)
    ids_ref, w_ref, err_ref = oracle.route_ex(x, w_r, b, k, **kw_ref)
    dv = cuda_dev
    kw = dict(score=score)
    if o.get("media"):
        kw.update(vision_bias=vb.to(dv), is_media=torch.from_numpy(media).to(dv))
    if o.get("hash"):
        kw.update(tid2eid=torch.from_numpy(table).to(dv), token_ids=torch.from_numpy(tok).to(dv))
    err = torch.zeros(1, dtype=torch.int32, device=dv)
    ws = torch.zeros(api.moe_route_workspace(T, E), dtype=torch.uint8, device=dv)
    for _ in range(2):   # the second call reuses the workspace
        ids, w = api.moe_route_ex(x.to(dv), w_r.to(dv), b.to(dv), k, ws=ws, dev_err=err, **kw)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        assert np.array_equal(w.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))
    assert int(err) == err_ref == 0


@pytest.mark.parametrize("T", [4, 8, 40])
def test_route_ex_defaults_equal_moe_route(cuda_dev, T):
    x, w_r, b, _, _, _, _ = _variant_case(T, 512, 384, 6, 3)
    ids0, w0 = api.moe_route(x.to(cuda_dev), w_r.to(cuda_dev), b.to(cuda_dev), 6)
    ids1, w1 = api.moe_route_ex(x.to(cuda_dev), w_r.to(cuda_dev), b.to(cuda_dev), 6)
    assert torch.equal(ids0, ids1) and torch.equal(w0.view(torch.int32), w1.view(torch.int32))


@pytest.mark.parametrize("T", [3, 40])
def test_route_ex_hash_errors(cuda_dev, T):
    """A token outside the table gives ids -1 and weights 0 (BRE_DEVERR_ROW_ID); a table id
    outside [0, E) is passed on with weight 0 (BRE_DEVERR_EXPERT_ID) -- as the oracle."""
    d, E, k = 256, 40, 6
    x, w_r, b, _, _, _, _ = _variant_case(T, d, E, k, 8)
    table = np.array([[0, 1, 2, 3, 4, 5], [7, 99, 8, 9, 10, -2]], dtype=np.int32)
    tok = np.resize(np.array([1, 5, 0], dtype=np.int32), T)
    ids_ref, w_ref, err_ref = oracle.route_ex(x, w_r, b, k, tid2eid=table, token_ids=tok)
    assert err_ref == 3
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    ids, w = api.moe_route_ex(x.to(cuda_dev), w_r.to(cuda_dev), b.to(cuda_dev), k,
                              tid2eid=torch.from_numpy(table).to(cuda_dev),
                              token_ids=torch.from_numpy(tok).to(cuda_dev), dev_err=err)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), w_ref.view(np.uint32))
    assert int(err) == err_ref


@pytest.mark.parametrize("T", [3, 40])
def test_route_ties_and_zero_bias(cuda_dev, T):
    """Equal keys go to the lower id, NaN keys rank after every number (T = 3: the small-batch
    kernel; T = 40: the tiled logits and the warp top k)."""
    d, E, k = 64, 16, 6
    x = synth.x_bf16(2, 0, 0, T, d)
    w_r = torch.zeros((d, E))
    b = torch.zeros(E)
    b[9] = 0.25
    b[12] = 0.25
    bn = torch.full((E,), float("nan"))   # only experts 2, 7, 11 and 14 have a number
    bn[2] = 0.1
    bn[7] = -0.2
    bn[11] = 0.1
    bn[14] = 0.3
    for bias in (None, b, bn):
        ids_ref, w_ref = oracle.route(x, w_r, bias, k)
        ids, w = api.moe_route(x.to(cuda_dev), w_r.to(cuda_dev), None if bias is None else bias.to(cuda_dev), k)
        assert np.array_equal(ids.cpu().numpy(), ids_ref)
        assert np.array_equal(w.cpu().numpy(), w_ref)


@pytest.mark.parametrize("T,k,E", [(1, 6, 384), (8, 6, 384), (5, 6, 384), (4, 6, 32), (8192, 6, 384), (3000, 8, 1024),
                                   (7, 1, 1)])
def test_permute_bit_exact(cuda_dev, T, k, E):
    rng = np.random.default_rng(T * 31 + E)
    if T == 8192:   # the skewed prefill routing: a few experts take most pairs
        p = np.exp(-np.arange(E) / 3.0)
        p /= p.sum()
        ids = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    else:
        ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32)
    ref = oracle.permute(ids, E)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    got = api.moe_permute(torch.from_numpy(ids).to(cuda_dev), E, dev_err=err)
    for key in ("offsets", "perm", "inv"):
        assert np.array_equal(got[key].cpu().numpy(), ref[key]), key
    na = int(got["n_active"])
    assert na == ref["n_active"]
    assert np.array_equal(got["active"].cpu().numpy()[:na], ref["active"])
    assert np.all(got["active"].cpu().numpy()[na:] == -1)
    assert int(err) == 0


def test_permute_bad_ids(cuda_dev):
    ids = np.array([[0, 5], [40, 1], [-3, 5]], dtype=np.int32)
    ref = oracle.permute(ids, 8)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    got = api.moe_permute(torch.from_numpy(ids).to(cuda_dev), 8, dev_err=err)
    for key in ("offsets", "perm", "inv"):
        assert np.array_equal(got[key].cpu().numpy(), ref[key]), key
    assert int(err) & 1


@pytest.mark.parametrize("T", [5, 40])
def test_expert_ffn_pairs_with_invalid_ids(cuda_dev, T):
    """moe_expert_ffn on a permutation whose ids include -1 and E (both paths: T = 5 decode, T = 40
    grouped GEMM): every valid pair's y row and the shared expert's rows match the oracle's expert
    FFN of that token; the rows of the parked invalid pairs are not written."""
    shape = synth.MoeShape(d=512, E=8, k=3, F=256, F_shared=256, bias_half_width=0.1)
    lw = synth.layer_weights(11, 0, shape)
    routed = api.routed_weights(lw.gate.to(cuda_dev), lw.up.to(cuda_dev), lw.down.to(cuda_dev), shape.d, shape.F)
    shared = FfnWeights(lw.sh_gate.to(cuda_dev), lw.sh_up.to(cuda_dev), lw.sh_down.to(cuda_dev), BRE_FMT_Q8_0,
                        shape.d, shape.F_shared)
    rng = np.random.default_rng(T)
    ids = np.stack([rng.permutation(shape.E)[:shape.k] for _ in range(T)]).astype(np.int32)
    ids[0, 1] = -1
    ids[T // 2, 0] = shape.E
    ids[T - 1, 2] = 1 << 20
    x = synth.x_bf16(11, 0, T, T, shape.d)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    perm = api.moe_permute(torch.from_numpy(ids).to(cuda_dev), shape.E, dev_err=err)
    P = T * shape.k
    y = torch.full((P, shape.d), float("nan"), dtype=torch.float32, device=cuda_dev)
    ys = torch.full((T, shape.d), float("nan"), dtype=torch.float32, device=cuda_dev)
    api.moe_expert_ffn(routed, shared, x.to(cuda_dev), shape.k, perm, dev_err=err, y_pairs=y, y_shared=ys)
    _sync()
    assert int(err) & 1   # the permutation reported the bad ids
    n_valid = int(perm["offsets"][shape.E])
    assert n_valid == P - 3
    inv = perm["inv"].cpu().numpy()
    got = y.cpu().double().numpy()
    assert np.all(np.isnan(got[n_valid:])), "rows of invalid pairs were written"
    rows, refs = [], []
    for q in range(P):
        t, e = q // shape.k, int(ids.reshape(-1)[q])
        if not 0 <= e < shape.E:
            continue
        refs.append(oracle.expert_ffn(BRE_FMT_Q2_K, lw.gate[e].numpy(), lw.up[e].numpy(), lw.down[e].numpy(),
                                      shape.d, shape.F, x[t:t + 1])[0])
        rows.append(got[inv[q]])
    refs.append(oracle.expert_ffn(BRE_FMT_Q8_0, lw.sh_gate.numpy(), lw.sh_up.numpy(), lw.sh_down.numpy(), shape.d,
                                  shape.F_shared, x))
    rows.append(ys.cpu().double().numpy())
    ref, g = np.concatenate([r.reshape(-1, shape.d) for r in refs]), np.concatenate([r.reshape(-1, shape.d) for r in rows])
    assert np.all(np.isfinite(g))
    rms = float(np.sqrt(np.mean(ref * ref)))
    err = np.abs(g - ref)
    if T <= 8:
        # the decode path: the layer bar on these intermediate outputs (exact weights, h in BF16)
        assert float(err.max()) <= 1e-2 * rms
    else:
        # the grouped GEMM holds the dequantised weights and h in BF16, two roundings of at most
        # 2^-9 each per product term that the layer's weighted sum of pairs averages down: the
        # intermediate rows are held to 1e-2 of rms in the rms of the error and 2e-2 in its maximum
        assert float(np.sqrt(np.mean(err * err))) <= 1e-2 * rms
        assert float(err.max()) <= 2e-2 * rms


# --------------------------------------------------------------------------- #
# MoE layer
# --------------------------------------------------------------------------- #

def test_layer_tiny(cuda_dev):
    shape = synth.TINY
    layer = device_layer(SEED, 0, shape, 8, cuda_dev)
    for T in (1, 4, 8):
        for tset in range(3):
            x = synth.x_bf16(SEED, 0, tset, T, shape.d)
            out, of, info = run_layer(layer, x.to(cuda_dev))
            ref = oracle_layer(SEED, 0, shape, x)
            assert np.array_equal(info["ids"].cpu().numpy(), ref["ids"])
            assert_layer_close(out, of, ref)
            assert int(layer.dev_err) == 0


def test_layer_tiny_without_shared_expert(cuda_dev):
    shape = synth.TINY
    layer = device_layer(SEED, 0, shape, 8, cuda_dev, with_shared=False)
    x = synth.x_bf16(SEED, 0, 5, 6, shape.d)
    out, of, info = run_layer(layer, x.to(cuda_dev))
    ref = oracle_layer(SEED, 0, shape, x, with_shared=False)
    assert_layer_close(out, of, ref)


def test_layer_one_expert_all_tokens(cuda_dev):
    # k = E = 1: every token hits the same expert (8 columns of one tile)
    shape = synth.MoeShape(d=512, E=1, k=1, F=256, F_shared=256, bias_half_width=0.0)
    layer = device_layer(3, 0, shape, 8, cuda_dev)
    x = synth.x_bf16(3, 0, 0, 8, shape.d)
    out, of, _ = run_layer(layer, x.to(cuda_dev))
    assert_layer_close(out, of, oracle_layer(3, 0, shape, x))


@pytest.mark.parametrize("scale_exp", [20, -20])
def test_layer_decode_activation_scales(cuda_dev, scale_exp):
    # activations scaled by a power of two (exact in BF16): the intermediate h then lies far
    # outside FP16's range (~2^40 or ~2^-40), which the decode path's shared down projection, fed
    # h as FP16 scaled per 32-row block, has to absorb; the grouped-GEMM path is run on the same
    shape = synth.TINY
    layer = device_layer(SEED, 0, shape, 64, cuda_dev)
    for T in (1, 5, 64):   # 64: the grouped-GEMM path, whose intermediate stays BF16
        x = (synth.x_bf16(SEED, 0, 40 + T, T, shape.d).float() * 2.0 ** scale_exp).to(torch.bfloat16)
        out, of, info = run_layer(layer, x.to(cuda_dev))
        ref = oracle_layer(SEED, 0, shape, x)
        assert np.array_equal(info["ids"].cpu().numpy(), ref["ids"])
        assert_layer_close(out, of, ref)
        assert int(layer.dev_err) == 0


@pytest.mark.parametrize("E,k,T", [(64, 8, 8), (96, 12, 8), (80, 11, 6)])
def test_layer_decode_many_pairs(cuda_dev, E, k, T):
    # decode batches with many (token, expert) pairs: up to 96 pairs over up to 96 active experts
    shape = synth.MoeShape(d=512, E=E, k=k, F=256, F_shared=256, bias_half_width=0.1)
    layer = device_layer(5, 0, shape, 8, cuda_dev)
    x = synth.x_bf16(5, 0, 1, T, shape.d)
    out, of, info = run_layer(layer, x.to(cuda_dev))
    ref = oracle_layer(5, 0, shape, x)
    assert np.array_equal(info["ids"].cpu().numpy(), ref["ids"])
    assert_layer_close(out, of, ref)
    assert int(layer.dev_err) == 0


def test_layer_decode_full_shape(cuda_dev):
    # every decode batch size: each has its own K-part plan for the two phases
    shape = synth.V41
    layer = device_layer(SEED, 0, shape, 8, cuda_dev)
    for T in range(1, 9):
        x = synth.x_bf16(SEED, 0, 100 + T, T, shape.d)
        out, of, info = run_layer(layer, x.to(cuda_dev))
        ref = oracle_layer(SEED, 0, shape, x, threads=4)
        assert np.array_equal(info["ids"].cpu().numpy(), ref["ids"])
        assert_layer_close(out, of, ref)
        assert int(layer.dev_err) == 0


def test_layer_workspace_shared_across_paths(cuda_dev):
    """One workspace serves decode calls (which keep K-part counters in it between calls) and a
    grouped-GEMM call in between; the repeated decode call is bit-identical."""
    shape = synth.V41
    layer = device_layer(SEED, 0, shape, 64, cuda_dev)
    x8 = synth.x_bf16(SEED, 0, 41, 8, shape.d).to(cuda_dev)
    x2 = synth.x_bf16(SEED, 0, 42, 2, shape.d).to(cuda_dev)
    x64 = synth.x_bf16(SEED, 0, 43, 64, shape.d).to(cuda_dev)
    a, _ = layer.forward(x8)
    a = a.clone()
    layer.forward(x2)
    layer.forward(x64)
    b, _ = layer.forward(x8)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert int(layer.dev_err) == 0


def test_layer_repeatable(cuda_dev):
    shape = synth.V41
    layer = device_layer(SEED, 0, shape, 8, cuda_dev)
    x = synth.x_bf16(SEED, 0, 7, 8, shape.d).to(cuda_dev)
    a, _ = layer.forward(x)
    b, _ = layer.forward(x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_residual_norm_bit_exact(cuda_dev):
    x = (synth.x_bf16(SEED, 0, 0, 5, 4096).float() * 13).to(torch.bfloat16)
    m = synth.x_bf16(SEED, 0, 1, 5, 4096)
    s = float(np.float32(1 / math.sqrt(2)))
    xo, uo = api.moe_residual_norm(x.to(cuda_dev), m.to(cuda_dev), s, 1e-6)
    xr = oracle.residual(x, m, s)
    ur = oracle.rmsnorm(torch.from_numpy(xr.view(np.int16)).view(torch.bfloat16), 1e-6)
    assert np.array_equal(bf16_bits(xo), xr)
    assert np.array_equal(bf16_bits(uo), ur)


# --------------------------------------------------------------------------- #
# grouped-GEMM path (T > 8)
# --------------------------------------------------------------------------- #

@pytest.mark.parametrize("T", [9, 64, 300])
def test_layer_gemm_tiny_ragged(cuda_dev, T):
    shape = synth.TINY
    layer = device_layer(SEED, 0, shape, T, cuda_dev)
    x = synth.x_bf16(SEED, 0, 50 + T, T, shape.d)
    out, of, info = run_layer(layer, x.to(cuda_dev))
    ref = oracle_layer(SEED, 0, shape, x)
    assert np.array_equal(info["ids"].cpu().numpy(), ref["ids"])
    assert_layer_close(out, of, ref)
    assert int(layer.dev_err) == 0


def test_layer_gemm_matches_decode_path(cuda_dev):
    # the same 8 tokens through both paths (a 9th token forces the GEMM path)
    shape = synth.TINY
    x9 = synth.x_bf16(SEED, 0, 77, 9, shape.d)
    layer = device_layer(SEED, 0, shape, 9, cuda_dev)
    _, f9, _ = run_layer(layer, x9.to(cuda_dev))
    _, f8, _ = run_layer(layer, x9[:8].contiguous().to(cuda_dev))
    a = f9[:8].cpu().numpy()
    b = f8.cpu().numpy()
    rms = float(np.sqrt(np.mean(b.astype(np.float64) ** 2)))
    assert np.max(np.abs(a - b)) <= 1e-2 * rms


def test_layer_prefill_full_shape_sampled(cuda_dev):
    shape, T = synth.V41_PREFILL, 8192
    layer = device_layer(SEED, 0, shape, T, cuda_dev)
    x = synth.x_bf16(SEED, 0, 0, T, shape.d)
    out, of, info = run_layer(layer, x.to(cuda_dev))
    ids = info["ids"].cpu().numpy()
    # sample: the first and last tokens plus tokens that cover every active expert
    chosen = {0, T - 1}
    seen = set()
    for t in range(T):
        new = set(ids[t]) - seen
        if new:
            chosen.add(t)
            seen |= new
        if len(chosen) >= 24:
            break
    sample = np.array(sorted(chosen))
    ref = oracle_layer(SEED, 0, shape, x[sample])
    assert np.array_equal(ids[sample], ref["ids"])
    assert_layer_close(out[sample], of[sample], ref)
    assert int(layer.dev_err) == 0


def test_layer_prefill_every_m_tile_sampled(cuda_dev):
    """The prefill layer (T = 8192, Zipf-skewed routing) on a sample that reaches every 256-pair
    M tile of every active expert's group (one pair at a varying row inside each tile, plus each
    group's last pair, so the ragged last tiles are in) and every 256-token tile of the shared
    expert; the oracle runs on the sampled tokens."""
    shape, T = synth.V41_PREFILL, 8192
    layer = device_layer(SEED, 0, shape, T, cuda_dev)
    x = synth.x_bf16(SEED, 0, 0, T, shape.d)
    out, of, info = run_layer(layer, x.to(cuda_dev))
    ids = info["ids"].cpu().numpy()
    offsets = info["offsets"].cpu().numpy()
    perm = info["perm"].cpu().numpy()
    k = shape.k
    chosen = set()
    n_group_tiles = 0
    for e in range(shape.E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for m, start in enumerate(range(lo, hi, 256)):
            n = min(256, hi - start)
            chosen.add(int(perm[start + (37 * m + 11) % n]) // k)
            n_group_tiles += 1
        if hi > lo:
            chosen.add(int(perm[hi - 1]) // k)
    for m in range(T // 256):                       # the shared expert's M tiles (all tokens)
        chosen.add(256 * m + (53 * m) % 256)
    sample = np.array(sorted(chosen))
    assert n_group_tiles >= (T * k) // 256
    ref = oracle_layer(SEED, 0, shape, x[sample], threads=16)
    assert np.array_equal(ids[sample], ref["ids"])
    assert_layer_close(out[sample], of[sample], ref)
    assert int(layer.dev_err) == 0


def test_layer_gemm_tiny_dominant_expert(cuda_dev):
    """Grouped-GEMM path with one expert holding every token: 900 pairs = three full 256-pair M
    tiles and a ragged fourth; the whole [T, d] output is compared with the oracle."""
    shape, T = synth.TINY, 900
    lw = synth.layer_weights(SEED, 0, shape, device=cuda_dev)
    bias = synth.route_bias(SEED, 0, shape.E, shape.bias_half_width).clone()
    bias[5] += 4.0                                  # sigmoid scores lie in (0, 1): expert 5 always wins
    layer = MoeLayer(lw.w_r.to(cuda_dev), bias.to(cuda_dev), api.routed_weights(lw.gate, lw.up, lw.down, shape.d, shape.F),
                     FfnWeights(lw.sh_gate, lw.sh_up, lw.sh_down, BRE_FMT_Q8_0, shape.d, shape.F_shared), shape.k, T)
    x = synth.x_bf16(SEED, 0, 61, T, shape.d)
    out, of, info = run_layer(layer, x.to(cuda_dev))
    offsets = info["offsets"].cpu().numpy()
    assert offsets[6] - offsets[5] == T
    ref = oracle_layer(SEED, 0, shape, x, bias=bias, threads=8)
    assert np.array_equal(info["ids"].cpu().numpy(), ref["ids"])
    assert_layer_close(out, of, ref)
    assert int(layer.dev_err) == 0


# --------------------------------------------------------------------------- #
# verify batch through a 24-layer stack (teacher-forced per layer)
# --------------------------------------------------------------------------- #

def test_verify_stack_24_layers_teacher_forced(cuda_dev):
    shape, T, L = synth.V41, 5, 24
    layers = [device_layer(SEED, l, shape, T, cuda_dev) for l in range(L)]
    stack = api.MoeStack(layers)
    x0 = synth.x_bf16(SEED, 0, 999, T, shape.d).to(cuda_dev)
    trace = []
    xf = stack.forward(x0, trace=trace)
    torch.cuda.synchronize()
    assert torch.isfinite(xf.float()).all()
    for l in (0, 11, 23):
        x_l, u_l, out_l, f_l, info = trace[l]
        # the norm of the layer input is bit-exact
        u_ref = oracle.rmsnorm(x_l.cpu(), 1e-6)
        assert np.array_equal(bf16_bits(u_l), u_ref)
        # ids bit-exact and the layer output within tolerance, on the device's own input
        ref = oracle_layer(SEED, l, shape, u_l.cpu())
        assert np.array_equal(info["ids"].cpu().numpy(), ref["ids"])
        assert_layer_close(out_l, f_l, ref)
        # the residual update is bit-exact given the layer output
        nxt = trace[l + 1][0] if l + 1 < L else xf
        assert np.array_equal(bf16_bits(nxt), oracle.residual(x_l.cpu(), out_l.cpu(), stack.scale))


# --------------------------------------------------------------------------- #
# Engram gate and residual injection
# --------------------------------------------------------------------------- #

def _bf16_ulp(a):
    """Spacing of BF16 at |a| (2^(e-7) for normal values)."""
    a = np.abs(np.asarray(a, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("T,R,W", [(1, 24, 5120), (8, 24, 5120), (5, 2, 256), (11, 3, 512), (20, 1, 128)])
def test_engram_inject_parity(cuda_dev, T, R, W):
    """engram_inject against the FP64 oracle: kv within the FP32 dot-product bound, gates within
    1e-4, every updated BF16 value within one BF16 step of the result plus one step of the value
    times the gate (the two roundings either side may take), masked tokens byte for byte."""
    nrows = 4096
    table = synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE, 5), nrows)
    ids = synth.engram_ids_uniform(SEED + T, T * R, nrows).view(T, R)
    K, N = 256 * R, 5 * W
    w_kv = synth.engram_kv_weight(SEED, R, N, K)
    resid = synth.engram_residual(SEED, 0, T, T, W)
    qn = synth.engram_norm_weights(SEED, 0, 0, W)
    kn = synth.engram_norm_weights(SEED, 0, 1, W)
    mask = (np.arange(T) % 3 == 2).astype(np.uint8)
    rows_bits, err_ref = oracle.engram_gather([table] * R, ids.numpy().reshape(T, R, 1))
    rows = torch.from_numpy(rows_bits.view(np.int16)).view(torch.bfloat16)
    kv_ref = oracle.engram_kv(rows, w_kv)
    out_ref, g_ref = oracle.engram_gate(kv_ref, resid, qn, kn, mask=mask)
    dv = cuda_dev
    r_gpu = resid.to(dv).clone()
    kv = torch.empty((T, N), dtype=torch.float32, device=dv)
    g = torch.empty((T, 4), dtype=torch.float32, device=dv)
    err = torch.zeros(1, dtype=torch.int32, device=dv)
    api.engram_inject(table.to(dv), ids.to(dv), w_kv.to(dv), r_gpu, qn.to(dv), kn.to(dv),
                      mask=torch.from_numpy(mask).to(dv), kv_out=kv, gate_out=g, dev_err=err)
    assert int(err) == err_ref == 0
    # kv: FP32 accumulation of K exact products (tensor-core sums, then K parts in order)
    mag = np.abs(rows.double().numpy()) @ np.abs(w_kv.double().numpy()).T
    bound = (K + 8) * 2.0 ** -23 * mag
    assert np.all(np.abs(kv.cpu().double().numpy() - kv_ref) <= bound)
    gg = g.cpu().double().numpy()
    assert np.all(gg[mask == 1] == 0)
    assert np.max(np.abs(gg - g_ref)[mask == 0]) <= 1e-4
    got = r_gpu.cpu()
    rb = resid.view(torch.int16).numpy().view(np.uint16)
    gb = got.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(gb[mask == 1], rb[mask == 1])
    ref_f = torch.from_numpy(out_ref.view(np.int16)).view(torch.bfloat16).double().numpy()
    got_f = got.double().numpy()
    v_ref = kv_ref[:, 4 * W:][:, None, :]
    tol = _bf16_ulp(ref_f) + g_ref[:, :, None] * _bf16_ulp(v_ref) + 1e-4 * np.abs(v_ref)
    assert np.all(np.abs(got_f - ref_f)[mask == 0] <= tol[mask == 0])


def test_engram_inject_bad_rows_and_repeat(cuda_dev):
    """Row ids outside the table decode as zeros and set BRE_DEVERR_ROW_ID (as the oracle's
    gather); a second call on the same workspace gives the same bits."""
    T, R, W, nrows = 4, 2, 256, 512
    table = synth.engram_table(SEED, synth.stream(synth.S_ENGRAM_TABLE, 6), nrows)
    ids = synth.engram_ids_uniform(SEED, T * R, nrows).view(T, R).clone()
    ids[1, 0] = nrows
    ids[2, 1] = -5
    w_kv = synth.engram_kv_weight(SEED, 9, 5 * W, 256 * R)
    resid = synth.engram_residual(SEED, 1, 0, T, W)
    qn = synth.engram_norm_weights(SEED, 1, 0, W)
    kn = synth.engram_norm_weights(SEED, 1, 1, W)
    rows_bits, err_ref = oracle.engram_gather([table] * R, ids.numpy().reshape(T, R, 1))
    assert err_ref == 2
    kv_ref = oracle.engram_kv(torch.from_numpy(rows_bits.view(np.int16)).view(torch.bfloat16), w_kv)
    _, g_ref = oracle.engram_gate(kv_ref, resid, qn, kn)
    dv = cuda_dev
    ws = torch.zeros(api.engram_inject_workspace(T, R, W), dtype=torch.uint8, device=dv)
    outs = []
    for _ in range(2):
        r_gpu = resid.to(dv).clone()
        g = torch.empty((T, 4), dtype=torch.float32, device=dv)
        err = torch.zeros(1, dtype=torch.int32, device=dv)
        api.engram_inject(table.to(dv), ids.to(dv), w_kv.to(dv), r_gpu, qn.to(dv), kn.to(dv), gate_out=g,
                          dev_err=err, ws=ws)
        assert int(err) == 2
        assert np.max(np.abs(g.cpu().double().numpy() - g_ref)) <= 1e-4
        outs.append(r_gpu.cpu())
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
