// Expert FFN for decode-sized batches (at most 8 tokens per expert).
//
// Strata-DSV4.1 README, V4-Flash "How it works" (experts, then the finish step:
// shared expert + routed sum) and "Verifying it" (the expert tier is checked
// against a dequantised F32 reference); SwiGLU from the V4-Flash description.
//
// Design (GB300): the path is bound by streaming 2-bit weights from HBM, so every
// byte is read once.  Each warp owns a two-stage ring in shared memory that the TMA
// engine fills with 16-row chunks of one expert matrix (one tensor copy per chunk, or
// one bulk copy when a whole 16-row tile fits a stage); the warp dequantises in
// registers straight into mma.sync A fragments and multiplies by the expert's tokens
// (N = 8 columns).  Work items (expert, 16-row tile) are handed out by an atomic
// counter so that busy SMs take fewer items.
//
// Exactness: a Q2_K weight is (d*sc)*q - dmin*m.  The A fragment holds the
// integer 128 + sc*q (exact in BF16), so one 256-weight block contributes
//   d * (P' - 128*X) - dmin * (M' - 128*X)
// with P' = sum (128 + sc*q) x, M' = sum_j (128 + m_j) X_j, X_j the 16-value
// sub-block sums of the activations (three BF16 limbs) and X = sum_j X_j.  A Q8_0
// weight d*q is split into nibbles: q + 128 = 16*hi + lo, each held as 128 + nibble.
// Products are exact; accumulation is FP32.
//
// K order: the MMA sums over k, so the k order inside a block is free as long as A
// and B agree.  For Q2_K, step (jj, s) of thread t uses sub-block 4t+jj and codes
// s, 4+s, 8+s, 12+s of it (the four codes of one byte lane after one shift), and the
// activations are stored permuted to match.  Q8_0 uses natural order.
#include <algorithm>
#include <mutex>

#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

namespace {

constexpr int NS = 2;                 // ring stages per warp
constexpr int STAGE = 5376;           // bytes per stage: 16 rows x 336 B of one matrix
constexpr int MAX_WARPS = 16;         // phase 1 (at most 128 registers a thread; fewer when the
                                      // activation package leaves less shared memory)
constexpr int MAX_WARPS_P2 = 16;      // phase 2 (at most 128 registers a thread)
constexpr uint32_t SEL_LO = 0x4140u;  // bytes 0,1 -> (128+b0, 128+b1) as bf16x2
constexpr uint32_t SEL_HI = 0x4342u;  // bytes 2,3
constexpr long long WAIT_LIMIT = 2000000000LL;  // cycles (~1 s) before a wait gives up
constexpr int BAR_BYTES = 512;                  // mbarrier region: MAX_WARPS * NS ring barriers + package barrier
static_assert((MAX_WARPS * NS + 1) * 8 <= BAR_BYTES, "mbarrier region too small");

// n / d as a multiply and shift, for 0 <= n < 2^31 (round-up multiplier m = ceil(2^(31+l) / d),
// 2^l >= d; the error n (m - 2^(31+l)/d) / 2^(31+l) stays below 1/d, so the floor is exact).
struct FDiv {
  uint32_t m;
  int sh;
};
__host__ __device__ __forceinline__ int fdiv(int n, FDiv f) {
  return (int)(((unsigned long long)(unsigned)n * f.m) >> f.sh);
}
static FDiv make_fdiv(unsigned d) {
  int l = 0;
  while ((1ull << l) < d) ++l;
  return FDiv{(uint32_t)(((1ull << (31 + l)) + d - 1) / d), 31 + l};
}

// Bit patterns the dequant combines with every weight word, held in registers (kernel
// parameters) rather than rebuilt as immediates inside the loops: m43 = 0x43004300 (BF16 128 in
// both halves, the exponent OR-ed onto codes), k43 = 0x43434343 (PRMT source of that exponent
// byte), m128 = 0xC300C300 (BF16 -128 in both halves).
struct DecConst {
  uint32_t m43, k43, m128;
};

struct DecParams {
  const uint8_t* rw0;  // routed: phase 1 gate, phase 2 down
  const uint8_t* rw1;  // routed: phase 1 up
  long long rs0, rs1;  // routed expert strides (bytes)
  const uint8_t* sw0;  // shared expert (Q8_0): phase 1 gate, phase 2 down
  const uint8_t* sw1;  // shared: phase 1 up
  int has_shared;
  int d, F, Fs, T, k;
  int rows_r, rows_s;  // rows per matrix of a routed / the shared expert
  int nb_r, nb_s;      // blocks per row
  int cb_r, cb_s;      // blocks per chunk
  int whole_r, whole_s;
  const uint16_t* x;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* n_active;
  int E;
  uint16_t* hB;   // routed h (BF16), permuted: [P][F/256][4][4][4][4]
  uint16_t* HBm;  // routed sub-block sums of h, 3 limbs: [P][F/256][4][3][4]
  uint16_t* hS;   // shared h, natural, 2 limbs: [T][2][Fs]
  float* HS16;    // shared 16-row sums of h: [T][Fs/16]
  float* y_pairs;
  float* y_shared;
  int* counters;
  int32_t* err;
  int xstride;  // bytes per token row of the permuted activations in shared memory
  const unsigned char* pkg;  // activation package in global memory (phase 1)
  DecConst kc;
  int kp_r, kp_s;            // K parts per 16-row tile: items are (tile, K part)
  int C_r, C_s;              // chunks per matrix row of a routed / the shared expert
  int cpi_r, cpi_s;          // chunks per matrix in one item (C / K parts)
  FDiv fd_kps, fd_kpr, fd_trk, fd_k;   // divisors: K parts (shared, routed), routed tiles * K parts, k
  float* part_r;             // routed partial sums: [pair position][tile][K part][16 rows] x (gate, up)
                             // in phase 1, x (y) in phase 2
  float* part_s;             // shared partial sums: [token][tile][K part][16 rows] x (2 | 1)
  int* tile_cnt;             // per tile count of finished K parts (zero between calls)
};

struct Item {
  int id;       // -1: none
  bool shared;
  int e, off, n;
  int tile;
  int nb, cb, C, whole, bb;
  int KP, kp;   // K parts of the tile and this item's part
  int cpi;      // chunks per matrix in this item (C / KP)
  int nch;      // chunks of the item: cpi per matrix, gate then up in phase 1
  int slot;     // tile index for the K-part fix-up
  const uint8_t* src0;
  const uint8_t* src1;
};

template <int PHASE>
__device__ __forceinline__ Item decode_item(const DecParams& p, int id, int n_act, int tiles_s, int tiles_r) {
  Item it;
  it.id = id;
  if (id < 0) return it;
  const int kps = p.kp_s, kpr = p.kp_r;
  if (id < tiles_s * kps) {
    it.shared = true;
    it.tile = fdiv(id, p.fd_kps);
    it.KP = kps;
    it.kp = id - it.tile * kps;
    it.slot = it.tile;
    it.e = -1;
    it.off = 0;
    it.n = p.T;
    it.nb = p.nb_s;
    it.cb = p.cb_s;
    it.whole = p.whole_s;
    it.bb = Q80_BB;
    it.src0 = p.sw0;
    it.src1 = p.sw1;
  } else {
    const int r = id - tiles_s * kps;
    const int a = fdiv(r, p.fd_trk), rt = r - a * (tiles_r * kpr);
    it.shared = false;
    it.tile = fdiv(rt, p.fd_kpr);
    it.KP = kpr;
    it.kp = rt - it.tile * kpr;
    it.slot = tiles_s + a * tiles_r + it.tile;
    it.e = __ldg(p.active + a);
    if ((unsigned)it.e >= (unsigned)p.E) {
      // an expert id the weights do not hold: no columns, and no copy outside the weights
      set_err(p.err, BRE_DEVERR_EXPERT_ID);
      it.e = 0;
      it.off = 0;
      it.n = 0;
    } else {
      it.off = __ldg(p.offsets + it.e);
      it.n = __ldg(p.offsets + it.e + 1) - it.off;
    }
    it.nb = p.nb_r;
    it.cb = p.cb_r;
    it.whole = p.whole_r;
    it.bb = Q2K_BB;
    it.src0 = p.rw0 + (long long)it.e * p.rs0;
    it.src1 = (PHASE == 1) ? p.rw1 + (long long)it.e * p.rs1 : nullptr;
  }
  it.C = it.shared ? p.C_s : p.C_r;
  it.cpi = it.shared ? p.cpi_s : p.cpi_r;
  it.nch = (PHASE == 1 ? 2 : 1) * it.cpi;
  return it;
}


// Lane 0 issues the copy of chunk cc of `it` into `stage`: one bulk copy of a whole 16-row tile,
// or one tensor copy of a 16-row x cb-block box (maps: [experts][rows][row words]).
template <int PHASE>
__device__ __forceinline__ void issue_chunk(const Item& it, int cc, unsigned char* stage, uint64_t* bar, int lane,
                                            const CUtensorMap* map0, const CUtensorMap* map1) {
  if (lane != 0) return;
  const int m = (PHASE == 1 && cc >= it.cpi) ? 1 : 0;
  const int c = it.kp * it.cpi + (cc - m * it.cpi);
  const int chunk_bytes = it.cb * it.bb;
  const uint32_t bytes = 16u * chunk_bytes;
  mbar_arrive_expect_tx(bar, bytes);
  if (it.whole) {
    const uint8_t* src = (m ? it.src1 : it.src0) + (long long)it.tile * 16 * chunk_bytes;
    bulk_g2s(stage, src, bytes, bar);
  } else {
    tma_load_3d(stage, m ? map1 : map0, c * (chunk_bytes / 4), it.tile * 16, it.shared ? 0 : it.e, bar);
  }
}

__device__ __forceinline__ uint32_t lds_u32(const unsigned char* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint32_t lds_u16(const unsigned char* p) {
  return *reinterpret_cast<const unsigned short*>(p);
}
__device__ __forceinline__ uint32_t lds_u32_a2(const unsigned char* p) {  // 2-byte aligned
  return lds_u16(p) | (lds_u16(p + 2) << 16);
}

// Q2_K A fragments of one row for step s, codes left in place: one LOP3 per register gives the
// BF16 pair 128 + c * 4^e (e = min(s, 2); the code occupies mantissa bits 2e, 2e+1).  lo holds
// codes (s, 8+s) of the sub-block word (bytes 0 and 2), hi codes (4+s, 12+s) (bytes 1 and 3).
// m43 is the exponent pattern 0x43004300 held in a register (a kernel parameter, so that the
// mask can be the instruction's immediate and the OR needs no second instruction).
__device__ __forceinline__ void q2k_pairs(uint32_t w, int s, uint32_t m43, uint32_t& lo, uint32_t& hi) {
  if (s < 3) {
    const uint32_t m = 0x00030003u << (2 * s);
    lo = (w & m) | m43;
    hi = ((w >> 8) & m) | m43;
  } else {
    const uint32_t m = 0x00030003u << 4;
    lo = ((w >> 2) & m) | m43;
    hi = ((w >> 10) & m) | m43;
  }
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// (sc, sc) and (-128 sc, -128 sc) as BF16 pairs for one sub-block byte of a scales word
// (exact); sel selects the byte (RotConst), k43 is 0x43434343 and m43 0x43004300 (128, 128),
// m128 0xC300C300 (-128, -128): registers (kernel parameters), so that no constant is
// rebuilt inside the loops.
__device__ __forceinline__ void q2k_scale_pairs(uint32_t sclo, uint32_t sel, const DecConst& k, uint32_t& sc2,
                                                uint32_t& nsc2) {
  const uint32_t u = prmt(sclo, k.k43, sel);   // 128 + sc
  sc2 = bf16x2_sub(u, k.m43);                  // sc
  nsc2 = bf16x2_mul(sc2, k.m128);              // -128 sc
}

// Fragment step jj of thread quad t works on sub-block 4t + rot_sub(t, jj) of a block.  Rotating
// the sub-block with t spreads one load instruction's code words over all 32 banks: the 16 rows
// of a stage lie 84 * cb bytes apart, a multiple of four words, so a common sub-block would put
// four of a warp's 32 words in each of 8 banks.
__host__ __device__ __forceinline__ int rot_sub(int t, int jj) { return (t + jj) & 3; }

// Per-thread constants of the rotation: byte offsets of the code words inside a block row and
// PRMT selectors of the matching scale bytes, for steps jj = 0..3.
struct RotConst {
  int qoff[4];
  uint32_t ssel[4];
};

__device__ __forceinline__ RotConst rot_const(int t) {
  RotConst r;
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int j = rot_sub(t, jj);
    r.qoff[jj] = 16 + 16 * t + 4 * j;
    r.ssel[jj] = (uint32_t)(j * 0x0101 + 0x4040);
  }
  return r;
}

// A fragments of the min-term MMA: the 4-bit mins of the lane's four sub-blocks for rows g
// (scales word sw0) and g + 8 (sw1) as exact BF16 pairs, m = (128 + m) - 128.
__device__ __forceinline__ void min_frags(uint32_t sw0, uint32_t sw1, const DecConst& k, uint32_t& A0, uint32_t& A1,
                                          uint32_t& A2, uint32_t& A3) {
  const uint32_t mg = (sw0 >> 4) & 0x0F0F0F0Fu, mg8 = (sw1 >> 4) & 0x0F0F0F0Fu;
  A0 = bf16x2_sub(prmt(mg, k.k43, SEL_LO), k.m43);
  A1 = bf16x2_sub(prmt(mg8, k.k43, SEL_LO), k.m43);
  A2 = bf16x2_sub(prmt(mg, k.k43, SEL_HI), k.m43);
  A3 = bf16x2_sub(prmt(mg8, k.k43, SEL_HI), k.m43);
}

// Q8_0 nibble planes of one row word (4 consecutive int8): (128+lo) and (128+hi') pairs.
__device__ __forceinline__ void q80_frag(uint32_t w, uint32_t k43, uint32_t& lo01, uint32_t& lo23, uint32_t& hi01,
                                         uint32_t& hi23) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = ((w >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;
  lo01 = prmt(lo, k43, SEL_LO);
  lo23 = prmt(lo, k43, SEL_HI);
  hi01 = prmt(hi, k43, SEL_LO);
  hi23 = prmt(hi, k43, SEL_HI);
}

// ----------------------------------------------------------------------------
// phase 1, routed Q2_K: 16 rows of one matrix (gate or up) over one chunk
// ----------------------------------------------------------------------------
// The block loop stays rolled (unrolled it outgrows the instruction cache); CB > 0 fixes the
// chunk's block count at compile time so that addresses are base + immediate, CB == 0 takes cb_rt.
template <int CB>
__device__ __forceinline__ void p1_q2k_mat(const unsigned char* stage, int cb_rt, int c, int g, int t,
                                           const unsigned char* xb_g,    // permuted x of column g
                                           const unsigned char* xbm_g,   // XBm of column g
                                           const RotConst& rc, const DecConst& k, float (&acc)[4]) {
  const int cb = CB > 0 ? CB : cb_rt;
  const int chunk_bytes = cb * Q2K_BB;
#pragma unroll 1
  for (int bl = 0; bl < cb; ++bl) {
    const int b = c * cb + bl;
    uint32_t qw[2][4], sw[2], dd[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const unsigned char* base = stage + (g + 8 * rr) * chunk_bytes + bl * Q2K_BB;
      sw[rr] = lds_u32(base + 4 * t);
      dd[rr] = lds_u32(base + 80);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) qw[rr][jj] = lds_u32(base + rc.qoff[jj]);
    }
    // one accumulator chain, started by a C = 0 MMA (the MMAs are far apart in the instruction
    // stream, so the chain costs no waiting)
    float P[4], M[4];
    const unsigned char* xblk = xb_g + b * 512;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint32_t sc2[2], nsc2[2];
      q2k_scale_pairs(sw[0] & 0x0F0F0F0Fu, rc.ssel[jj], k, sc2[0], nsc2[0]);
      q2k_scale_pairs(sw[1] & 0x0F0F0F0Fu, rc.ssel[jj], k, sc2[1], nsc2[1]);
      uint4 bq[2];   // steps s = 0, 1 and 2, 3: one 16-byte load each
#pragma unroll
      for (int sp = 0; sp < 2; ++sp) bq[sp] = *reinterpret_cast<const uint4*>(xblk + ((jj * 2 + sp) * 4 + t) * 16);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint2 bv = (s & 1) ? make_uint2(bq[s >> 1].z, bq[s >> 1].w) : make_uint2(bq[s >> 1].x, bq[s >> 1].y);
        uint32_t a0, a1, a2, a3;
        q2k_pairs(qw[0][jj], s, k.m43, a0, a2);
        q2k_pairs(qw[1][jj], s, k.m43, a1, a3);
        a0 = bf16x2_fma(a0, sc2[0], nsc2[0]);
        a2 = bf16x2_fma(a2, sc2[0], nsc2[0]);
        a1 = bf16x2_fma(a1, sc2[1], nsc2[1]);
        a3 = bf16x2_fma(a3, sc2[1], nsc2[1]);
        if (jj == 0 && s == 0)
          mma_bf16_16816_z(P, a0, a1, a2, a3, bv.x, bv.y);
        else
          mma_bf16_16816(P, a0, a1, a2, a3, bv.x, bv.y);
      }
    }
    // min term: M = sum_j m_j X_j over the 16 sub-blocks, X_j in three limbs
    {
      uint32_t A0, A1, A2, A3;
      min_frags(sw[0], sw[1], k, A0, A1, A2, A3);
#pragma unroll
      for (int limb = 0; limb < 3; ++limb) {
        const uint2 bm = *reinterpret_cast<const uint2*>(xbm_g + ((b * 4 + t) * 3 + limb) * 8);
        if (limb == 0)
          mma_bf16_16816_z(M, A0, A1, A2, A3, bm.x, bm.y);
        else
          mma_bf16_16816(M, A0, A1, A2, A3, bm.x, bm.y);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t ddv = dd[i >> 1];
      const float dv = f16_bits_to_f32(ddv & 0xFFFFu), dmv = f16_bits_to_f32(ddv >> 16);
      acc[i] = fmaf(dv, P[i], fmaf(-dmv, M[i], acc[i]));
    }
  }
}

// ----------------------------------------------------------------------------
// phase 1, shared Q8_0: 16 rows of one matrix over one chunk (natural k order)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void p1_q80_mat(const unsigned char* stage, int cb, int c, int g, int t,
                                           const uint16_t* xrow_g,  // global x row of column g
                                           const float* x32_0, const float* x32_1, uint32_t k43, float (&acc)[4]) {
  const int chunk_bytes = cb * Q80_BB;
  // B (x from global memory) of block bl + 1 loads while block bl is processed
  auto load_b = [&](int bq, uint2 (&b)[2]) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
      b[hf] = __ldg(reinterpret_cast<const uint2*>(xrow_g + 32 * bq + 16 * hf + 4 * t));
  };
  uint2 bcur[2], bnext[2];
  load_b(c * cb, bcur);
  for (int bl = 0; bl < cb; ++bl) {
    const int bq = c * cb + bl;
    if (bl + 1 < cb) load_b(bq + 1, bnext);
    float Ph[4], Pl[4];
    uint32_t dd[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint2 bv = bcur[hf];
      uint32_t l01[2], l23[2], h01[2], h23[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const unsigned char* base = stage + (g + 8 * rr) * chunk_bytes + bl * Q80_BB;
        if (hf == 0) dd[rr] = lds_u16(base);
        q80_frag(lds_u32_a2(base + 2 + 16 * hf + 4 * t), k43, l01[rr], l23[rr], h01[rr], h23[rr]);
      }
      if (hf == 0) {
        mma_bf16_16816_z(Pl, l01[0], l01[1], l23[0], l23[1], bv.x, bv.y);
        mma_bf16_16816_z(Ph, h01[0], h01[1], h23[0], h23[1], bv.x, bv.y);
      } else {
        mma_bf16_16816(Pl, l01[0], l01[1], l23[0], l23[1], bv.x, bv.y);
        mma_bf16_16816(Ph, h01[0], h01[1], h23[0], h23[1], bv.x, bv.y);
      }
    }
    const float x0 = __ldg(x32_0 + bq), x1 = __ldg(x32_1 + bq);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float dv = f16_bits_to_f32(dd[i >> 1]);
      const float xs = (i & 1) ? x1 : x0;
      const float v = fmaf(-2304.0f, xs, fmaf(16.0f, Ph[i], Pl[i]));
      acc[i] = fmaf(dv, v, acc[i]);
    }
    bcur[0] = bnext[0];
    bcur[1] = bnext[1];
  }
}

// B operand of one block for column g: 8 uint4 (h in BF16, fragment order; entry jj * 2 + sp
// holds steps s = 2 sp and 2 sp + 1 of step jj).
struct P2B {
  uint4 v[8];
};

__device__ __forceinline__ void p2_load_b(P2B& B, const uint16_t* __restrict__ hB, int pos_g, int nb, int b, int t) {
  const uint16_t* hblk = hB + ((long long)pos_g * nb + b) * 256;
#pragma unroll
  for (int q = 0; q < 8; ++q) B.v[q] = __ldg(reinterpret_cast<const uint4*>(hblk + (q * 4 + t) * 8));
}

// One 256-column block of 16 rows of the down projection.
// B holds this block's h on entry; each sub-block step, once its MMAs are issued, refills its
// registers with the same step of hnext (the next block's h), so that those loads have a
// whole block of work to arrive.
__device__ __forceinline__ void p2_q2k_block(const unsigned char* blk, int row_bytes, int g, int t, P2B& B,
                                             const uint16_t* __restrict__ hnext, const uint16_t* __restrict__ hm,
                                             const RotConst& rc, const DecConst& k, float (&acc)[4]) {
  // the three limbs of the sub-block sums are first needed at the block's end: loaded here
  uint2 bm[3];
#pragma unroll
  for (int limb = 0; limb < 3; ++limb) bm[limb] = __ldg(reinterpret_cast<const uint2*>(hm + limb * 4));
  uint32_t qw[2][4], sw[2], dd[2];
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const unsigned char* base = blk + (g + 8 * rr) * row_bytes;
    sw[rr] = lds_u32(base + 4 * t);
    dd[rr] = lds_u32(base + 80);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) qw[rr][jj] = lds_u32(base + rc.qoff[jj]);
  }
  // jj outer, s inner (one sub-block's scales live at a time); consecutive MMAs alternate
  // between two accumulators
  float P[2][4], M[4];
  const uint32_t sl0 = sw[0] & 0x0F0F0F0Fu, sl1 = sw[1] & 0x0F0F0F0Fu;
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    uint32_t sc2[2], nsc2[2];
    q2k_scale_pairs(sl0, rc.ssel[jj], k, sc2[0], nsc2[0]);
    q2k_scale_pairs(sl1, rc.ssel[jj], k, sc2[1], nsc2[1]);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      uint32_t a0, a1, a2, a3;
      q2k_pairs(qw[0][jj], s, k.m43, a0, a2);
      q2k_pairs(qw[1][jj], s, k.m43, a1, a3);
      a0 = bf16x2_fma(a0, sc2[0], nsc2[0]);
      a2 = bf16x2_fma(a2, sc2[0], nsc2[0]);
      a1 = bf16x2_fma(a1, sc2[1], nsc2[1]);
      a3 = bf16x2_fma(a3, sc2[1], nsc2[1]);
      const uint4 bq = B.v[jj * 2 + (s >> 1)];
      const uint32_t b0 = (s & 1) ? bq.z : bq.x, b1 = (s & 1) ? bq.w : bq.y;
      if (jj == 0 && s < 2)
        mma_bf16_16816_z(P[s & 1], a0, a1, a2, a3, b0, b1);
      else
        mma_bf16_16816(P[s & 1], a0, a1, a2, a3, b0, b1);
    }
#pragma unroll
    for (int sp = 0; sp < 2; ++sp)
      B.v[jj * 2 + sp] = __ldg(reinterpret_cast<const uint4*>(hnext + ((jj * 2 + sp) * 4 + t) * 8));
  }
  {
    uint32_t A0, A1, A2, A3;
    min_frags(sw[0], sw[1], k, A0, A1, A2, A3);
#pragma unroll
    for (int limb = 0; limb < 3; ++limb) {
      const uint2 b2 = bm[limb];
      if (limb == 0)
        mma_bf16_16816_z(M, A0, A1, A2, A3, b2.x, b2.y);
      else
        mma_bf16_16816(M, A0, A1, A2, A3, b2.x, b2.y);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t ddv = dd[i >> 1];
    const float dv = f16_bits_to_f32(ddv & 0xFFFFu), dmv = f16_bits_to_f32(ddv >> 16);
    acc[i] = fmaf(dv, P[0][i] + P[1][i], fmaf(-dmv, M[i], acc[i]));
  }
}

// ----------------------------------------------------------------------------
// phase 2, routed Q2_K down: 16 rows over one chunk; B = h from global memory, one register
// set refilled a block ahead (the last block of the chunk refills from itself, an L1 hit)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void p2_q2k_chunk(const unsigned char* stage, int cb, int c, int nb, int g, int t,
                                             int pos_g, const uint16_t* __restrict__ hB,
                                             const uint16_t* __restrict__ HBm, const RotConst& rc,
                                             const DecConst& k, float (&acc)[4]) {
  const int chunk_bytes = cb * Q2K_BB;
  const int b0 = c * cb;
  const uint16_t* hcol = hB + (long long)pos_g * nb * 256;              // h of column g, block 0
  const uint16_t* hmcol = HBm + ((long long)pos_g * nb * 4 + t) * 12;   // its sub-block sum limbs
  P2B B;
  p2_load_b(B, hB, pos_g, nb, b0, t);
#pragma unroll 1
  for (int bl = 0; bl < cb; ++bl) {
    const int b = b0 + bl;
    const int bn = bl + 1 < cb ? b + 1 : b;
    p2_q2k_block(stage + bl * Q2K_BB, chunk_bytes, g, t, B, hcol + bn * 256, hmcol + b * 48, rc, k, acc);
  }
}

// ----------------------------------------------------------------------------
// phase 2, shared Q8_0 down: 16 rows over one chunk; B = h limbs (natural order)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void p2_q80_chunk(const unsigned char* stage, int cb, int c, int g, int t, int Fs,
                                             const uint16_t* hrow_g,  // hS[tok_g][0][:]
                                             const float* hs16_0, const float* hs16_1, uint32_t k43, float (&acc)[4]) {
  const int chunk_bytes = cb * Q80_BB;
  // B (both limbs of h) and the 16-row sums of block bl + 1 load while block bl is processed
  auto load_b = [&](int bq, uint2 (&b)[4], float (&xs2)[2]) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      b[2 * hf] = __ldg(reinterpret_cast<const uint2*>(hrow_g + 32 * bq + 16 * hf + 4 * t));
      b[2 * hf + 1] = __ldg(reinterpret_cast<const uint2*>(hrow_g + Fs + 32 * bq + 16 * hf + 4 * t));
    }
    xs2[0] = hs16_0[2 * bq] + hs16_0[2 * bq + 1];
    xs2[1] = hs16_1[2 * bq] + hs16_1[2 * bq + 1];
  };
  uint2 bcur[4], bnext[4];
  float xcur[2], xnext[2];
  load_b(c * cb, bcur, xcur);
  for (int bl = 0; bl < cb; ++bl) {
    const int bq = c * cb + bl;
    if (bl + 1 < cb) load_b(bq + 1, bnext, xnext);
    float Ph[4], Pl[4];
    uint32_t dd[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint2 bh = bcur[2 * hf], blo = bcur[2 * hf + 1];
      uint32_t l01[2], l23[2], h01[2], h23[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const unsigned char* base = stage + (g + 8 * rr) * chunk_bytes + bl * Q80_BB;
        if (hf == 0) dd[rr] = lds_u16(base);
        q80_frag(lds_u32_a2(base + 2 + 16 * hf + 4 * t), k43, l01[rr], l23[rr], h01[rr], h23[rr]);
      }
      if (hf == 0) {
        mma_bf16_16816_z(Pl, l01[0], l01[1], l23[0], l23[1], bh.x, bh.y);
        mma_bf16_16816_z(Ph, h01[0], h01[1], h23[0], h23[1], bh.x, bh.y);
      } else {
        mma_bf16_16816(Pl, l01[0], l01[1], l23[0], l23[1], bh.x, bh.y);
        mma_bf16_16816(Ph, h01[0], h01[1], h23[0], h23[1], bh.x, bh.y);
      }
      mma_bf16_16816(Pl, l01[0], l01[1], l23[0], l23[1], blo.x, blo.y);
      mma_bf16_16816(Ph, h01[0], h01[1], h23[0], h23[1], blo.x, blo.y);
    }
    const float x0 = xcur[0], x1 = xcur[1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float dv = f16_bits_to_f32(dd[i >> 1]);
      const float xs = (i & 1) ? x1 : x0;
      const float v = fmaf(-2304.0f, xs, fmaf(16.0f, Ph[i], Pl[i]));
      acc[i] = fmaf(dv, v, acc[i]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) bcur[q] = bnext[q];
    xcur[0] = xnext[0];
    xcur[1] = xnext[1];
  }
}

__device__ __forceinline__ float silu_mul(float gv, float uv) { return gv / (1.0f + expf(-gv)) * uv; }

// ----------------------------------------------------------------------------
// activation package: x permuted into the Q2_K fragment order, the 16-value sub-block
// sums of x as three BF16 limbs, and 32-value sums for Q8_0.  Built once per call by
// ffn_prep_kernel; phase 1 copies the first two parts into shared memory.
// ----------------------------------------------------------------------------
struct PkgLayout {
  int xB, XBm, X32, total;
};

__host__ __device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }

// bytes per token row of the permuted activations: 16 bytes a lane per load, and a pitch of
// 16 (mod 32) words puts the rows of a quarter warp's loads in different bank halves
__host__ __device__ __forceinline__ int x_stride(int d) { return d * 2 + 64; }

__host__ __device__ __forceinline__ PkgLayout pkg_layout(int T, int d) {
  const int nbx = d / 256, xstride = x_stride(d);
  PkgLayout L;
  L.xB = 0;
  L.XBm = T * xstride;
  L.X32 = L.XBm + T * nbx * 96;
  L.total = L.X32 + round16(T * (d / 32) * 4);
  return L;
}

// grid (d/256, T), 256 threads: thread i owns value k = 256*b + i of token t.
//   xB: x (BF16) permuted into the Q2_K fragment order; XBm: 16-value sub-block sums as
//   three BF16 limbs; X32: 32-value sums (Q8_0 shared expert).
__global__ void __launch_bounds__(256) ffn_prep_kernel(const uint16_t* __restrict__ x, int T, int d,
                                                       unsigned char* __restrict__ pkg) {
  // x was final before the preceding launch (the router) passed its own wait, and nothing before
  // this kernel touches the package, so the work runs first and the wait (which the kernels
  // after this one rely on) comes last: behind a router that triggers early, it overlaps it
  const int b = blockIdx.x, t = blockIdx.y, i = threadIdx.x, lane = i & 31;
  const int nbx = d / 256;
  const PkgLayout L = pkg_layout(T, d);
  const uint32_t v = x[(size_t)t * d + 256 * b + i];
  {
    // fragment order: step (jj, s) of thread tq holds codes s, 8+s | 4+s, 12+s of sub-block
    // 4tq + rot_sub(tq, jj), each activation scaled by 4^-min(s,2) to match the code left in
    // place in the A fragment; steps s = 2sp, 2sp+1 are adjacent (one 16-byte load)
    const int j = i >> 4, tq = j >> 2, jr = j & 3, ip = i & 15;
    const int jj = (jr - tq) & 3;   // the step at which thread quad tq works on sub-block j
    const int byte = ip >> 2, s = ip & 3;
    const int v4 = (byte & 1) * 2 + (byte >> 1);
    const int rem = (((((b * 4 + jj) * 2 + (s >> 1)) * 4 + tq) * 2 + (s & 1)) * 4 + v4);
    const float scaled = __fmul_rn(bf16_bits_to_f32(v), s == 0 ? 1.0f : (s == 1 ? 0.25f : 0.0625f));
    reinterpret_cast<uint16_t*>(pkg + L.xB + (size_t)t * x_stride(d))[rem] = (uint16_t)f32_to_bf16_rne(scaled);
  }
  const float f = bf16_bits_to_f32(v);
  // 16-value sub-block sum (lanes of a half warp), fixed tree order
  float s16 = f;
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) s16 += __shfl_xor_sync(0xffffffffu, s16, o);
  // 32-value sum
  float s32 = s16 + __shfl_xor_sync(0xffffffffu, s16, 16);
  if (lane == 0) reinterpret_cast<float*>(pkg + L.X32)[(size_t)t * (d / 32) + b * 8 + (i >> 5)] = s32;
  if ((i & 15) == 0) {
    const int j = i >> 4;
    const uint32_t hi = f32_to_bf16_rne(s16);
    const float r1 = s16 - bf16_bits_to_f32(hi);
    const uint32_t mid = f32_to_bf16_rne(r1);
    const uint32_t lo = f32_to_bf16_rne(r1 - bf16_bits_to_f32(mid));
    uint16_t* dst = reinterpret_cast<uint16_t*>(pkg + L.XBm + (size_t)t * nbx * 96) + ((b * 4 + (j >> 2)) * 3) * 4 + (j & 3);
    dst[0] = (uint16_t)hi;
    dst[4] = (uint16_t)mid;
    dst[8] = (uint16_t)lo;
  }
  pdl_wait();
}

// ----------------------------------------------------------------------------
// the kernel
// ----------------------------------------------------------------------------
template <int PHASE>
__global__ void __launch_bounds__((PHASE == 1 ? MAX_WARPS : MAX_WARPS_P2) * 32, 1)
    ffn_decode_kernel(const DecParams p, const __grid_constant__ CUtensorMap map_r0,
                      const __grid_constant__ CUtensorMap map_r1, const __grid_constant__ CUtensorMap map_s0,
                      const __grid_constant__ CUtensorMap map_s1) {
  extern __shared__ __align__(128) unsigned char sm[];
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const RotConst rc = rot_const(t);
  unsigned char* stages = sm;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + nw * NS * STAGE);
  uint64_t* pkg_bar = bars + MAX_WARPS * NS;
  unsigned char* xprep = reinterpret_cast<unsigned char*>(bars) + BAR_BYTES;

  pdl_wait();
  if (threadIdx.x < nw * NS) mbar_init(&bars[threadIdx.x], 1);
  if (threadIdx.x == 0) mbar_init(pkg_bar, 1);
  fence_mbar_init();
  __syncthreads();
  const PkgLayout PL = pkg_layout(p.T, p.d);
  if (PHASE == 1 && threadIdx.x == 0) {
    mbar_arrive_expect_tx(pkg_bar, PL.X32);
    bulk_g2s(xprep, p.pkg, PL.X32, pkg_bar);   // xB and XBm (a multiple of 16 bytes)
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) p.counters[PHASE == 1 ? 1 : 0] = 0;

  const int n_act = *p.n_active;
  const int tiles_s = p.has_shared ? p.rows_s / 16 : 0;
  const int tiles_r = p.rows_r / 16;
  const int n_items = tiles_s * p.kp_s + n_act * tiles_r * p.kp_r;

  unsigned char* my_stage = stages + warp * NS * STAGE;
  uint64_t* my_bar = bars + warp * NS;

  auto fetch = [&]() -> int {
    int i = 0;
    if (lane == 0) i = atomicAdd(&p.counters[PHASE - 1], 1);
    i = __shfl_sync(0xffffffffu, i, 0);
    return i < n_items ? i : -1;
  };

  // ids of the items whose chunks are issued but not yet consumed (at most NS + 1).  Phase 1
  // keeps them in three registers (an indexed array would live in local memory); phase 2, at
  // its register limit, keeps the array (touched once per item).
  static_assert(NS + 1 <= 3, "item queue holds three ids");
  int q0 = -1, q1 = -1, q2 = -1, qn = 0;
  int qarr[4];
  int qh = 0, qt = 0;
  auto q_push = [&](int v) {
    if constexpr (PHASE == 1) {
      if (qn == 0) q0 = v;
      else if (qn == 1) q1 = v;
      else q2 = v;
      ++qn;
    } else {
      qarr[qt++ & 3] = v;
    }
  };
  auto q_front = [&]() -> int {
    if constexpr (PHASE == 1) return q0;
    else return qarr[qh & 3];
  };
  auto q_pop = [&]() {
    if constexpr (PHASE == 1) {
      q0 = q1;
      q1 = q2;
      --qn;
    } else {
      ++qh;
    }
  };
  int ld_id = fetch();
  q_push(ld_id);
  Item ld_it = decode_item<PHASE>(p, ld_id, n_act, tiles_s, tiles_r);
  int ld_c = 0, ld_seq = 0;
  auto issue_next = [&]() {
    if (ld_it.id < 0) return;
    issue_chunk<PHASE>(ld_it, ld_c, my_stage + (ld_seq % NS) * STAGE, &my_bar[ld_seq % NS], lane,
                       ld_it.shared ? &map_s0 : &map_r0, ld_it.shared ? &map_s1 : &map_r1);
    ++ld_seq;
    if (++ld_c == ld_it.nch) {
      ld_id = fetch();
      q_push(ld_id);
      ld_it = decode_item<PHASE>(p, ld_id, n_act, tiles_s, tiles_r);
      ld_c = 0;
    }
  };
  for (int i = 0; i < NS; ++i) issue_next();

  // ---- phase 1: the activation package arrives in shared memory by one bulk copy
  const int d = p.d;
  const int nbx = d / 256;
  unsigned char* xB = xprep + PL.xB;                                   // [T][xstride]
  unsigned char* XBm = xprep + PL.XBm;                                 // [T][nbx][4][3][4] bf16
  // the 32-value sums (read only by the shared expert's items) stay in global memory, so that
  // the package in shared memory leaves room for one more ring at T = 8
  const float* X32 = reinterpret_cast<const float*>(p.pkg + PL.X32);  // [T][d/32]
  if (PHASE == 1) {
    if (!mbar_wait_bounded(pkg_bar, 0, WAIT_LIMIT)) {
      if (lane == 0) set_err(p.err, BRE_DEVERR_TIMEOUT);
      for (int q = 0; q < ld_seq; ++q) mbar_wait_bounded(&my_bar[q % NS], (q / NS) & 1, WAIT_LIMIT);
      return;
    }
  }

  int cs_seq = 0;
  const int Fnb = p.F / 256;
  while (true) {
    const int id = q_front();
    if (id < 0) break;
    const Item it = decode_item<PHASE>(p, id, n_act, tiles_s, tiles_r);
    const int r0 = it.tile * 16;
    // column -> token (phase 1) or h row (phase 2)
    auto col_src = [&](int col) -> int {
      if (col >= it.n) return -1;
      if (it.shared) return col;                                  // token; phase-2 h row of the shared expert
      const int pos = it.off + col;
      return (PHASE == 1) ? fdiv(__ldg(p.perm + pos), p.fd_k) : pos;
    };
    const int sg = col_src(g), sc0 = col_src(2 * t), sc1 = col_src(2 * t + 1);
    // data sources: an absent column (>= n) reads column 0's data (or row 0), whose products
    // land only in that column's outputs, which are never stored; this keeps the inner loops
    // free of presence tests
    const int src0 = it.n > 0 ? col_src(0) : 0;
    const int dg = sg >= 0 ? sg : src0, d0 = sc0 >= 0 ? sc0 : src0, d1 = sc1 >= 0 ? sc1 : src0;
    float acc2[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc2[m][i] = 0.0f;

    for (int cc = 0; cc < it.nch; ++cc) {
      const int st = cs_seq % NS;
      if (!mbar_wait_bounded(&my_bar[st], (cs_seq / NS) & 1, WAIT_LIMIT)) {
        if (lane == 0) set_err(p.err, BRE_DEVERR_TIMEOUT);
        for (int q = cs_seq + 1; q < ld_seq; ++q) mbar_wait_bounded(&my_bar[q % NS], (q / NS) & 1, WAIT_LIMIT);
        return;
      }
      const unsigned char* stage = my_stage + st * STAGE;
      if (PHASE == 1) {
        const int m = cc >= it.cpi ? 1 : 0;
        const int c = it.kp * it.cpi + (cc - m * it.cpi);
        // one call site per format (the matrix's accumulator is selected into accm), so that
        // the hot loop's code stays small
        float accm[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) accm[i] = m ? acc2[1][i] : acc2[0][i];
        if (it.shared) {
          const uint16_t* xr = p.x + (size_t)dg * d;
          const float* x0 = X32 + d0 * (d / 32);
          const float* x1 = X32 + d1 * (d / 32);
          p1_q80_mat(stage, it.cb, c, g, t, xr, x0, x1, p.kc.k43, accm);
        } else {
          const unsigned char* xb = xB + (size_t)dg * p.xstride;
          const unsigned char* xm = XBm + (size_t)dg * nbx * 96;
          if (it.cb == 4)
            p1_q2k_mat<4>(stage, 4, c, g, t, xb, xm, rc, p.kc, accm);
          else
            p1_q2k_mat<0>(stage, it.cb, c, g, t, xb, xm, rc, p.kc, accm);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc2[0][i] = m ? acc2[0][i] : accm[i];
          acc2[1][i] = m ? accm[i] : acc2[1][i];
        }
      } else {
        const int c = it.kp * it.cpi + cc;
        if (it.shared) {
          p2_q80_chunk(stage, it.cb, c, g, t, p.Fs, p.hS + (size_t)dg * 2 * p.Fs, p.HS16 + (size_t)d0 * (p.Fs / 16),
                       p.HS16 + (size_t)d1 * (p.Fs / 16), p.kc.k43, acc2[0]);
        } else {
          p2_q2k_chunk(stage, it.cb, c, Fnb, g, t, dg, p.hB, p.HBm, rc, p.kc, acc2[0]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      ++cs_seq;
      issue_next();
    }
    q_pop();

    // ---- phase 1 ends an item by storing its FP32 (gate, up) partial sums for the expert's real
    // columns; ffn_finish_kernel adds the K parts in order and forms h.  Phase 2 stores y.
    if (PHASE == 1) {
      float* base = it.shared ? p.part_s + (size_t)it.tile * it.KP * 32 : p.part_r + (size_t)it.tile * it.KP * 32;
      const size_t col_stride = (size_t)(it.shared ? tiles_s : tiles_r) * it.KP * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int col = 2 * t + (i & 1), row = g + 8 * (i >> 1);
        if (col < it.n) {
          const size_t src = it.shared ? (size_t)col : (size_t)(it.off + col);   // token / pair position
          *reinterpret_cast<float2*>(base + src * col_stride + (it.kp * 16 + row) * 2) =
              make_float2(acc2[0][i], acc2[1][i]);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int cs = (i & 1) ? sc1 : sc0;
        if (cs >= 0) {
          const int row = r0 + g + 8 * (i >> 1);
          if (it.shared)
            p.y_shared[(size_t)cs * p.d + row] = acc2[0][i];
          else
            p.y_pairs[(size_t)cs * p.d + row] = acc2[0][i];
        }
      }
    }
  }
}

// ----------------------------------------------------------------------------
// finish: for every (pair or token, row) add the K-part partial sums of gate and up in order
// 0..KP-1, form h = silu(gate) * up and store it in the layouts phase 2 reads (routed: BF16 of
// h * 4^-min(s,2) in the (lane-rotated) fragment order plus three limbs of each 16-row sum of
// the BF16 h; shared: two limbs in natural order plus FP32 16-row sums).  One warp per 32 rows
// of one pair/token.
// ----------------------------------------------------------------------------
struct FinishParams {
  const float* part_r;
  const float* part_s;
  int kp_r, kp_s;
  int F, Fs, P, T, E;
  const int32_t* offsets;
  uint16_t* hB;
  uint16_t* HBm;
  uint16_t* hS;
  float* HS16;
};

__global__ void __launch_bounds__(256) ffn_finish_kernel(const FinishParams f) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int gr = f.F / 32, gs = f.Fs / 32;
  const long long nr = (long long)f.P * gr;
  const bool shared = w >= nr;
  int src, rg;
  if (!shared) {
    src = (int)(w / gr);
    rg = (int)(w % gr);
    if (src >= __ldg(f.offsets + f.E)) return;   // no pair there (fewer valid pairs than T * k)
  } else {
    const long long w2 = w - nr;
    if (w2 >= (long long)f.T * gs) return;
    src = (int)(w2 / gs);
    rg = (int)(w2 % gs);
  }
  const int rows = shared ? f.Fs : f.F;
  const int KP = shared ? f.kp_s : f.kp_r;
  const int row = rg * 32 + lane, tile = row >> 4, r = row & 15;
  const float* pc = (shared ? f.part_s : f.part_r) + ((size_t)src * (rows / 16) + tile) * KP * 32 + r * 2;
  // every part's load is issued before the sum (up to four at once)
  float gv = 0.0f, uv = 0.0f;
  for (int q0 = 0; q0 < KP; q0 += 4) {
    float2 v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      v[q] = (q0 + q < KP) ? *reinterpret_cast<const float2*>(pc + (q0 + q) * 32) : make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q0 + q < KP) {
        gv = (q0 + q == 0) ? v[q].x : gv + v[q].x;
        uv = (q0 + q == 0) ? v[q].y : uv + v[q].y;
      }
    }
  }
  const float h = silu_mul(gv, uv);
  uint32_t hi, lo;
  split_bf16x2(h, hi, lo);
  float hq = bf16_bits_to_f32(hi) + bf16_bits_to_f32(lo);
  const int Fnb = f.F / 256;
  if (shared) {
    f.hS[((size_t)src * 2 + 0) * f.Fs + row] = (uint16_t)hi;
    f.hS[((size_t)src * 2 + 1) * f.Fs + row] = (uint16_t)lo;
  } else {
    const int b2 = row >> 8, j = (row >> 4) & 15, ip = row & 15;
    const int byte = ip >> 2, s = ip & 3, v4 = (byte & 1) * 2 + (byte >> 1);
    const int tq = j >> 2, jj = ((j & 3) - tq) & 3;   // fragment step of sub-block j (rot_sub)
    // BF16 of h * 4^-min(s,2) (the down projection's A fragments keep codes in place); a power
    // of two commutes with the rounding, so the 16-row sums below use h rounded to BF16
    const float hs = __fmul_rn(h, s == 0 ? 1.0f : (s == 1 ? 0.25f : 0.0625f));
    const size_t idx = (((((size_t)src * Fnb + b2) * 4 + jj) * 2 + (s >> 1)) * 4 + tq) * 8 + (s & 1) * 4 + v4;
    f.hB[idx] = (uint16_t)f32_to_bf16_rne(hs);
    hq = bf16_bits_to_f32(f32_to_bf16_rne(h));
  }
  // 16-row sums of the limb values (half warps)
#pragma unroll
  for (int o = 1; o <= 8; o <<= 1) hq += __shfl_xor_sync(0xffffffffu, hq, o);
  if ((lane & 15) == 0) {
    if (shared) {
      f.HS16[(size_t)src * (f.Fs / 16) + tile] = hq;
    } else {
      const int b2 = tile >> 4, j = tile & 15;
      const uint32_t h1 = f32_to_bf16_rne(hq);
      const float r1 = hq - bf16_bits_to_f32(h1);
      const uint32_t h2 = f32_to_bf16_rne(r1);
      const uint32_t h3 = f32_to_bf16_rne(r1 - bf16_bits_to_f32(h2));
      uint16_t* dst = f.HBm + (((size_t)src * Fnb + b2) * 4 + (j >> 2)) * 12 + (j & 3);
      dst[0] = (uint16_t)h1;
      dst[4] = (uint16_t)h2;
      dst[8] = (uint16_t)h3;
    }
  }
}

int pick_chunk(int nb, int bb, int cap_per_mat, int align_blocks, int* whole) {
  if (16 * nb * bb <= cap_per_mat) {
    *whole = 1;
    return nb;
  }
  *whole = 0;
  int cb = cap_per_mat / (16 * bb);
  cb -= cb % align_blocks;
  while (cb > 0 && nb % cb) cb -= align_blocks;
  return cb;
}

// K parts per tile of a phase whose rows hold nb_r Q2_K / nb_s Q8_0 blocks: routed tiles split
// into one item per chunk; shared (Q8_0) tiles into at most 4 parts (a divisor of their chunk
// count).
void phase_kparts(int nb_r, int nb_s, bool has_shared, int* kpr, int* kps) {
  int whole = 0;
  const int cbr = pick_chunk(nb_r, Q2K_BB, STAGE, 4, &whole);
  *kpr = cbr > 0 ? nb_r / cbr : 1;
  *kps = 1;
  if (has_shared) {
    const int cbs = pick_chunk(nb_s, Q80_BB, STAGE, 8, &whole);
    const int Cs = cbs > 0 ? nb_s / cbs : 1;
    for (int q = Cs < 4 ? Cs : 4; q >= 1; --q)
      if (Cs % q == 0) {
        *kps = q;
        break;
      }
  }
}

}  // namespace

// 1 KB of work counters, then one K-part counter per tile of the largest decode batch (shared
// tiles + DECODE_T_MAX * k routed pairs' tiles, the larger of the two phases).
size_t ffn_reserved_bytes(int k, int d, int F, int Fs) {
  const size_t s1 = (size_t)Fs / 16 + (size_t)DECODE_T_MAX * k * (F / 16);
  const size_t s2 = (Fs > 0 ? (size_t)d / 16 : 0) + (size_t)DECODE_T_MAX * k * (d / 16);
  const size_t slots = s1 > s2 ? s1 : s2;
  return 1024 + ((slots * 4 + 255) & ~(size_t)255);
}

namespace {

// Workspace of the decode path, in order.
struct DecWs {
  size_t pkg, hB, HBm, hS, HS16, cnt, part_r, part_s, total;
};

DecWs dec_ws_layout(int T, int k, int d, int F, int Fs) {
  const size_t P = (size_t)T * k;
  int kpr1 = 1, kps1 = 1;
  phase_kparts(d / 256, d / 32, Fs > 0, &kpr1, &kps1);
  // partials: phase 1's (gate, up) pairs over d_ff rows (phase 2 adds its K halves into the
  // outputs themselves)
  const size_t pr = P * (F / 16) * kpr1 * 16 * 2 * 4;
  const size_t ps = (size_t)T * (Fs / 16) * kps1 * 16 * 2 * 4;
  auto up256 = [](size_t v) { return (v + 255) & ~(size_t)255; };
  DecWs w;
  w.cnt = 1024;                                                  // after the work counters
  w.pkg = ffn_reserved_bytes(k, d, F, Fs);
  w.hB = up256(w.pkg + pkg_layout(T, d).total);
  w.HBm = up256(w.hB + P * (F / 256) * 256 * 2);
  w.hS = up256(w.HBm + P * (F / 256) * 4 * 12 * 2);
  w.HS16 = up256(w.hS + (size_t)T * 2 * Fs * 2);
  w.part_r = up256(w.HS16 + (size_t)T * (Fs / 16) * 4);
  w.part_s = up256(w.part_r + pr);
  w.total = up256(w.part_s + (Fs > 0 ? ps : 0));
  return w;
}

}  // namespace

size_t ffn_ws_bytes(int T, int k, int E, int d, int F, int Fs) {
  (void)E;
  // monotone in T: a workspace sized for T also serves every smaller batch (either path)
  if (T > DECODE_T_MAX)
    return std::max(ffn_gemm_ws_bytes(T, k, d, F, Fs), dec_ws_layout(DECODE_T_MAX, k, d, F, Fs).total);
  return dec_ws_layout(T, k, d, F, Fs).total;
}

bre_status ffn_check_shapes(const bre_ffn_weights* r, const bre_ffn_weights* sh, int T) {
  const int d = r->d, F = r->d_ff;
  if (d <= 0 || F <= 0 || d % 256 || F % 256) return BRE_ERR_UNSUPPORTED;
  if (sh && (sh->d != d || sh->d_ff <= 0 || sh->d_ff % 256)) return BRE_ERR_UNSUPPORTED;
  if (T <= DECODE_T_MAX) {
    // Q2_K rows go to shared memory as whole 16-row tiles when a tile fits a stage (rows of at
    // most 4 blocks), otherwise as tensor copies of 4-block (336-byte) pieces, which needs rows
    // a multiple of 4 blocks long (16-byte row pitch)
    if (!(d <= 1024 || d % 1024 == 0)) return BRE_ERR_UNSUPPORTED;
    if (!(F <= 1024 || F % 1024 == 0)) return BRE_ERR_UNSUPPORTED;
  }
  return BRE_OK;
}

// Tensor map over quantised expert matrices viewed as 32-bit words, [experts][rows][row words],
// box = (chunk words, 16 rows, 1 expert).  Encodings are cached: decode calls repeat the same
// few maps, and an encode costs host time on every call.
static bool weight_map(CUtensorMap* m, const void* base, int n_exp, long long exp_stride, int rows, int row_bytes,
                       int chunk_bytes) {
  struct Entry {
    const void* base;
    long long n_exp, exp_stride, rows, row_bytes, chunk_bytes;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n_cached = 0, next = 0;
  if (n_exp <= 1 || exp_stride <= 0) exp_stride = (long long)rows * row_bytes;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cached; ++i) {
    const Entry& c = cache[i];
    if (c.base == base && c.n_exp == n_exp && c.exp_stride == exp_stride && c.rows == rows &&
        c.row_bytes == row_bytes && c.chunk_bytes == chunk_bytes) {
      *m = c.map;
      return true;
    }
  }
  const uint64_t dims[3] = {(uint64_t)(row_bytes / 4), (uint64_t)rows, (uint64_t)(n_exp > 0 ? n_exp : 1)};
  const uint64_t strides[2] = {(uint64_t)row_bytes, (uint64_t)exp_stride};
  const uint32_t box[3] = {(uint32_t)(chunk_bytes / 4), 16u, 1u};
  if (row_bytes % 16 || chunk_bytes % 16 || exp_stride % 16) return false;
  if (!encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return false;
  Entry& slot = cache[next];
  slot = Entry{base, n_exp, exp_stride, rows, row_bytes, chunk_bytes, *m};
  next = (next + 1) % 32;
  if (n_cached < 32) ++n_cached;
  return true;
}

static cudaError_t launch_decode(const FfnArgs& a, cudaStream_t s) {
  const bre_ffn_weights* R = a.routed;
  const bre_ffn_weights* S = a.shared;
  DecParams p{};
  p.d = R->d;
  p.F = R->d_ff;
  p.Fs = S ? S->d_ff : 0;
  p.T = a.T;
  p.k = a.k;
  p.E = R->n_experts;
  p.has_shared = S ? 1 : 0;
  p.x = a.x;
  p.offsets = a.offsets;
  p.perm = a.perm;
  p.active = a.active;
  p.n_active = a.n_active;
  p.y_pairs = a.y_pairs;
  p.y_shared = a.y_shared;
  p.err = a.err;
  char* w = reinterpret_cast<char*>(a.ws);
  const DecWs L = dec_ws_layout(a.T, a.k, p.d, p.F, p.Fs);
  p.counters = reinterpret_cast<int*>(w);
  p.pkg = reinterpret_cast<const unsigned char*>(w + L.pkg);
  unsigned char* pkg_w = reinterpret_cast<unsigned char*>(w + L.pkg);
  p.hB = reinterpret_cast<uint16_t*>(w + L.hB);
  p.HBm = reinterpret_cast<uint16_t*>(w + L.HBm);
  p.hS = reinterpret_cast<uint16_t*>(w + L.hS);
  p.HS16 = reinterpret_cast<float*>(w + L.HS16);
  p.tile_cnt = reinterpret_cast<int*>(w + L.cnt);
  p.part_r = reinterpret_cast<float*>(w + L.part_r);
  p.part_s = reinterpret_cast<float*>(w + L.part_s);
  p.xstride = x_stride(p.d);
  p.kc = DecConst{0x43004300u, 0x43434343u, 0xC300C300u};

  const int sms = device_sm_count();
  const int smem_max = device_max_smem_optin();
  const dim3 prep_grid(p.d / 256, a.T);
  {
    const cudaError_t le = launch_k(ffn_prep_kernel, dim3(prep_grid), dim3(256), 0, s, a.x, a.T, p.d, pkg_w);
    if (le != cudaSuccess) return le;
  }
  {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  for (int phase = 1; phase <= 2; ++phase) {
    if (phase == 1) {
      p.rw0 = static_cast<const uint8_t*>(R->gate);
      p.rw1 = static_cast<const uint8_t*>(R->up);
      p.rs0 = R->expert_stride_gate;
      p.rs1 = R->expert_stride_up;
      p.sw0 = S ? static_cast<const uint8_t*>(S->gate) : nullptr;
      p.sw1 = S ? static_cast<const uint8_t*>(S->up) : nullptr;
      p.rows_r = p.F;
      p.rows_s = p.Fs;
      p.nb_r = p.d / 256;
      p.nb_s = p.d / 32;
    } else {
      p.rw0 = static_cast<const uint8_t*>(R->down);
      p.rw1 = nullptr;
      p.rs0 = R->expert_stride_down;
      p.rs1 = 0;
      p.sw0 = S ? static_cast<const uint8_t*>(S->down) : nullptr;
      p.sw1 = nullptr;
      p.rows_r = p.d;
      p.rows_s = p.d;
      p.nb_r = p.F / 256;
      p.nb_s = p.Fs / 32;
    }
    p.cb_r = pick_chunk(p.nb_r, Q2K_BB, STAGE, 4, &p.whole_r);
    p.cb_s = S ? pick_chunk(p.nb_s, Q80_BB, STAGE, 8, &p.whole_s) : 1;
    if (p.cb_r <= 0 || p.cb_s <= 0) return cudaErrorInvalidValue;
    p.C_r = p.nb_r / p.cb_r;
    p.C_s = S ? p.nb_s / p.cb_s : 1;
    // phase 1 splits tiles along K into parts the finish kernel sums (whole-tile items, two
    // per warp, left SMs idle); phase 2 is not split (its halves would add into the outputs,
    // and the per-item work that costs was measured to outweigh the shorter last wave)
    if (phase == 1) {
      phase_kparts(p.nb_r, p.nb_s, S != nullptr, &p.kp_r, &p.kp_s);
    } else {
      p.kp_r = 1;
      p.kp_s = 1;
    }
    {
      const int kpr = p.kp_r, kps = p.kp_s;
      p.fd_kpr = make_fdiv(kpr);
      p.fd_kps = make_fdiv(kps);
      p.fd_trk = make_fdiv((unsigned)(p.rows_r / 16 * kpr));
      p.fd_k = make_fdiv((unsigned)a.k);
      p.cpi_r = p.C_r / kpr;
      p.cpi_s = p.C_s / kps;
      if (p.cpi_r * kpr != p.C_r || p.cpi_s * kps != p.C_s) return cudaErrorInvalidValue;
    }
    // tensor maps for chunked rows (unused when whole tiles fit a stage)
    CUtensorMap mr0{}, mr1{}, ms0{}, ms1{};
    if (!p.whole_r) {
      if (!weight_map(&mr0, p.rw0, R->n_experts, p.rs0, p.rows_r, p.nb_r * Q2K_BB, p.cb_r * Q2K_BB)) return cudaErrorInvalidValue;
      if (phase == 1 &&
          !weight_map(&mr1, p.rw1, R->n_experts, p.rs1, p.rows_r, p.nb_r * Q2K_BB, p.cb_r * Q2K_BB))
        return cudaErrorInvalidValue;
    }
    if (S && !p.whole_s) {
      if (!weight_map(&ms0, p.sw0, 1, 0, p.rows_s, p.nb_s * Q80_BB, p.cb_s * Q80_BB)) return cudaErrorInvalidValue;
      if (phase == 1 && !weight_map(&ms1, p.sw1, 1, 0, p.rows_s, p.nb_s * Q80_BB, p.cb_s * Q80_BB))
        return cudaErrorInvalidValue;
    }
    const size_t xbytes = (phase == 1) ? (size_t)pkg_layout(a.T, p.d).X32 : 0;   // shared-memory part
    int nw = (phase == 1) ? MAX_WARPS : MAX_WARPS_P2;
    while (nw > 1 && (size_t)nw * NS * STAGE + BAR_BYTES + xbytes > (size_t)smem_max) --nw;
    const size_t smem = (size_t)nw * NS * STAGE + BAR_BYTES + xbytes;
    if (smem > (size_t)smem_max) return cudaErrorInvalidValue;
    cudaError_t e;
    if (phase == 1) {
      e = cudaFuncSetAttribute(ffn_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      {
        const cudaError_t le = launch_k(ffn_decode_kernel<1>, dim3(sms), dim3(nw * 32), smem, s, p, mr0, mr1, ms0,
                                        ms1);
        if (le != cudaSuccess) return le;
      }
      FinishParams fp;
      fp.part_r = p.part_r;
      fp.part_s = p.part_s;
      fp.kp_r = p.kp_r;
      fp.kp_s = p.kp_s;
      fp.F = p.F;
      fp.Fs = p.Fs;
      fp.P = (int)((size_t)a.T * a.k);
      fp.T = a.T;
      fp.E = p.E;
      fp.offsets = a.offsets;
      fp.hB = p.hB;
      fp.HBm = p.HBm;
      fp.hS = p.hS;
      fp.HS16 = p.HS16;
      const long long warps = (long long)fp.P * (p.F / 32) + (S ? (long long)a.T * (p.Fs / 32) : 0);
      const cudaError_t le = launch_k(ffn_finish_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, fp);
      if (le != cudaSuccess) return le;
    } else {
      e = cudaFuncSetAttribute(ffn_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      {
        const cudaError_t le = launch_k(ffn_decode_kernel<2>, dim3(sms), dim3(nw * 32), smem, s, p, mr0, mr1, ms0,
                                        ms1);
        if (le != cudaSuccess) return le;
      }
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_ffn(const FfnArgs& a, cudaStream_t s) {
  if (a.T <= DECODE_T_MAX) return launch_decode(a, s);
  return launch_gemm(a, s);
}

}  // namespace bre
