// Expert FFN for decode-sized batches (at most 8 tokens per expert).
//
// Strata-DSV4.1 README, V4-Flash "How it works" (experts, then the finish step:
// shared expert + routed sum) and "Verifying it" (the expert tier is checked
// against a dequantised F32 reference); SwiGLU from the V4-Flash description.
//
// Design (GB300): the path is bound by streaming 2-bit weights from HBM, so every
// byte is read once.  Each warp owns a two-stage ring in shared memory that
// bulk-copy (TMA) engines fill with 16-row tiles of an expert matrix; the warp
// dequantises in registers straight into mma.sync A fragments and multiplies by
// the expert's tokens (N = 8 columns).  Work items (expert, 16-row tile) are
// handed out by an atomic counter so that busy SMs take fewer items.
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
#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

namespace {

constexpr int NS = 2;                 // ring stages per warp
constexpr int STAGE = 10752;          // bytes per stage (2 x 16 rows x 336 B)
constexpr int MAX_WARPS = 8;
constexpr uint32_t C43 = 0x43434343u;
constexpr uint32_t SEL_LO = 0x4140u;  // bytes 0,1 -> (128+b0, 128+b1) as bf16x2
constexpr uint32_t SEL_HI = 0x4342u;  // bytes 2,3
constexpr long long WAIT_LIMIT = 2000000000LL;  // cycles (~1 s) before a wait gives up
constexpr int BAR_BYTES = 256;                  // mbarrier region: MAX_WARPS * NS ring barriers + package

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
  uint16_t* hB;   // routed h, permuted, 2 limbs: [P][F/256][4][4][4][2][4]
  uint16_t* HBm;  // routed sub-block sums of h, 3 limbs: [P][F/256][4][3][4]
  uint16_t* hS;   // shared h, natural, 2 limbs: [T][2][Fs]
  float* HS16;    // shared 16-row sums of h: [T][Fs/16]
  float* y_pairs;
  float* y_shared;
  int* counters;
  int32_t* err;
  int xstride;  // bytes per token row of the permuted activations in shared memory
  const unsigned char* pkg;  // activation package in global memory (phase 1)
};

struct Item {
  int id;       // -1: none
  bool shared;
  int e, off, n;
  int tile;
  int nb, cb, C, whole, bb;
  const uint8_t* src0;
  const uint8_t* src1;
};

template <int PHASE>
__device__ __forceinline__ Item decode_item(const DecParams& p, int id, int n_act, int tiles_s, int tiles_r) {
  Item it;
  it.id = id;
  if (id < 0) return it;
  if (id < tiles_s) {
    it.shared = true;
    it.tile = id;
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
    const int r = id - tiles_s;
    const int a = r / tiles_r;
    it.shared = false;
    it.tile = r % tiles_r;
    it.e = __ldg(p.active + a);
    it.off = __ldg(p.offsets + it.e);
    it.n = __ldg(p.offsets + it.e + 1) - it.off;
    it.nb = p.nb_r;
    it.cb = p.cb_r;
    it.whole = p.whole_r;
    it.bb = Q2K_BB;
    it.src0 = p.rw0 + (long long)it.e * p.rs0;
    it.src1 = (PHASE == 1) ? p.rw1 + (long long)it.e * p.rs1 : nullptr;
  }
  it.C = it.nb / it.cb;
  return it;
}

// Issue the bulk copies of chunk c of `it` into `stage` (warp-wide; lane 0 arms the barrier).
template <int PHASE>
__device__ __forceinline__ void issue_chunk(const Item& it, int c, unsigned char* stage, uint64_t* bar, int lane) {
  constexpr int NMAT = (PHASE == 1) ? 2 : 1;
  const int row_bytes = it.nb * it.bb;
  const int chunk_bytes = it.cb * it.bb;
  const uint32_t mat_bytes = 16u * chunk_bytes;
  if (lane == 0) mbar_arrive_expect_tx(bar, NMAT * mat_bytes);
  __syncwarp();
  if (it.whole) {
    if (lane < NMAT) {
      const uint8_t* src = (lane == 0 ? it.src0 : it.src1) + (long long)it.tile * 16 * row_bytes;
      bulk_g2s(stage + lane * mat_bytes, src, mat_bytes, bar);
    }
  } else {
    if (lane < 16 * NMAT) {
      const int m = lane >> 4, r = lane & 15;
      const uint8_t* src = (m == 0 ? it.src0 : it.src1) + (long long)(it.tile * 16 + r) * row_bytes +
                           (long long)c * chunk_bytes;
      bulk_g2s(stage + m * mat_bytes + r * chunk_bytes, src, chunk_bytes, bar);
    }
  }
}

__device__ __forceinline__ uint32_t lds_u32(const unsigned char* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint32_t lds_u16(const unsigned char* p) {
  return *reinterpret_cast<const unsigned short*>(p);
}
__device__ __forceinline__ uint32_t lds_u32_a2(const unsigned char* p) {  // 2-byte aligned
  return lds_u16(p) | (lds_u16(p + 2) << 16);
}

// Q2_K A fragment of one row for step s: 4 codes x sc as (128 + sc*q) bf16 pairs.
__device__ __forceinline__ void q2k_frag(uint32_t qw, uint32_t sc, int s, uint32_t& lo, uint32_t& hi) {
  const uint32_t v = ((qw >> (2 * s)) & 0x03030303u) * sc;
  lo = prmt(v, C43, SEL_LO);
  hi = prmt(v, C43, SEL_HI);
}

// Q2_K A fragments of one row for step s, codes left in place: one LOP3 per register gives the
// BF16 pair 128 + c * 4^e (e = min(s, 2); the code occupies mantissa bits 2e, 2e+1).  lo holds
// codes (s, 8+s) of the sub-block word (bytes 0 and 2), hi codes (4+s, 12+s) (bytes 1 and 3).
__device__ __forceinline__ void q2k_pairs(uint32_t w, int s, uint32_t& lo, uint32_t& hi) {
  constexpr uint32_t M43 = 0x43004300u;
  if (s < 3) {
    const uint32_t m = 0x00030003u << (2 * s);
    lo = (w & m) | M43;
    hi = ((w >> 8) & m) | M43;
  } else {
    const uint32_t m = 0x00030003u << 4;
    lo = ((w >> 2) & m) | M43;
    hi = ((w >> 10) & m) | M43;
  }
}

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// (sc, sc) and (-128 sc, -128 sc) as BF16 pairs for sub-block byte jj of a scales word (exact).
__device__ __forceinline__ void q2k_scale_pairs(uint32_t sclo, int jj, uint32_t& sc2, uint32_t& nsc2) {
  const uint32_t u = prmt(sclo, C43, (uint32_t)(jj | (4 << 4) | (jj << 8) | (4 << 12)));   // 128 + sc
  sc2 = bf16x2_fma(u, 0x3F803F80u, 0xC300C300u);                                          // u - 128
  nsc2 = bf16x2_fma(u, 0xC300C300u, 0x46804680u);                                         // 16384 - 128 u
}

// Q8_0 nibble planes of one row word (4 consecutive int8): (128+lo) and (128+hi') pairs.
__device__ __forceinline__ void q80_frag(uint32_t w, uint32_t& lo01, uint32_t& lo23, uint32_t& hi01,
                                         uint32_t& hi23) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = ((w >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;
  lo01 = prmt(lo, C43, SEL_LO);
  lo23 = prmt(lo, C43, SEL_HI);
  hi01 = prmt(hi, C43, SEL_LO);
  hi23 = prmt(hi, C43, SEL_HI);
}

// ----------------------------------------------------------------------------
// phase 1, routed Q2_K: gate and up of 16 rows over one chunk
// ----------------------------------------------------------------------------
__device__ __forceinline__ void p1_q2k_chunk(const unsigned char* stage, int cb, int c, int g, int t,
                                             const unsigned char* xb_g,    // permuted x of column g (or null)
                                             const unsigned char* xbm_g,   // XBm of column g (or null)
                                             const float* xbM0, const float* xbM1,  // XbM rows of columns 2t, 2t+1
                                             float (&acc)[2][4]) {
  const int chunk_bytes = cb * Q2K_BB;
  const int mat_bytes = 16 * chunk_bytes;
  for (int bl = 0; bl < cb; ++bl) {
    const int b = c * cb + bl;
    uint32_t qw[2][2][4], sw[2][2], dd[2][2];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const unsigned char* base = stage + m * mat_bytes + (g + 8 * rr) * chunk_bytes + bl * Q2K_BB;
        sw[m][rr] = lds_u32(base + 4 * t);
        dd[m][rr] = lds_u32(base + 80);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) qw[m][rr][jj] = lds_u32(base + 16 + 16 * t + 4 * jj);
      }
    // one accumulator per (matrix, jj): four independent MMA chains per matrix
    float P[2][4][4], M[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) P[m][jj][i] = 0.0f;
        M[m][i] = 0.0f;
      }
    const unsigned char* xblk = xb_g ? xb_g + b * 512 : nullptr;
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint32_t sc2[2][2], nsc2[2][2];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) q2k_scale_pairs(sw[m][rr] & 0x0F0F0F0Fu, jj, sc2[m][rr], nsc2[m][rr]);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        uint2 bv = make_uint2(0u, 0u);
        if (xblk) bv = *reinterpret_cast<const uint2*>(xblk + ((jj * 4 + s) * 4 + t) * 8);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          uint32_t a0, a1, a2, a3;
          q2k_pairs(qw[m][0][jj], s, a0, a2);
          q2k_pairs(qw[m][1][jj], s, a1, a3);
          a0 = bf16x2_fma(a0, sc2[m][0], nsc2[m][0]);
          a2 = bf16x2_fma(a2, sc2[m][0], nsc2[m][0]);
          a1 = bf16x2_fma(a1, sc2[m][1], nsc2[m][1]);
          a3 = bf16x2_fma(a3, sc2[m][1], nsc2[m][1]);
          mma_bf16_16816(P[m][jj], a0, a1, a2, a3, bv.x, bv.y);
        }
      }
    }
    // min term: M' = sum_j (128 + m_j) X_j over the 16 sub-blocks, X_j in three limbs
#pragma unroll
    for (int limb = 0; limb < 3; ++limb) {
      uint2 bm = make_uint2(0u, 0u);
      if (xbm_g) bm = *reinterpret_cast<const uint2*>(xbm_g + ((b * 4 + t) * 3 + limb) * 8);
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        const uint32_t mg = (sw[m][0] >> 4) & 0x0F0F0F0Fu;
        const uint32_t mg8 = (sw[m][1] >> 4) & 0x0F0F0F0Fu;
        mma_bf16_16816(M[m], prmt(mg, C43, SEL_LO), prmt(mg8, C43, SEL_LO), prmt(mg, C43, SEL_HI),
                       prmt(mg8, C43, SEL_HI), bm.x, bm.y);
      }
    }
    const float x0 = xbM0 ? xbM0[b] : 0.0f, x1 = xbM1 ? xbM1[b] : 0.0f;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t ddv = dd[m][i >> 1];
        const float dv = f16_bits_to_f32(ddv & 0xFFFFu), dmv = f16_bits_to_f32(ddv >> 16);
        const float xs = (i & 1) ? x1 : x0;
        const float psum = (P[m][0][i] + P[m][1][i]) + (P[m][2][i] + P[m][3][i]);
        const float mv = fmaf(-128.0f, xs, M[m][i]);
        acc[m][i] = fmaf(dv, psum, fmaf(-dmv, mv, acc[m][i]));
      }
  }
}

// ----------------------------------------------------------------------------
// phase 1, shared Q8_0: gate and up of 16 rows over one chunk (natural k order)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void p1_q80_chunk(const unsigned char* stage, int cb, int c, int g, int t,
                                             const uint16_t* xrow_g,  // global x row of column g (or null)
                                             const float* x32_0, const float* x32_1, float (&acc)[2][4]) {
  const int chunk_bytes = cb * Q80_BB;
  const int mat_bytes = 16 * chunk_bytes;
  for (int bl = 0; bl < cb; ++bl) {
    const int bq = c * cb + bl;
    float Ph[2][4], Pl[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        Ph[m][i] = 0.0f;
        Pl[m][i] = 0.0f;
      }
    uint32_t dd[2][2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint2 bv = make_uint2(0u, 0u);
      if (xrow_g) bv = __ldg(reinterpret_cast<const uint2*>(xrow_g + 32 * bq + 16 * hf + 4 * t));
#pragma unroll
      for (int m = 0; m < 2; ++m) {
        uint32_t l01[2], l23[2], h01[2], h23[2];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const unsigned char* base = stage + m * mat_bytes + (g + 8 * rr) * chunk_bytes + bl * Q80_BB;
          if (hf == 0) dd[m][rr] = lds_u16(base);
          q80_frag(lds_u32_a2(base + 2 + 16 * hf + 4 * t), l01[rr], l23[rr], h01[rr], h23[rr]);
        }
        mma_bf16_16816(Pl[m], l01[0], l01[1], l23[0], l23[1], bv.x, bv.y);
        mma_bf16_16816(Ph[m], h01[0], h01[1], h23[0], h23[1], bv.x, bv.y);
      }
    }
    const float x0 = x32_0 ? x32_0[bq] : 0.0f, x1 = x32_1 ? x32_1[bq] : 0.0f;
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float dv = f16_bits_to_f32(dd[m][i >> 1]);
        const float xs = (i & 1) ? x1 : x0;
        const float v = fmaf(-2304.0f, xs, fmaf(16.0f, Ph[m][i], Pl[m][i]));
        acc[m][i] = fmaf(dv, v, acc[m][i]);
      }
  }
}

// ----------------------------------------------------------------------------
// phase 2, routed Q2_K down: 16 rows over one chunk; B = h limbs from global memory
// ----------------------------------------------------------------------------
__device__ __forceinline__ void p2_q2k_chunk(const unsigned char* stage, int cb, int c, int nb, int g, int t,
                                             int pos_g, const uint16_t* __restrict__ hB,
                                             const uint16_t* __restrict__ HBm, float (&acc)[4]) {
  const int chunk_bytes = cb * Q2K_BB;
  for (int bl = 0; bl < cb; ++bl) {
    const int b = c * cb + bl;
    uint32_t qw[2][4], sw[2], dd[2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const unsigned char* base = stage + (g + 8 * rr) * chunk_bytes + bl * Q2K_BB;
      sw[rr] = lds_u32(base + 4 * t);
      dd[rr] = lds_u32(base + 80);
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) qw[rr][jj] = lds_u32(base + 16 + 16 * t + 4 * jj);
    }
    float P[4][4], M[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
      for (int i = 0; i < 4; ++i) P[jj][i] = 0.0f;
    const uint16_t* hblk = (pos_g >= 0) ? hB + ((long long)pos_g * nb + b) * 512 : nullptr;
    uint4 bvs[16];
#pragma unroll
    for (int q = 0; q < 16; ++q)
      bvs[q] = hblk ? __ldg(reinterpret_cast<const uint4*>(hblk + (q * 4 + t) * 8)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      uint32_t sc2[2], nsc2[2];
      q2k_scale_pairs(sw[0] & 0x0F0F0F0Fu, jj, sc2[0], nsc2[0]);
      q2k_scale_pairs(sw[1] & 0x0F0F0F0Fu, jj, sc2[1], nsc2[1]);
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint4 bv = bvs[jj * 4 + s];
        uint32_t a0, a1, a2, a3;
        q2k_pairs(qw[0][jj], s, a0, a2);
        q2k_pairs(qw[1][jj], s, a1, a3);
        a0 = bf16x2_fma(a0, sc2[0], nsc2[0]);
        a2 = bf16x2_fma(a2, sc2[0], nsc2[0]);
        a1 = bf16x2_fma(a1, sc2[1], nsc2[1]);
        a3 = bf16x2_fma(a3, sc2[1], nsc2[1]);
        mma_bf16_16816(P[jj], a0, a1, a2, a3, bv.x, bv.y);
        mma_bf16_16816(P[jj], a0, a1, a2, a3, bv.z, bv.w);
      }
    }
    float hsum = 0.0f;
    {
      const uint32_t mg = (sw[0] >> 4) & 0x0F0F0F0Fu, mg8 = (sw[1] >> 4) & 0x0F0F0F0Fu;
      const uint32_t A0 = prmt(mg, C43, SEL_LO), A1 = prmt(mg8, C43, SEL_LO);
      const uint32_t A2 = prmt(mg, C43, SEL_HI), A3 = prmt(mg8, C43, SEL_HI);
      const uint16_t* hm = (pos_g >= 0) ? HBm + (((long long)pos_g * nb + b) * 4 + t) * 12 : nullptr;
#pragma unroll
      for (int limb = 0; limb < 3; ++limb) {
        uint2 bm = make_uint2(0u, 0u);
        if (hm) bm = __ldg(reinterpret_cast<const uint2*>(hm + limb * 4));
        mma_bf16_16816(M, A0, A1, A2, A3, bm.x, bm.y);
        hsum += bf16_bits_to_f32(bm.x & 0xFFFFu) + bf16_bits_to_f32(bm.x >> 16) +
                bf16_bits_to_f32(bm.y & 0xFFFFu) + bf16_bits_to_f32(bm.y >> 16);
      }
    }
    // block sum of h for column g, then for the C-fragment columns 2t and 2t+1
    hsum += __shfl_xor_sync(0xffffffffu, hsum, 1);
    hsum += __shfl_xor_sync(0xffffffffu, hsum, 2);
    const float x0 = __shfl_sync(0xffffffffu, hsum, (2 * t) * 4);
    const float x1 = __shfl_sync(0xffffffffu, hsum, (2 * t + 1) * 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t ddv = dd[i >> 1];
      const float dv = f16_bits_to_f32(ddv & 0xFFFFu), dmv = f16_bits_to_f32(ddv >> 16);
      const float xs = (i & 1) ? x1 : x0;
      const float psum = (P[0][i] + P[1][i]) + (P[2][i] + P[3][i]);
      const float mv = fmaf(-128.0f, xs, M[i]);
      acc[i] = fmaf(dv, psum, fmaf(-dmv, mv, acc[i]));
    }
  }
}

// ----------------------------------------------------------------------------
// phase 2, shared Q8_0 down: 16 rows over one chunk; B = h limbs (natural order)
// ----------------------------------------------------------------------------
__device__ __forceinline__ void p2_q80_chunk(const unsigned char* stage, int cb, int c, int g, int t, int Fs,
                                             const uint16_t* hrow_g,  // hS[tok_g][0][:] or null
                                             const float* hs16_0, const float* hs16_1, float (&acc)[4]) {
  const int chunk_bytes = cb * Q80_BB;
  for (int bl = 0; bl < cb; ++bl) {
    const int bq = c * cb + bl;
    float Ph[4] = {0.f, 0.f, 0.f, 0.f}, Pl[4] = {0.f, 0.f, 0.f, 0.f};
    uint32_t dd[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint2 bh = make_uint2(0u, 0u), blo = make_uint2(0u, 0u);
      if (hrow_g) {
        bh = __ldg(reinterpret_cast<const uint2*>(hrow_g + 32 * bq + 16 * hf + 4 * t));
        blo = __ldg(reinterpret_cast<const uint2*>(hrow_g + Fs + 32 * bq + 16 * hf + 4 * t));
      }
      uint32_t l01[2], l23[2], h01[2], h23[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const unsigned char* base = stage + (g + 8 * rr) * chunk_bytes + bl * Q80_BB;
        if (hf == 0) dd[rr] = lds_u16(base);
        q80_frag(lds_u32_a2(base + 2 + 16 * hf + 4 * t), l01[rr], l23[rr], h01[rr], h23[rr]);
      }
      mma_bf16_16816(Pl, l01[0], l01[1], l23[0], l23[1], bh.x, bh.y);
      mma_bf16_16816(Pl, l01[0], l01[1], l23[0], l23[1], blo.x, blo.y);
      mma_bf16_16816(Ph, h01[0], h01[1], h23[0], h23[1], bh.x, bh.y);
      mma_bf16_16816(Ph, h01[0], h01[1], h23[0], h23[1], blo.x, blo.y);
    }
    const float x0 = hs16_0 ? hs16_0[2 * bq] + hs16_0[2 * bq + 1] : 0.0f;
    const float x1 = hs16_1 ? hs16_1[2 * bq] + hs16_1[2 * bq + 1] : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float dv = f16_bits_to_f32(dd[i >> 1]);
      const float xs = (i & 1) ? x1 : x0;
      const float v = fmaf(-2304.0f, xs, fmaf(16.0f, Ph[i], Pl[i]));
      acc[i] = fmaf(dv, v, acc[i]);
    }
  }
}

__device__ __forceinline__ float silu_mul(float gv, float uv) { return gv / (1.0f + expf(-gv)) * uv; }

// ----------------------------------------------------------------------------
// activation package: x permuted into the Q2_K fragment order, the 16-value sub-block
// sums of x as three BF16 limbs, their block totals, and 32-value sums for Q8_0.  Built
// once per call by ffn_prep_kernel and copied whole into shared memory by phase 1.
// ----------------------------------------------------------------------------
struct PkgLayout {
  int xB, XBm, XbM, X32, total;
};

__host__ __device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }

__host__ __device__ __forceinline__ PkgLayout pkg_layout(int T, int d) {
  const int nbx = d / 256, xstride = d * 2 + 32;
  PkgLayout L;
  L.xB = 0;
  L.XBm = T * xstride;
  L.XbM = L.XBm + T * nbx * 96;
  L.X32 = L.XbM + round16(T * nbx * 4);
  L.total = L.X32 + round16(T * (d / 32) * 4);
  return L;
}

// grid (d/256, T), 256 threads: thread i owns value k = 256*b + i of token t.
//   xB: x (BF16) permuted into the Q2_K fragment order; XBm: 16-value sub-block sums as
//   three BF16 limbs; XbM: their block total; X32: 32-value sums (Q8_0 shared expert).
__global__ void __launch_bounds__(256) ffn_prep_kernel(const uint16_t* __restrict__ x, int T, int d,
                                                       unsigned char* __restrict__ pkg) {
  __shared__ float sub_limbs[16];
  pdl_wait();
  const int b = blockIdx.x, t = blockIdx.y, i = threadIdx.x, lane = i & 31;
  const int nbx = d / 256;
  const PkgLayout L = pkg_layout(T, d);
  const uint32_t v = x[(size_t)t * d + 256 * b + i];
  {
    // fragment order: step (jj, s) of thread tq holds codes s, 8+s | 4+s, 12+s of sub-block 4tq+jj,
    // each activation scaled by 4^-min(s,2) to match the code left in place in the A fragment
    const int j = i >> 4, tq = j >> 2, jj = j & 3, ip = i & 15;
    const int byte = ip >> 2, s = ip & 3;
    const int v4 = (byte & 1) * 2 + (byte >> 1);
    const int rem = ((((b * 4 + jj) * 4 + s) * 4 + tq) * 4 + v4);
    const float scaled = __fmul_rn(bf16_bits_to_f32(v), s == 0 ? 1.0f : (s == 1 ? 0.25f : 0.0625f));
    reinterpret_cast<uint16_t*>(pkg + L.xB + (size_t)t * (d * 2 + 32))[rem] = (uint16_t)f32_to_bf16_rne(scaled);
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
    sub_limbs[j] = (bf16_bits_to_f32(hi) + bf16_bits_to_f32(mid)) + bf16_bits_to_f32(lo);
  }
  __syncthreads();
  if (i == 0) {
    float sacc = 0.0f;
    for (int j = 0; j < 16; ++j) sacc += sub_limbs[j];
    reinterpret_cast<float*>(pkg + L.XbM)[(size_t)t * nbx + b] = sacc;
  }
}

// ----------------------------------------------------------------------------
// the kernel
// ----------------------------------------------------------------------------
template <int PHASE>
__global__ void __launch_bounds__(MAX_WARPS * 32, 1) ffn_decode_kernel(const DecParams p) {
  extern __shared__ __align__(128) unsigned char sm[];
  const int nw = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
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
    mbar_arrive_expect_tx(pkg_bar, PL.total);
    bulk_g2s(xprep, p.pkg, PL.total, pkg_bar);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) p.counters[PHASE == 1 ? 1 : 0] = 0;

  const int n_act = *p.n_active;
  const int tiles_s = p.has_shared ? p.rows_s / 16 : 0;
  const int tiles_r = p.rows_r / 16;
  const int n_items = tiles_s + n_act * tiles_r;

  unsigned char* my_stage = stages + warp * NS * STAGE;
  uint64_t* my_bar = bars + warp * NS;

  auto fetch = [&]() -> int {
    int i = 0;
    if (lane == 0) i = atomicAdd(&p.counters[PHASE - 1], 1);
    i = __shfl_sync(0xffffffffu, i, 0);
    return i < n_items ? i : -1;
  };

  int queue[NS + 2];
  int qh = 0, qt = 0;
  int ld_id = fetch();
  queue[qt++ % (NS + 2)] = ld_id;
  Item ld_it = decode_item<PHASE>(p, ld_id, n_act, tiles_s, tiles_r);
  int ld_c = 0, ld_seq = 0;
  auto issue_next = [&]() {
    if (ld_it.id < 0) return;
    issue_chunk<PHASE>(ld_it, ld_c, my_stage + (ld_seq % NS) * STAGE, &my_bar[ld_seq % NS], lane);
    ++ld_seq;
    if (++ld_c == ld_it.C) {
      ld_id = fetch();
      queue[qt++ % (NS + 2)] = ld_id;
      ld_it = decode_item<PHASE>(p, ld_id, n_act, tiles_s, tiles_r);
      ld_c = 0;
    }
  };
  for (int i = 0; i < NS; ++i) issue_next();

  // ---- phase 1: the activation package arrives in shared memory by one bulk copy
  const int T = p.T;
  const int d = p.d;
  const int nbx = d / 256;
  unsigned char* xB = xprep + PL.xB;                                   // [T][xstride]
  unsigned char* XBm = xprep + PL.XBm;                                 // [T][nbx][4][3][4] bf16
  float* XbM = reinterpret_cast<float*>(xprep + PL.XbM);              // [T][nbx]
  float* X32 = reinterpret_cast<float*>(xprep + PL.X32);              // [T][d/32]
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
    const int id = queue[qh % (NS + 2)];
    if (id < 0) break;
    const Item it = decode_item<PHASE>(p, id, n_act, tiles_s, tiles_r);
    const int r0 = it.tile * 16;
    // column -> token (phase 1) or h row (phase 2)
    auto col_src = [&](int col) -> int {
      if (col >= it.n) return -1;
      if (it.shared) return col;                                  // token; phase-2 h row of the shared expert
      const int pos = it.off + col;
      return (PHASE == 1) ? __ldg(p.perm + pos) / p.k : pos;
    };
    const int sg = col_src(g), sc0 = col_src(2 * t), sc1 = col_src(2 * t + 1);
    float acc2[2][4];
#pragma unroll
    for (int m = 0; m < 2; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc2[m][i] = 0.0f;

    for (int c = 0; c < it.C; ++c) {
      const int st = cs_seq % NS;
      if (!mbar_wait_bounded(&my_bar[st], (cs_seq / NS) & 1, WAIT_LIMIT)) {
        if (lane == 0) set_err(p.err, BRE_DEVERR_TIMEOUT);
        for (int q = cs_seq + 1; q < ld_seq; ++q) mbar_wait_bounded(&my_bar[q % NS], (q / NS) & 1, WAIT_LIMIT);
        return;
      }
      const unsigned char* stage = my_stage + st * STAGE;
      if (PHASE == 1) {
        if (it.shared) {
          p1_q80_chunk(stage, it.cb, c, g, t, sg >= 0 ? p.x + (size_t)sg * d : nullptr,
                       sc0 >= 0 ? X32 + sc0 * (d / 32) : nullptr, sc1 >= 0 ? X32 + sc1 * (d / 32) : nullptr, acc2);
        } else {
          p1_q2k_chunk(stage, it.cb, c, g, t, sg >= 0 ? xB + (size_t)sg * p.xstride : nullptr,
                       sg >= 0 ? XBm + (size_t)sg * nbx * 96 : nullptr, sc0 >= 0 ? XbM + sc0 * nbx : nullptr,
                       sc1 >= 0 ? XbM + sc1 * nbx : nullptr, acc2);
        }
      } else {
        if (it.shared) {
          p2_q80_chunk(stage, it.cb, c, g, t, p.Fs, sg >= 0 ? p.hS + (size_t)sg * 2 * p.Fs : nullptr,
                       sc0 >= 0 ? p.HS16 + (size_t)sc0 * (p.Fs / 16) : nullptr,
                       sc1 >= 0 ? p.HS16 + (size_t)sc1 * (p.Fs / 16) : nullptr, acc2[0]);
        } else {
          p2_q2k_chunk(stage, it.cb, c, Fnb, g, t, sg, p.hB, p.HBm, acc2[0]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      ++cs_seq;
      issue_next();
    }
    ++qh;

    // ---- epilogue
    if (PHASE == 1) {
      // h = silu(gate) * up, stored as two bf16 limbs; per-column sums over the 16 rows
      float hs[2] = {0.0f, 0.0f};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int col_src_i = (i & 1) ? sc1 : sc0;
        const int row = r0 + g + 8 * (i >> 1);
        float h = silu_mul(acc2[0][i], acc2[1][i]);
        uint32_t hi, lo;
        split_bf16x2(h, hi, lo);
        const float hq = bf16_bits_to_f32(hi) + bf16_bits_to_f32(lo);
        if (col_src_i >= 0) {
          hs[i & 1] += hq;
          if (it.shared) {
            p.hS[((size_t)col_src_i * 2 + 0) * p.Fs + row] = (uint16_t)hi;
            p.hS[((size_t)col_src_i * 2 + 1) * p.Fs + row] = (uint16_t)lo;
          } else {
            const int pos = it.off + 2 * t + (i & 1);
            const int b2 = row >> 8, j = (row >> 4) & 15, ip = row & 15;
            const int byte = ip >> 2, s = ip & 3, v4 = (byte & 1) * 2 + (byte >> 1);
            // limbs of h * 4^-min(s,2) (the down projection's A fragments keep codes in place)
            uint32_t shi, slo;
            split_bf16x2(__fmul_rn(h, s == 0 ? 1.0f : (s == 1 ? 0.25f : 0.0625f)), shi, slo);
            const size_t base = ((((size_t)pos * Fnb + b2) * 4 + (j & 3)) * 4 + s) * 4 * 8 + (size_t)(j >> 2) * 8;
            p.hB[base + v4] = (uint16_t)shi;
            p.hB[base + 4 + v4] = (uint16_t)slo;
          }
        }
      }
#pragma unroll
      for (int o = 4; o <= 16; o <<= 1) {
        hs[0] += __shfl_xor_sync(0xffffffffu, hs[0], o);
        hs[1] += __shfl_xor_sync(0xffffffffu, hs[1], o);
      }
      if (g == 0) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int col = 2 * t + q;
          if (col < it.n) {
            if (it.shared) {
              p.HS16[(size_t)col * (p.Fs / 16) + (r0 >> 4)] = hs[q];
            } else {
              const int pos = it.off + col;
              const int b2 = r0 >> 8, j = (r0 >> 4) & 15;
              uint32_t hi = f32_to_bf16_rne(hs[q]);
              const float r1 = hs[q] - bf16_bits_to_f32(hi);
              uint32_t mid = f32_to_bf16_rne(r1);
              uint32_t lo = f32_to_bf16_rne(r1 - bf16_bits_to_f32(mid));
              uint16_t* dst = p.HBm + (((size_t)pos * Fnb + b2) * 4 + (j >> 2)) * 12 + (j & 3);
              dst[0] = (uint16_t)hi;
              dst[4] = (uint16_t)mid;
              dst[8] = (uint16_t)lo;
            }
          }
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

}  // namespace

size_t ffn_ws_bytes(int T, int k, int E, int d, int F, int Fs) {
  (void)E;
  if (T > DECODE_T_MAX) return ffn_gemm_ws_bytes(T, k, d, F, Fs);
  const size_t P = (size_t)T * k;
  size_t s = 1024 + pkg_layout(T, d).total;              // counters, activation package
  s += P * (F / 256) * 512 * 2;                          // hB
  s += P * (F / 256) * 4 * 12 * 2;                       // HBm
  s += (size_t)T * 2 * Fs * 2;                           // hS
  s += (size_t)T * (Fs / 16) * 4;                        // HS16
  return (s + 255) & ~(size_t)255;
}

bre_status ffn_check_shapes(const bre_ffn_weights* r, const bre_ffn_weights* sh, int T) {
  const int d = r->d, F = r->d_ff;
  if (d <= 0 || F <= 0 || d % 256 || F % 256) return BRE_ERR_UNSUPPORTED;
  if (sh && (sh->d != d || sh->d_ff <= 0 || sh->d_ff % 256)) return BRE_ERR_UNSUPPORTED;
  if (T <= DECODE_T_MAX) {
    // Q2_K rows go to shared memory by 16-byte aligned bulk copies: whole 16-row tiles when
    // they fit a stage, otherwise 4-block (336-byte) pieces of rows a multiple of 4 blocks long
    if (!(d <= 1024 || d % 1024 == 0)) return BRE_ERR_UNSUPPORTED;
    if (!(F <= 2048 || F % 1024 == 0)) return BRE_ERR_UNSUPPORTED;
  }
  return BRE_OK;
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
  const size_t P = (size_t)a.T * a.k;
  char* w = reinterpret_cast<char*>(a.ws);
  p.counters = reinterpret_cast<int*>(w);
  w += 1024;
  p.pkg = reinterpret_cast<const unsigned char*>(w);
  unsigned char* pkg_w = reinterpret_cast<unsigned char*>(w);
  w += pkg_layout(a.T, p.d).total;
  p.hB = reinterpret_cast<uint16_t*>(w);
  w += P * (p.F / 256) * 512 * 2;
  p.HBm = reinterpret_cast<uint16_t*>(w);
  w += P * (p.F / 256) * 4 * 12 * 2;
  p.hS = reinterpret_cast<uint16_t*>(w);
  w += (size_t)a.T * 2 * p.Fs * 2;
  p.HS16 = reinterpret_cast<float*>(w);
  p.xstride = p.d * 2 + 32;

  const int sms = device_sm_count();
  const int smem_max = device_max_smem_optin();
  ffn_prep_kernel<<<dim3(p.d / 256, a.T), 256, 0, s>>>(a.x, a.T, p.d, pkg_w);
  {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  for (int phase = 1; phase <= 2; ++phase) {
    const int cap = (phase == 1) ? STAGE / 2 : STAGE;
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
    p.cb_r = pick_chunk(p.nb_r, Q2K_BB, cap, 4, &p.whole_r);
    p.cb_s = S ? pick_chunk(p.nb_s, Q80_BB, cap, 8, &p.whole_s) : 1;
    if (p.cb_r <= 0 || p.cb_s <= 0) return cudaErrorInvalidValue;
    const size_t xbytes = (phase == 1) ? (size_t)pkg_layout(a.T, p.d).total : 0;
    int nw = MAX_WARPS;
    while (nw > 1 && (size_t)nw * NS * STAGE + BAR_BYTES + xbytes > (size_t)smem_max) --nw;
    const size_t smem = (size_t)nw * NS * STAGE + BAR_BYTES + xbytes;
    if (smem > (size_t)smem_max) return cudaErrorInvalidValue;
    cudaError_t e;
    if (phase == 1) {
      e = cudaFuncSetAttribute(ffn_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      ffn_decode_kernel<1><<<sms, nw * 32, smem, s>>>(p);
    } else {
      e = cudaFuncSetAttribute(ffn_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      ffn_decode_kernel<2><<<sms, nw * 32, smem, s>>>(p);
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
