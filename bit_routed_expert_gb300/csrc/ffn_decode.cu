// Expert FFN for decode-sized batches (at most 8 tokens per expert).
//
// Strata-DSV4.1 README, V4-Flash "How it works" (experts, then the finish step:
// shared expert + routed sum) and "Verifying it" (the expert tier is checked
// against a dequantised F32 reference); SwiGLU from the V4-Flash description.
//
// Design (GB300): the path is bound by streaming 2-bit weights from HBM, so every byte is read
// once and the work per byte is kept small.  The routed experts are stored in the Q2_K_R16
// layout (repack.cu): each 1344-byte tile holds one 256-weight block of 16 rows arranged so
// that lane L of a warp finds the codes of its two fragment rows as one 16-byte word group,
// and the scale and min nibbles of its sub-blocks in one 8-byte pair.  Each consumer warp owns
// a two-stage ring in shared memory that a producer warp fills with one-dimensional bulk copies
// of whole tiles; the consumer dequantises in registers straight into mma.sync A fragments and
// multiplies by the expert's tokens (N = 8 columns).  After a fixed first item per consumer,
// work items are handed out by an atomic counter so that busy SMs take fewer items.
//
// Exactness: a Q2_K weight is (d*sc)*q - dmin*m.  A fragment register holds two BF16 values
// sc*q*4^e (e in {0, 1, 2}, exact): a mask leaves the code in place inside the mantissa of 128
// and one bf16x2 FMA with (sc, -128 sc) removes the 128; the activations carry 4^-e (exact).
// One 256-weight block of a row contributes d * P - dmin * M with P = sum sc q x and
// M = sum_j m_j X_j, X_j the 16-value sub-block sums of the activations (three BF16 limbs, a
// second small MMA whose A fragments are the 4-bit mins).  A Q8_0 weight d*q is split into
// nibbles in phase 1 (q + 128 = 16*hi + lo, each held as BF16 128 + nibble) and held as FP16
// 1024 + (q + 128) in phase 2, against h as block-scaled FP16.  Products are exact; accumulation
// is FP32.
//
// K order: the MMA sums over k, so the k order inside a block is free as long as A and B
// agree.  Step s (0..15) of lane (g, t) takes, for rows g and g + 8, word 2p + w of the lane's
// codes (p = s / 8, w = (s / 4) % 2) and in it slots 2u and 2u + 1 (u = s % 4; slot v holds
// code 8w + v of the sub-blocks 4t + 2p (low half) and 4t + 2p + 1 (high half)); the
// activations are stored in that order (frag_pos).  Q8_0 uses natural order.
#include <cuda_fp16.h>

#include <algorithm>
#include <mutex>

#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

namespace {

constexpr int NS = 2;                 // ring stages per warp
constexpr int TAIL_ROUNDS = 1;        // phase 1: finer K parts for about this many items per consumer
constexpr int STAGE = 5376;           // bytes per stage: four Q2_K_R16 tiles, or 16 Q8_0 rows x 8 blocks
constexpr int R16 = 1344;             // bytes per Q2_K_R16 tile (16 rows x one block)
constexpr int MAX_CONS = 15;          // consumer warps (plus one producer warp: 128 registers a
                                      // thread); fewer when the activation package leaves less
                                      // shared memory
constexpr int RT1 = 2;                // row tiles per item, phase 1 (one B load serves both)
constexpr int RT2 = 2;                // row tiles per item, phase 2 (one B load from global memory serves both)
constexpr uint32_t SEL_LO = 0x4140u;  // bytes 0,1 -> (128+b0, 128+b1) as bf16x2
constexpr uint32_t SEL_HI = 0x4342u;  // bytes 2,3
constexpr long long WAIT_LIMIT = 2000000000LL;  // cycles (~1 s) before a wait gives up
constexpr int BAR_BYTES = 1024;                 // mbarriers: full and empty per ring stage + the package's
constexpr int DESC_BYTES = MAX_CONS * NS * 64;  // stage descriptors: 16 ints per ring stage
static_assert((2 * MAX_CONS * NS + 1) * 8 <= BAR_BYTES, "mbarrier region too small");
static_assert(RT1 * 2 * R16 == STAGE && RT2 * 2 * R16 == STAGE, "a full stage holds four tiles");

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

// Bit patterns held in registers (kernel parameters) rather than rebuilt as immediates inside
// the loops: m43 = BF16 (128, 128), m128 = (-128, -128), k16384 = (16384, 16384), k43 = the
// byte 0x43 four times (PRMT source of the exponent byte of 128), k64 = the byte 0x64 four
// times (the high byte of FP16 1024 + u, u < 256).
struct DecConst {
  uint32_t m43, m128, k16384, k43, k64;
};

struct DecParams {
  const uint8_t* rw0;  // routed (Q2_K_R16): phase 1 gate, phase 2 down
  const uint8_t* rw1;  // routed: phase 1 up
  long long rs0, rs1;  // routed expert strides (bytes)
  const uint8_t* sw0;  // shared expert (Q8_0): phase 1 gate, phase 2 down
  const uint8_t* sw1;  // shared: phase 1 up
  int has_shared;
  int d, F, Fs, T, k, E;
  int rows_r, rows_s;  // rows per matrix of a routed / the shared expert
  int nb_r, nb_s;      // blocks per row (Q2_K: 256 weights, Q8_0: 32)
  int bps;             // routed blocks per stage
  int cb_s, whole_s;   // shared: blocks per chunk, whole 16-row tile in one bulk copy
  int n_mat;           // matrices per phase (2: gate and up items, 1: down)
  int rg_r;            // routed row groups per matrix (rows_r / (16 * RT))
  int tiles_s;         // shared 16-row tiles per matrix
  int kp_r, kp_s;      // K parts of a routed row group / a shared tile
  int cpp_r, cpp_s;    // stages of a routed / shared item (per K part)
  // phase 1 tail: the last experts of the active list take kp_t (= 2 kp_r when the row's stages
  // allow it) K parts of cpp_t stages, so that the items claimed last are short; enough experts
  // for about tail_items items.  Partial sums of every routed item use the stride kp_t.
  int kp_t, cpp_t, tail_items;
  FDiv fd_kps, fd_tkps, fd_kpr, fd_rgkpr, fd_per_exp, fd_k, fd_kpt, fd_rgkpt, fd_per_exp_t;
  const uint16_t* x;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* n_active;
  const unsigned char* pkg;  // activation package in global memory (phase 1)
  int xstride, xlstride;     // bytes per token of the package's fragment-order x and limb rows
  const uint16_t* hf;        // phase 2: routed h (BF16), fragment order: [P][F/256][256]
  const uint16_t* hl;        // phase 2: routed 16-row sums of h, 3 limbs: [P][F/256][3][4][4]
  const uint16_t* hS16;      // phase 2: shared h as block-scaled FP16 (block_f16), natural order: [T][Fs]
  const float2* HQ;          // phase 2: per 32-row block of it, (sum of the 32 FP16 values, 2^s): [T][Fs/32]
  float* part_r;             // phase 1 partial sums: [pair][tile][K part][gate|up][16 rows]
  float* part_s;             // phase 1 partial sums: [token][tile][K part][gate|up][16 rows]
  float* y_pairs;
  float* y_shared;
  int red_r, red_s;          // phase 2: routed / shared outputs are sums of two K parts added into zeros
  int* counters;
  int32_t* err;
  long long wait;            // budget (cycles) of the ring and package waits; drains use WAIT_LIMIT
  DecConst kc;
};

struct Item {
  int id;       // -1: none
  bool shared;
  int m;        // matrix: 0 gate / down, 1 up
  int e, off, n;
  int grp;      // routed row group or shared 16-row tile
  int kp;       // K part
  int nch;      // stages of the item
  const uint8_t* src;
};

// Experts at the end of the active list that take the tail's finer K parts (phase 1): enough
// of them for about tail_items items, none when the K parts cannot be split further.
__host__ __device__ __forceinline__ int tail_experts(int n_act, int per_exp_t, int tail_items, int kp_t, int kp_r) {
  if (kp_t == kp_r || n_act <= 0) return 0;
  const int n = (tail_items + per_exp_t - 1) / per_exp_t;
  return n < n_act ? n : n_act;
}

// Items: the shared expert's (matrix, tile, K part) first, then per active expert (matrix, row
// group, K part); in phase 1 the experts from a_split on take the tail's K parts.
template <int PHASE>
__device__ __forceinline__ Item decode_item(const DecParams& p, int id, int n_shared_items, int a_split) {
  Item it;
  it.id = id;
  if (id < 0) return it;
  if (id < n_shared_items) {
    it.shared = true;
    it.m = fdiv(id, p.fd_tkps);
    const int r = id - it.m * (p.tiles_s * p.kp_s);
    it.grp = fdiv(r, p.fd_kps);
    it.kp = r - it.grp * p.kp_s;
    it.e = -1;
    it.off = 0;
    it.n = p.T;
    it.nch = p.cpp_s;
    it.src = it.m ? p.sw1 : p.sw0;
  } else {
    const int r = id - n_shared_items;
    const int per_exp = p.n_mat * p.rg_r * p.kp_r;
    int a, r2, kpn;
    if (PHASE == 2 || r < a_split * per_exp) {
      a = fdiv(r, p.fd_per_exp);
      r2 = r - a * per_exp;
      it.m = fdiv(r2, p.fd_rgkpr);
      const int r3 = r2 - it.m * (p.rg_r * p.kp_r);
      it.grp = fdiv(r3, p.fd_kpr);
      it.kp = r3 - it.grp * p.kp_r;
      kpn = 0;
    } else {
      const int rt = r - a_split * per_exp;
      const int at = fdiv(rt, p.fd_per_exp_t);
      a = a_split + at;
      r2 = rt - at * (p.n_mat * p.rg_r * p.kp_t);
      it.m = fdiv(r2, p.fd_rgkpt);
      const int r3 = r2 - it.m * (p.rg_r * p.kp_t);
      it.grp = fdiv(r3, p.fd_kpt);
      it.kp = r3 - it.grp * p.kp_t;
      kpn = 1;
    }
    it.shared = false;
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
    it.nch = kpn ? p.cpp_t : p.cpp_r;
    it.src = it.m ? p.rw1 + (long long)it.e * p.rs1 : p.rw0 + (long long)it.e * p.rs0;
  }
  return it;
}

// Lane 0 issues the copies of stage c of `it` into `stage`.  Routed: for each of the item's RT
// row tiles one bulk copy of bps consecutive R16 tiles (stage layout [row tile][block][1344]).
// Shared: one bulk copy of a whole 16-row tile, or one tensor copy of a 16-row x cb-block box.
template <int RT>
__device__ __forceinline__ void issue_stage(const DecParams& p, const Item& it, int c, unsigned char* stage,
                                            uint64_t* bar, int lane, const CUtensorMap* map_s0,
                                            const CUtensorMap* map_s1) {
  if (lane != 0) return;
  if (it.shared) {
    const int chunk_bytes = p.cb_s * Q80_BB;
    const uint32_t bytes = 16u * chunk_bytes;
    mbar_arrive_expect_tx(bar, bytes);
    if (p.whole_s) {
      bulk_g2s(stage, it.src + (long long)it.grp * 16 * chunk_bytes, bytes, bar);
    } else {
      const int ch = it.kp * p.cpp_s + c;
      tma_load_3d(stage, it.m ? map_s1 : map_s0, ch * (chunk_bytes / 4), it.grp * 16, 0, bar);
    }
  } else {
    const uint32_t span = (uint32_t)p.bps * R16;
    mbar_arrive_expect_tx(bar, RT * span);
    const int b0 = (it.kp * it.nch + c) * p.bps;
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const long long tile = (long long)(it.grp * RT + r) * p.nb_r + b0;
      bulk_g2s(stage + r * span, it.src + tile * R16, span, bar);
    }
  }
}

__device__ __forceinline__ uint32_t lds_u16(const unsigned char* p) {
  return *reinterpret_cast<const unsigned short*>(p);
}
__device__ __forceinline__ uint32_t lds_u32_a2(const unsigned char* p) {  // 2-byte aligned
  return lds_u16(p) | (lds_u16(p + 2) << 16);
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

// ----------------------------------------------------------------------------
// fragment order of a 256-value block (activations x in phase 1, h in phase 2)
// ----------------------------------------------------------------------------
// Value i of a block (sub-block j = i / 16, code r = i % 16) is the B operand of lane t = j / 4
// at step s = 8p + 4w + v / 2 (p = (j % 4) / 2, w = r / 8, v = r % 8), in half h = j % 2 of
// register b0 (v even) or b1 (v odd), scaled by 4^-e (e = v % 3 for v < 6, v - 6 after: the
// code's position inside its 16-bit half after the word's shift by 0, 6 or 12).  Storage
// [s / 2][t][step parity][b0.lo, b0.hi, b1.lo, b1.hi]: lane t loads 16 bytes per step pair.
__host__ __device__ __forceinline__ int frag_pos(int i, int* e) {
  const int j = i >> 4, r = i & 15;
  const int t = j >> 2, p = (j >> 1) & 1, h = j & 1;
  const int w = r >> 3, v = r & 7;
  const int s = 8 * p + 4 * w + (v >> 1);
  *e = v < 3 ? v : (v < 6 ? v - 3 : v - 6);
  return (((s >> 1) * 4 + t) * 2 + (s & 1)) * 4 + 2 * (v & 1) + h;
}

// Limbs of the 16-value sub-block sums: [limb][t][j % 4] per block (96 bytes); lane t loads the
// four sums of its sub-blocks 4t .. 4t+3 as one 8-byte word per limb.
__host__ __device__ __forceinline__ int limb_pos(int j, int limb) { return (limb * 4 + (j >> 2)) * 4 + (j & 3); }

// ----------------------------------------------------------------------------
// one 256-weight block of RT row tiles (Q2_K_R16), 16 rows each
// ----------------------------------------------------------------------------
// A fragments of step u (0..3) of one code word: slots 2u, 2u + 1 (codes at bits 2v' of the
// word shifted by 0, 6 or 12; the mask takes one code in each half, the OR the exponent of 128).
template <int U>
__device__ __forceinline__ void word_slots(uint32_t w0, uint32_t w6, uint32_t w12, uint32_t m43, uint32_t& ea,
                                           uint32_t& eb) {
  if constexpr (U == 0) {
    ea = (w0 & 0x00030003u) | m43;
    eb = (w0 & 0x000C000Cu) | m43;
  } else if constexpr (U == 1) {
    ea = (w0 & 0x00300030u) | m43;
    eb = (w6 & 0x00030003u) | m43;
  } else if constexpr (U == 2) {
    ea = (w6 & 0x000C000Cu) | m43;
    eb = (w6 & 0x00300030u) | m43;
  } else {
    ea = (w12 & 0x00030003u) | m43;
    eb = (w12 & 0x000C000Cu) | m43;
  }
}

__device__ __forceinline__ uint32_t u4_word(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// The block's B operand: PHASE 1 reads it from shared memory (xb: this lane's 16-byte column of
// the block), PHASE 2 from registers filled a block ahead (B), refilling each step pair from
// `next` once its MMAs are issued.
template <int PHASE, int RT, int TS>
__device__ __forceinline__ void q2k_block(const unsigned char* u0, int lane, int g, const unsigned char* xb,
                                          uint4 (&B)[8], const uint16_t* __restrict__ next, const uint2 (&bm)[3],
                                          const DecConst& k, float (&acc)[RT][4]) {
  uint4 c0[RT], c1[RT];
  uint2 sw[RT], dd[RT];
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    const unsigned char* u = u0 + r * TS;
    c0[r] = *reinterpret_cast<const uint4*>(u + 16 * lane);
    c1[r] = *reinterpret_cast<const uint4*>(u + 512 + 16 * lane);
    sw[r] = *reinterpret_cast<const uint2*>(u + 1024 + 8 * lane);
    dd[r] = *reinterpret_cast<const uint2*>(u + 1280 + 8 * g);
  }
  // scale pairs: index 2 rr + p -> (sc, sc') of row 8 rr + g, sub-blocks 4t + 2p, 4t + 2p + 1
  uint32_t sc2[RT][4], nsc2[RT][4];
#pragma unroll
  for (int r = 0; r < RT; ++r)
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t u = ((sw[r].x >> (4 * i)) & 0x000F000Fu) | k.m43;   // 128 + sc
      sc2[r][i] = bf16x2_sub(u, k.m43);
      nsc2[r][i] = bf16x2_fma(u, k.m128, k.k16384);                      // -128 sc
    }
  float P[RT][4];
#pragma unroll
  for (int pw = 0; pw < 4; ++pw) {   // word 2p + w of the lane's codes
    const int p = pw >> 1;
    uint32_t g0[RT], g6[RT], g12[RT], h0[RT], h6[RT], h12[RT];
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      g0[r] = u4_word(c0[r], pw);
      h0[r] = u4_word(c1[r], pw);
      g6[r] = g0[r] >> 6;
      g12[r] = g0[r] >> 12;
      h6[r] = h0[r] >> 6;
      h12[r] = h0[r] >> 12;
    }
#pragma unroll
    for (int sp = 0; sp < 2; ++sp) {   // step pair (2 sp, 2 sp + 1) within the word
      const int q = pw * 2 + sp;       // the block's step pair, 0..7
      uint4 bq;
      if constexpr (PHASE == 1)
        bq = *reinterpret_cast<const uint4*>(xb + q * 64);
      else
        bq = B[q];
#pragma unroll
      for (int ss = 0; ss < 2; ++ss) {
        const int u = 2 * sp + ss;
        const uint32_t b0 = ss ? bq.z : bq.x, b1 = ss ? bq.w : bq.y;
#pragma unroll
        for (int r = 0; r < RT; ++r) {
          uint32_t ea, eb, fa, fb;
          if (u == 0) {
            word_slots<0>(g0[r], g6[r], g12[r], k.m43, ea, eb);
            word_slots<0>(h0[r], h6[r], h12[r], k.m43, fa, fb);
          } else if (u == 1) {
            word_slots<1>(g0[r], g6[r], g12[r], k.m43, ea, eb);
            word_slots<1>(h0[r], h6[r], h12[r], k.m43, fa, fb);
          } else if (u == 2) {
            word_slots<2>(g0[r], g6[r], g12[r], k.m43, ea, eb);
            word_slots<2>(h0[r], h6[r], h12[r], k.m43, fa, fb);
          } else {
            word_slots<3>(g0[r], g6[r], g12[r], k.m43, ea, eb);
            word_slots<3>(h0[r], h6[r], h12[r], k.m43, fa, fb);
          }
          const uint32_t a0 = bf16x2_fma(ea, sc2[r][p], nsc2[r][p]);
          const uint32_t a2 = bf16x2_fma(eb, sc2[r][p], nsc2[r][p]);
          const uint32_t a1 = bf16x2_fma(fa, sc2[r][2 + p], nsc2[r][2 + p]);
          const uint32_t a3 = bf16x2_fma(fb, sc2[r][2 + p], nsc2[r][2 + p]);
          if (pw == 0 && u == 0)
            mma_bf16_16816_z(P[r], a0, a1, a2, a3, b0, b1);
          else
            mma_bf16_16816(P[r], a0, a1, a2, a3, b0, b1);
        }
      }
      if constexpr (PHASE == 2) B[q] = __ldg(reinterpret_cast<const uint4*>(next) + q * 4);
    }
  }
  // min term: M = sum_j m_j X_j over the 16 sub-blocks, X_j in three limbs
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    uint32_t am[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) am[i] = bf16x2_sub(((sw[r].y >> (4 * i)) & 0x000F000Fu) | k.m43, k.m43);
    float M[4];
    mma_bf16_16816_z(M, am[0], am[2], am[1], am[3], bm[0].x, bm[0].y);
    mma_bf16_16816(M, am[0], am[2], am[1], am[3], bm[1].x, bm[1].y);
    mma_bf16_16816(M, am[0], am[2], am[1], am[3], bm[2].x, bm[2].y);
    const float dg = f16_bits_to_f32(dd[r].x & 0xFFFFu), mg = f16_bits_to_f32(dd[r].x >> 16);
    const float d8 = f16_bits_to_f32(dd[r].y & 0xFFFFu), m8 = f16_bits_to_f32(dd[r].y >> 16);
    acc[r][0] = fmaf(dg, P[r][0], fmaf(-mg, M[0], acc[r][0]));
    acc[r][1] = fmaf(dg, P[r][1], fmaf(-mg, M[1], acc[r][1]));
    acc[r][2] = fmaf(d8, P[r][2], fmaf(-m8, M[2], acc[r][2]));
    acc[r][3] = fmaf(d8, P[r][3], fmaf(-m8, M[3], acc[r][3]));
  }
}

// One stage of a routed item: BPS consecutive blocks of RT row tiles (stage layout [row tile]
// [block][1344]).  xb / xl: this lane's column of the activation fragments / limbs at the stage's
// first block (phase 1); hcol / hl: the same for h in global memory (phase 2), with B holding the
// stage's first block and refilled a block ahead (at the item's last block from itself).
template <int PHASE, int RT, int BPS>
__device__ __forceinline__ void routed_stage(const unsigned char* stage, int lane, int g, const unsigned char* xb,
                                             const unsigned char* xl, uint4 (&B)[8], const uint16_t* hcol,
                                             const uint16_t* hl, bool item_last, const DecConst& k,
                                             float (&acc)[RT][4]) {
  if constexpr (RT * BPS <= 4) {
    if constexpr (PHASE == 1) {
      // the loop stays rolled (unrolled, its two row tiles per block run slower)
#pragma unroll 1
      for (int bl = 0; bl < BPS; ++bl) {
        uint2 bm[3];
#pragma unroll
        for (int l = 0; l < 3; ++l) bm[l] = __ldg(reinterpret_cast<const uint2*>(xl + l * 32));
        q2k_block<1, RT, BPS * R16>(stage, lane, g, xb, B, nullptr, bm, k, acc);
        xb += 512;
        xl += 96;
        stage += R16;
      }
    } else {
      // two row tiles share each block's B registers; the loop stays rolled (unrolled, its
      // registers spill): down launch at T = 8 about 1 us shorter than with one row tile an item
#pragma unroll 1
      for (int bl = 0; bl < BPS; ++bl) {
        uint2 bm[3];
#pragma unroll
        for (int l = 0; l < 3; ++l) bm[l] = __ldg(reinterpret_cast<const uint2*>(hl + l * 16));
        const bool last = item_last && bl + 1 == BPS;
        q2k_block<2, RT, BPS * R16>(stage, lane, g, nullptr, B, last ? hcol : hcol + 256, bm, k, acc);
        hcol += 256;
        hl += 48;
        stage += R16;
      }
    }
  }
}

// Q8_0 nibble planes of one row word (4 consecutive int8): (128+lo) and (128+hi') pairs.
__device__ __forceinline__ void q80_nibbles(uint32_t w, uint32_t k43, uint32_t& lo01, uint32_t& lo23, uint32_t& hi01,
                                         uint32_t& hi23) {
  const uint32_t lo = w & 0x0F0F0F0Fu;
  const uint32_t hi = ((w >> 4) ^ 0x08080808u) & 0x0F0F0F0Fu;
  lo01 = prmt(lo, k43, SEL_LO);
  lo23 = prmt(lo, k43, SEL_HI);
  hi01 = prmt(hi, k43, SEL_LO);
  hi23 = prmt(hi, k43, SEL_HI);
}

// ----------------------------------------------------------------------------
// phase 1, shared Q8_0: 16 rows of one matrix over one chunk (natural k order)
// ----------------------------------------------------------------------------
// CB > 0 fixes the chunk's block count at compile time (addresses base + immediate); CB == 0 takes cb_rt.
template <int CB>
__device__ __forceinline__ void p1_q80_mat(const unsigned char* stage, int cb_rt, int c, int g, int t,
                                           const uint16_t* xrow_g,  // global x row of column g
                                           const float* x32_0, const float* x32_1, uint32_t k43, float (&acc)[4]) {
  const int cb = CB > 0 ? CB : cb_rt;
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
        q80_nibbles(lds_u32_a2(base + 2 + 16 * hf + 4 * t), k43, l01[rr], l23[rr], h01[rr], h23[rr]);
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

// One Q8_0 row word (4 consecutive int8 codes q) as FP16 A fragments: u = q + 128 (flip the
// sign bit), then 1024 + u exactly (u sits in the mantissa of 1024) for codes 0, 1 and 2, 3.
__device__ __forceinline__ void q80_frag(uint32_t w, uint32_t k64, uint32_t& f01, uint32_t& f23) {
  const uint32_t u = w ^ 0x80808080u;
  f01 = prmt(u, k64, SEL_LO);
  f23 = prmt(u, k64, SEL_HI);
}

// h for the shared down projection's MMAs, one 32-value block (one value a lane) at a time:
// scaled by 2^-s, s from the block's largest magnitude so that every value is below 2^15, and
// rounded to FP16 (exact for BF16 values in FP16's normal range; smaller ones lose bits below
// 2^-24 of the block's largest).  Returns the lane's FP16 bits; sum = the FP32 sum of the 32 FP16 values
// (fixed butterfly order, the same in every lane), scale = 2^s.
__device__ __forceinline__ uint32_t block_f16(float v, float& sum, float& scale) {
  float m = fabsf(v);
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  int sh = 0;
  if (m > 0.0f) {
    const int e = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127;
    sh = min(max(e - 14, -100), 100);
  }
  const float down = __uint_as_float((uint32_t)(127 - sh) << 23);   // 2^-s
  scale = __uint_as_float((uint32_t)(127 + sh) << 23);               // 2^s
  const __half hv = __float2half_rn(__fmul_rn(v, down));
  float f = __half2float(hv);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) f = __fadd_rn(f, __shfl_xor_sync(0xffffffffu, f, o));
  sum = f;
  return (uint32_t)__half_as_ushort(hv);
}

// ----------------------------------------------------------------------------
// phase 2, shared Q8_0 down: 16 rows over one chunk (natural k order); B = block-scaled FP16 h of
// column g, q0 / q1 = (sum, 2^s) of the block for columns 2t, 2t + 1.
// Per 32-value block: P = sum (1152 + q) b over the FP16 MMAs, so sum q b = P - 1152 * sum b, and
// the row's d and the column's 2^s scale it back.
// ----------------------------------------------------------------------------
// CB > 0 fixes the chunk's block count at compile time (addresses base + immediate); CB == 0 takes cb_rt.
template <int CB>
__device__ __forceinline__ void q80_chunk(const unsigned char* stage, int cb_rt, int c, int g, int t,
                                          const uint16_t* brow_g, const float2* q0, const float2* q1, uint32_t k64,
                                          float (&acc)[4]) {
  const int cb = CB > 0 ? CB : cb_rt;
  const int chunk_bytes = cb * Q80_BB;
  // B and the block's (sum, scale) of block bl + 1 load while block bl is processed
  auto load_b = [&](int bq, uint2 (&b)[2], float2 (&q)[2]) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) b[hf] = __ldg(reinterpret_cast<const uint2*>(brow_g + 32 * bq + 16 * hf + 4 * t));
    q[0] = __ldg(q0 + bq);
    q[1] = __ldg(q1 + bq);
  };
  uint2 bcur[2], bnext[2];
  float2 qcur[2], qnext[2];
  load_b(c * cb, bcur, qcur);
  for (int bl = 0; bl < cb; ++bl) {
    const int bq = c * cb + bl;
    if (bl + 1 < cb) load_b(bq + 1, bnext, qnext);
    float P[4];
    uint32_t dd[2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      const uint2 bv = bcur[hf];
      uint32_t f01[2], f23[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const unsigned char* base = stage + (g + 8 * rr) * chunk_bytes + bl * Q80_BB;
        if (hf == 0) dd[rr] = lds_u16(base);
        q80_frag(lds_u32_a2(base + 2 + 16 * hf + 4 * t), k64, f01[rr], f23[rr]);
      }
      if (hf == 0)
        mma_f16_16816_z(P, f01[0], f01[1], f23[0], f23[1], bv.x, bv.y);
      else
        mma_f16_16816(P, f01[0], f01[1], f23[0], f23[1], bv.x, bv.y);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float dv = f16_bits_to_f32(dd[i >> 1]);
      const float2 q = (i & 1) ? qcur[1] : qcur[0];
      const float v = fmaf(-1152.0f, q.x, P[i]);
      acc[i] = fmaf(__fmul_rn(dv, q.y), v, acc[i]);
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      bcur[q] = bnext[q];
      qcur[q] = qnext[q];
    }
  }
}

__device__ __forceinline__ float silu_mul(float gv, float uv) { return gv / (1.0f + expf(-gv)) * uv; }

// ----------------------------------------------------------------------------
// activation package: x in the fragment order (frag_pos, scaled by 4^-e), the 16-value
// sub-block sums of x as three BF16 limbs (limb_pos), and 32-value sums for Q8_0.  Built once
// per call by ffn_prep_kernel; phase 1 copies the first two parts into shared memory.
// ----------------------------------------------------------------------------
struct PkgLayout {
  int xf, xl, x32, smem, total;
};

__host__ __device__ __forceinline__ int round16(int v) { return (v + 15) & ~15; }

// bytes per token row of the fragment-order activations: a pitch of 64 (mod 128) bytes puts the
// two tokens of a quarter warp's 16-byte loads in different bank halves
__host__ __device__ __forceinline__ int x_stride(int d) { return d * 2 + 64; }
// bytes per token row of the limbs (96 per block): 32 (mod 128), so that the four tokens of a
// half warp's 8-byte loads fall in different banks
__host__ __device__ __forceinline__ int xl_stride(int d) { return (((d / 256) * 96 + 127) & ~127) + 32; }

__host__ __device__ __forceinline__ PkgLayout pkg_layout(int T, int d) {
  PkgLayout L;
  L.xf = 0;
  L.smem = T * x_stride(d);   // the part phase 1 copies into shared memory
  L.xl = L.smem;
  L.x32 = L.xl + T * xl_stride(d);
  L.total = L.x32 + round16(T * (d / 32) * 4);
  return L;
}

// grid (d/256, T), 256 threads: thread i owns value i of block b of token t.
__global__ void __launch_bounds__(256) ffn_prep_kernel(const uint16_t* __restrict__ x, int T, int d,
                                                       unsigned char* __restrict__ pkg, int* __restrict__ counters) {
  // x was final before the preceding launch (the router) passed its own wait, and nothing before
  // this kernel touches the package, so the work runs first and the wait (which the kernels
  // after this one rely on) comes last: behind a router that triggers early, it overlaps it.
  // The gate/up launch may start at once: before its own wait it reads only weights.
  pdl_launch_dependents();
  const int b = blockIdx.x, t = blockIdx.y, i = threadIdx.x, lane = i & 31;
  const PkgLayout L = pkg_layout(T, d);
  const uint32_t v = x[(size_t)t * d + 256 * b + i];
  {
    int e;
    const int pos = frag_pos(i, &e);
    const float scaled = __fmul_rn(bf16_bits_to_f32(v), e == 0 ? 1.0f : (e == 1 ? 0.25f : 0.0625f));
    reinterpret_cast<uint16_t*>(pkg + L.xf + (size_t)t * x_stride(d))[b * 256 + pos] =
        (uint16_t)f32_to_bf16_rne(scaled);
  }
  const float f = bf16_bits_to_f32(v);
  // 16-value sub-block sum (lanes of a half warp), fixed tree order
  float s16 = f;
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) s16 += __shfl_xor_sync(0xffffffffu, s16, o);
  // 32-value sum
  const float s32 = s16 + __shfl_xor_sync(0xffffffffu, s16, 16);
  if (lane == 0) reinterpret_cast<float*>(pkg + L.x32)[(size_t)t * (d / 32) + b * 8 + (i >> 5)] = s32;
  if ((i & 15) == 0) {
    const int j = i >> 4;
    const uint32_t hi = f32_to_bf16_rne(s16);
    const float r1 = s16 - bf16_bits_to_f32(hi);
    const uint32_t mid = f32_to_bf16_rne(r1);
    const uint32_t lo = f32_to_bf16_rne(r1 - bf16_bits_to_f32(mid));
    uint16_t* dst = reinterpret_cast<uint16_t*>(pkg + L.xl + (size_t)t * xl_stride(d)) + b * 48;
    dst[limb_pos(j, 0)] = (uint16_t)hi;
    dst[limb_pos(j, 1)] = (uint16_t)mid;
    dst[limb_pos(j, 2)] = (uint16_t)lo;
  }
  pdl_wait();
  // both phases' item counters start from zero (behind the wait every earlier launch, the previous
  // call on this workspace included, has completed)
  if (b == 0 && t == 0 && i < 2) counters[i] = 0;
}

// ----------------------------------------------------------------------------
// the kernel: one producer warp, whose lane w feeds the ring of consumer warp w (it takes items
// from the launch's counter, decodes them, writes a stage descriptor and arms the stage's bulk
// copies), and up to MAX_CONS consumer warps that wait for a stage, multiply and release it.
// The consumers carry no item bookkeeping or copy issue of their own.
// ----------------------------------------------------------------------------
// Stage descriptor, written by the producer lane before it arms the stage:
//   [0] flags (DF_*) | matrix << 4;  [1] routed: first block of the stage, shared: chunk index;
//   [2] routed row group / shared tile;  [3] K part;  [4] columns n;  [5] pair offset;
//   [8 + c] data source of column c (token in phase 1, pair position in phase 2, the token itself
//   for the shared expert); an absent column (c >= n) repeats column 0's (0 when n == 0), whose
//   products land only in outputs that are never stored.
enum { DF_END = 1, DF_SHARED = 2, DF_FIRST = 4, DF_LAST = 8 };

__device__ __forceinline__ void mbar_arrive_plain(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// The lanes of the producer warp (lane w feeds consumer w; lanes < nc take part) step together:
// every round each lane whose consumer has released its next slot fills that slot, so that no
// lane's wait holds up the others; a round in which no lane could act sleeps briefly.
template <int PHASE>
__device__ __forceinline__ void produce(const DecParams& p, int nc, int lane, unsigned char* ring, uint64_t* full,
                                        uint64_t* empty, int* desc, const CUtensorMap* ms0, const CUtensorMap* ms1,
                                        uint64_t* pkg_bar, unsigned char* xprep, int pkg_bytes) {
  constexpr int RT = (PHASE == 1) ? RT1 : RT2;
  const unsigned lanes = nc >= 32 ? 0xffffffffu : ((1u << nc) - 1u);
  const int n_shared_items = p.has_shared ? p.n_mat * p.tiles_s * p.kp_s : 0;
  int seq = 0, cc = 0;
  Item it;
  it.id = -1;
  int src[8];
  // writes the descriptor of stage cc of `it` into slot `slot` and arms the slot's copies
  auto arm = [&](int slot) {
    int* dsc = desc + slot * 16;
    dsc[0] = (it.shared ? DF_SHARED : 0) | (cc == 0 ? DF_FIRST : 0) | (cc + 1 == it.nch ? DF_LAST : 0) | (it.m << 4);
    dsc[1] = it.shared ? it.kp * p.cpp_s + cc : (it.kp * it.nch + cc) * p.bps;
    dsc[2] = it.grp;
    dsc[3] = it.kp;
    dsc[4] = it.n;
    dsc[5] = it.off;
#pragma unroll
    for (int c = 0; c < 8; ++c) dsc[8 + c] = src[c];
    issue_stage<RT>(p, it, cc, ring + slot * STAGE, &full[slot], 0, ms0, ms1);
    if (++cc == it.nch) it.id = -1;
    ++seq;
  };
  // each lane's first item is fixed (CTA-major), the rest come from the launch's counter
  bool first_claim = true;
  if (PHASE == 1) {
    // A first item of the shared expert's needs only weights and shapes, so its first stage is
    // armed before the wait (the packing kernel lets this launch start at once, on the SMs the
    // router leaves); the package, the routing and the counters are read behind the wait.
    const int id0 = (int)blockIdx.x * nc + lane;
    if (id0 < n_shared_items) {
      it = decode_item<PHASE>(p, id0, n_shared_items, 0);
      first_claim = false;
#pragma unroll
      for (int c = 0; c < 8; ++c) src[c] = c < it.n ? c : 0;
      arm(0);
    }
    pdl_wait();
    if (lane == 0) {
      mbar_arrive_expect_tx(pkg_bar, (uint32_t)pkg_bytes);
      bulk_g2s(xprep, p.pkg, (uint32_t)pkg_bytes, pkg_bar);   // x fragments (a multiple of 16 bytes)
    }
  }
  const int n_act = *p.n_active;
  const int per_exp_t = p.n_mat * p.rg_r * p.kp_t;
  const int n_tail = PHASE == 1 ? tail_experts(n_act, per_exp_t, p.tail_items, p.kp_t, p.kp_r) : 0;
  const int a_split = n_act - n_tail;
  const int n_items = n_shared_items + a_split * p.n_mat * p.rg_r * p.kp_r + n_tail * per_exp_t;
  if (PHASE == 1 && blockIdx.x == 0 && lane == 0) {
    // the first pair of the tail's experts (their pairs come last: the active list and the pair
    // order both ascend by expert), for the finishing kernel, which reads it behind its wait
    p.counters[2] = n_tail > 0 ? __ldg(p.offsets + __ldg(p.active + a_split)) : 0x7FFFFFFF;
  }
  const int n_first = (int)gridDim.x * nc;
  bool more = true, done = false;
  long long t_last = clock64();
  bool triggered = false;
  while (true) {
    bool acted = false;
    if (!done) {
      if (it.id < 0 && more) {
        int id = first_claim ? (int)blockIdx.x * nc + lane : n_first + atomicAdd(&p.counters[PHASE - 1], 1);
        first_claim = false;
        if (id >= n_items) {
          id = -1;
          more = false;
        }
        it = decode_item<PHASE>(p, id, n_shared_items, a_split);
        cc = 0;
        if (id >= 0) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const int col = c < it.n ? c : 0;
            int v = 0;
            if (it.n > 0) {
              if (it.shared) v = col;
              else v = (PHASE == 1) ? fdiv(__ldg(p.perm + it.off + col), p.fd_k) : it.off + col;
            }
            src[c] = v;
          }
        }
      }
      const int slot = seq % NS;
      // the slot is free once its consumer has released the stage it held before
      if (mbar_test_wait(&empty[slot], ((seq / NS) & 1) ^ 1)) {
        acted = true;
        t_last = clock64();
        if (it.id < 0) {   // nothing left: an end marker, armed with no bytes
          desc[slot * 16] = DF_END;
          mbar_arrive_plain(&full[slot]);
          done = true;
          ++seq;
        } else {
          arm(slot);
        }
      } else if (clock64() - t_last > p.wait) {
        set_err(p.err, BRE_DEVERR_TIMEOUT);   // the consumer stopped releasing stages
        done = true;
      }
    }
    if (!triggered && !__any_sync(lanes, more)) {
      // every item of this launch has been taken: the next launch (after gate/up the finishing
      // launch and, behind it, the down projection's weight copies; after down whatever reads y,
      // which waits for this grid before it does) may be scheduled on the SMs this launch leaves
      pdl_launch_dependents();
      triggered = true;
    }
    if (__all_sync(lanes, done)) break;
    if (!__any_sync(lanes, acted)) __nanosleep(64);
  }
  // every stage this lane armed has landed before the warp leaves (the last phase of each slot)
  for (int q = seq - NS < 0 ? 0 : seq - NS; q < seq; ++q) mbar_wait_bounded(&full[q % NS], (q / NS) & 1, WAIT_LIMIT);
}

template <int PHASE>
__device__ __forceinline__ void consume(const DecParams& p, int lane, const unsigned char* ring, uint64_t* full,
                                        uint64_t* empty, const int* desc, const unsigned char* xF,
                                        const unsigned char* xLg, const float* X32) {
  constexpr int RT = (PHASE == 1) ? RT1 : RT2;
  const int g = lane >> 2, t = lane & 3;
  const int d = p.d;
  float acc[RT][4];
  uint4 B[8];
  int n = 0, off = 0, grp = 0, kp = 0, m = 0, dg = 0, d0 = 0, d1 = 0;
  bool shared = false;
  const uint16_t* hcol = nullptr;
  for (int seq = 0;; ++seq) {
    const int slot = seq % NS;
    if (!mbar_wait_bounded(&full[slot], (seq / NS) & 1, p.wait)) {
      if (lane == 0) set_err(p.err, BRE_DEVERR_TIMEOUT);
      return;   // the producer lane waits for the copies it armed
    }
    const int* dsc = desc + slot * 16;
    const int fl = dsc[0];
    if (fl & DF_END) return;
    const int c1 = dsc[1];
    if (fl & DF_FIRST) {
      shared = (fl & DF_SHARED) != 0;
      m = fl >> 4;
      grp = dsc[2];
      kp = dsc[3];
      n = dsc[4];
      off = dsc[5];
      dg = dsc[8 + g];
      d0 = dsc[8 + 2 * t];
      d1 = dsc[8 + 2 * t + 1];
#pragma unroll
      for (int r = 0; r < RT; ++r)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[r][i] = 0.0f;
      if (PHASE == 2 && !shared) {
        // the B registers of the item's first block (h of column dg)
        hcol = p.hf + (size_t)dg * (p.F / 256) * 256 + t * 8;
        const uint16_t* h0 = hcol + (size_t)c1 * 256;
#pragma unroll
        for (int q = 0; q < 8; ++q) B[q] = __ldg(reinterpret_cast<const uint4*>(h0) + q * 4);
      }
    }
    const unsigned char* stage = ring + slot * STAGE;
    if (shared) {
      if (PHASE == 1) {
        const uint16_t* xr = p.x + (size_t)dg * d;
        const float* x0 = X32 + d0 * (d / 32);
        const float* x1 = X32 + d1 * (d / 32);
        if (p.cb_s == 8)
          p1_q80_mat<8>(stage, 8, c1, g, t, xr, x0, x1, p.kc.k43, acc[0]);
        else
          p1_q80_mat<0>(stage, p.cb_s, c1, g, t, xr, x0, x1, p.kc.k43, acc[0]);
      } else {
        const uint16_t* hr = p.hS16 + (size_t)dg * p.Fs;
        const float2* q0 = p.HQ + (size_t)d0 * (p.Fs / 32);
        const float2* q1 = p.HQ + (size_t)d1 * (p.Fs / 32);
        if (p.cb_s == 8)
          q80_chunk<8>(stage, 8, c1, g, t, hr, q0, q1, p.kc.k64, acc[0]);
        else
          q80_chunk<0>(stage, p.cb_s, c1, g, t, hr, q0, q1, p.kc.k64, acc[0]);
      }
    } else {
      const int b0 = c1;
      const bool item_last = (fl & DF_LAST) != 0;
      const unsigned char* xb = nullptr;
      const unsigned char* xl = nullptr;
      const uint16_t* hc = nullptr;
      const uint16_t* hl = nullptr;
      if (PHASE == 1) {
        xb = xF + (size_t)dg * p.xstride + t * 16 + b0 * 512;
        xl = xLg + (size_t)dg * p.xlstride + t * 8 + b0 * 96;
      } else {
        hc = hcol + (size_t)b0 * 256;
        hl = p.hl + (size_t)dg * (p.F / 256) * 48 + t * 4 + b0 * 48;
      }
      if (p.bps == 4)
        routed_stage<PHASE, RT, 4>(stage, lane, g, xb, xl, B, hc, hl, item_last, p.kc, acc);
      else if (p.bps == 2)
        routed_stage<PHASE, RT, 2>(stage, lane, g, xb, xl, B, hc, hl, item_last, p.kc, acc);
      else
        routed_stage<PHASE, RT, 1>(stage, lane, g, xb, xl, B, hc, hl, item_last, p.kc, acc);
    }
    // the stage goes back to the producer
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive_plain(&empty[slot]);
    if (!(fl & DF_LAST)) continue;

    // ---- an item ends.  Phase 1 stores its FP32 partial sums of one matrix for the expert's real
    // columns (ffn_finish_kernel adds the K parts in order and forms h); phase 2 stores y (or adds
    // it into zeros when the call splits phase 2 into two K parts).
    if (PHASE == 1) {
      const int tiles = shared ? p.tiles_s : p.rows_r / 16;
      const int KP = shared ? p.kp_s : p.kp_t;   // the partial-sum stride
      float* base = shared ? p.part_s : p.part_r;
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        if (shared && r > 0) break;
        const int tile = shared ? grp : grp * RT + r;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int col = 2 * t + (i & 1), row = g + 8 * (i >> 1);
          if (col < n) {
            const size_t src = shared ? (size_t)col : (size_t)(off + col);   // token / pair position
            base[(((src * tiles + tile) * KP + kp) * 2 + m) * 16 + row] = acc[r][i];
          }
        }
      }
    } else {
#pragma unroll
      for (int r = 0; r < RT; ++r) {
        if (shared && r > 0) break;
        const int row0 = (shared ? grp : grp * RT + r) * 16;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int col = 2 * t + (i & 1);
          if (col < n) {
            const int cs = (i & 1) ? d1 : d0;
            const int row = row0 + g + 8 * (i >> 1);
            float* dst = shared ? p.y_shared + (size_t)cs * p.d + row : p.y_pairs + (size_t)cs * p.d + row;
            if (shared ? p.red_s : p.red_r)
              atomicAdd(dst, acc[r][i]);
            else
              *dst = acc[r][i];
          }
        }
      }
    }
  }
}

template <int PHASE>
__global__ void __launch_bounds__((MAX_CONS + 1) * 32, 1)
    ffn_decode_kernel(const DecParams p, const __grid_constant__ CUtensorMap map_s0,
                      const __grid_constant__ CUtensorMap map_s1) {
  extern __shared__ __align__(128) unsigned char sm[];
  const int nc = (blockDim.x >> 5) - 1;   // consumer warps; warp nc produces
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned char* stages = sm;
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + nc * NS * STAGE);
  uint64_t* empty = full + MAX_CONS * NS;
  uint64_t* pkg_bar = empty + MAX_CONS * NS;
  int* desc = reinterpret_cast<int*>(reinterpret_cast<unsigned char*>(full) + BAR_BYTES);   // [consumer][slot][16]
  unsigned char* xprep = reinterpret_cast<unsigned char*>(desc) + DESC_BYTES;

  // Both phases may be scheduled before their predecessor completes (the packing and finishing
  // launches let them start at once).  Phase 1's producer arms its shared-expert first stages
  // (weights only) before it waits; phase 2's producer reads only the weights, the routing and
  // its item counter, all final before the finishing launch began.  The consumers, which read
  // the package or h, wait.
  if (threadIdx.x < nc * NS) {
    mbar_init(&full[threadIdx.x], 1);
    mbar_init(&empty[threadIdx.x], 1);
  }
  if (threadIdx.x == 0) mbar_init(pkg_bar, 1);
  fence_mbar_init();
  __syncthreads();
  const PkgLayout PL = pkg_layout(p.T, p.d);

  if (warp == nc) {
    if (lane < nc)
      produce<PHASE>(p, nc, lane, stages + lane * NS * STAGE, full + lane * NS, empty + lane * NS,
                     desc + lane * NS * 16, &map_s0, &map_s1, pkg_bar, xprep, PL.smem);
    return;
  }

  // ---- consumers.  Phase 1: the activation package arrives in shared memory by one bulk copy;
  // its limbs and the 32-value sums (read only by the shared expert's items) stay in global memory
  const unsigned char* xF = xprep + PL.xf;                              // [T][xstride], shared memory
  const unsigned char* xLg = p.pkg + PL.xl;                             // [T][xlstride], global memory
  const float* X32 = reinterpret_cast<const float*>(p.pkg + PL.x32);   // [T][d/32]
  pdl_wait();
  if (PHASE == 1 && !mbar_wait_bounded(pkg_bar, 0, p.wait)) {
    if (lane == 0) set_err(p.err, BRE_DEVERR_TIMEOUT);
    mbar_wait_bounded(pkg_bar, 0, WAIT_LIMIT);   // the package copy lands before this warp leaves
    return;
  }
  consume<PHASE>(p, lane, stages + warp * NS * STAGE, full + warp * NS, empty + warp * NS, desc + warp * NS * 16, xF,
                 xLg, X32);
}

// ----------------------------------------------------------------------------
// finish: for every (pair or token, row) add the K-part partial sums of gate and up in order
// 0..KP-1, form h = silu(gate) * up and store it in the layouts phase 2 reads (routed: BF16 of
// h * 4^-e in the fragment order plus three limbs of each 16-row sum of the BF16 h; shared: the
// BF16 h in natural order plus FP32 16-row sums of it).  One warp per 32 rows of one pair/token.  When
// phase 2 adds two K parts into its outputs, the same warps zero those outputs first.
// ----------------------------------------------------------------------------
struct FinishParams {
  const float* part_r;
  const float* part_s;
  int kp_r, kp_s;
  int kp_t;                  // K parts of the tail's experts, and the routed partial-sum stride
  const int* tail_pos;       // first pair of the tail's experts (written by the gate/up launch)
  int F, Fs, P, T, E, d;
  const int32_t* offsets;
  uint16_t* hf;
  uint16_t* hl;
  uint16_t* hS16;
  float2* HQ;
  float* y_pairs;   // zeroed when red_r (valid pairs only)
  float* y_shared;  // zeroed when red_s
  int red_r, red_s;
};

// The launch lets the down projection be scheduled at once: that kernel's producers start the
// weight copies on the SMs this launch and the gate/up launch leave, and its consumers wait for
// this grid.  (Fewer, grid-stride CTAs, which leave more SMs, were measured slower: 64 CTAs
// +1.5 us at T = 8, +99 us on the 24-layer verify pass.)
__global__ void __launch_bounds__(256) ffn_finish_kernel(const FinishParams f) {
  pdl_launch_dependents();
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
  const int KP = shared ? f.kp_s : (src >= __ldg(f.tail_pos) ? f.kp_t : f.kp_r);   // parts to add
  const int KS = shared ? f.kp_s : f.kp_t;                                       // their stride
  if (shared ? f.red_s : f.red_r) {
    float* y = shared ? f.y_shared + (size_t)src * f.d : f.y_pairs + (size_t)src * f.d;
    for (int c = rg * 32 + lane; c < f.d; c += rows) y[c] = 0.0f;
  }
  const int row = rg * 32 + lane, tile = row >> 4, r = row & 15;
  const float* pc = (shared ? f.part_s : f.part_r) + ((size_t)src * (rows / 16) + tile) * KS * 32 + r;
  // every part's load is issued before the sum (up to four at once)
  float gv = 0.0f, uv = 0.0f;
  for (int q0 = 0; q0 < KP; q0 += 4) {
    float vg[4], vu[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      vg[q] = (q0 + q < KP) ? pc[(q0 + q) * 32] : 0.0f;
      vu[q] = (q0 + q < KP) ? pc[(q0 + q) * 32 + 16] : 0.0f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (q0 + q < KP) {
        gv = (q0 + q == 0) ? vg[q] : gv + vg[q];
        uv = (q0 + q == 0) ? vu[q] : uv + vu[q];
      }
    }
  }
  const float h = silu_mul(gv, uv);
  const uint32_t hi = f32_to_bf16_rne(h);   // the down projections read h rounded once to BF16
  float hq = bf16_bits_to_f32(hi);
  if (shared) {
    // the warp's 32 rows are one Q8_0 block of the shared down projection's K: block-scaled FP16
    float bsum, bscale;
    const uint32_t h16 = block_f16(hq, bsum, bscale);
    f.hS16[(size_t)src * f.Fs + row] = (uint16_t)h16;
    if (lane == 0) f.HQ[(size_t)src * (f.Fs / 32) + rg] = make_float2(bsum, bscale);
    return;
  }
  const int Fnb = f.F / 256;
  {
    int e;
    const int pos = frag_pos(row & 255, &e);
    // BF16 of h * 4^-e (the down projection's A fragments keep codes in place); a power of two
    // commutes with the rounding, so the 16-row sums below use h rounded to BF16
    const float hs = __fmul_rn(h, e == 0 ? 1.0f : (e == 1 ? 0.25f : 0.0625f));
    f.hf[((size_t)src * Fnb + (row >> 8)) * 256 + pos] = (uint16_t)f32_to_bf16_rne(hs);
  }
  // 16-row sums of the limb values (half warps)
#pragma unroll
  for (int o = 1; o <= 8; o <<= 1) hq += __shfl_xor_sync(0xffffffffu, hq, o);
  if ((lane & 15) == 0) {
    const int b2 = tile >> 4, j = tile & 15;
    const uint32_t h1 = f32_to_bf16_rne(hq);
    const float r1 = hq - bf16_bits_to_f32(h1);
    const uint32_t h2 = f32_to_bf16_rne(r1);
    const uint32_t h3 = f32_to_bf16_rne(r1 - bf16_bits_to_f32(h2));
    uint16_t* dst = f.hl + ((size_t)src * Fnb + b2) * 48;
    dst[limb_pos(j, 0)] = (uint16_t)h1;
    dst[limb_pos(j, 1)] = (uint16_t)h2;
    dst[limb_pos(j, 2)] = (uint16_t)h3;
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

// Largest of 4 / RT, 2 / RT, 1 blocks that divides a row's block count: routed blocks per stage.
int blocks_per_stage(int nb, int RT) {
  for (int b = 4 / RT; b > 1; b >>= 1)
    if (nb % b == 0) return b;
  return 1;
}

// K parts: the smallest power of two (dividing the row's stage count) that gives the launch at
// least `target` items, given an estimate of the active experts.
int pick_kparts(int stages_per_row, long long items_per_part, long long target) {
  int kp = 1;
  while (kp * 2 <= stages_per_row && stages_per_row % (kp * 2) == 0 && items_per_part * kp < target) kp *= 2;
  return kp;
}

// Distinct experts a batch of T tokens is expected to select (for work splitting only): T = 1
// selects exactly k; otherwise at most T * k, with repeats under a skewed bias.
long long expected_active(int T, int k, int E) {
  const long long tk = (long long)T * k;
  if (T <= 1) return std::min<long long>(tk, E);
  return std::max<long long>(k, std::min<long long>(E, tk * 3 / 4));
}

struct Split {
  int bps, kp_r, cpp_r, kp_t, cpp_t, cb_s, whole_s, C_s, kp_s, cpp_s;
};

// Stage and K-part plan of one phase (the same on every call with the same shapes, so the
// workspace layout follows from T alone).
Split plan_phase(int phase, int T, int k, int E, int nb_r, int rows_r, int nb_s, bool has_shared, int warps_total) {
  Split s{};
  const int RT = phase == 1 ? RT1 : RT2;
  s.bps = blocks_per_stage(nb_r, RT);
  const int stages_row = nb_r / s.bps;
  const int n_mat = phase == 1 ? 2 : 1;
  const long long n_est = expected_active(T, k, E);
  const long long target = 3LL * warps_total;
  if (phase == 1) {
    s.kp_r = pick_kparts(stages_row, n_est * n_mat * (rows_r / (16 * RT)), target);
  } else {
    // phase 2 splits into at most two K parts (added into zeroed outputs, which is order-free)
    s.kp_r = (stages_row % 2 == 0 && n_est * (rows_r / (16 * RT)) < target) ? 2 : 1;
  }
  s.cpp_r = stages_row / s.kp_r;
  // phase 1's tail experts: twice the K parts when the row's stages divide that way
  s.kp_t = (phase == 1 && stages_row % (2 * s.kp_r) == 0) ? 2 * s.kp_r : s.kp_r;
  s.cpp_t = stages_row / s.kp_t;
  s.cb_s = 1;
  s.whole_s = 0;
  s.C_s = 1;
  s.kp_s = 1;
  s.cpp_s = 1;
  if (has_shared) {
    s.cb_s = pick_chunk(nb_s, Q80_BB, STAGE, 8, &s.whole_s);
    s.C_s = s.cb_s > 0 ? nb_s / s.cb_s : 1;
    if (phase == 1) {
      // about as many bytes per shared item as per routed item
      const long long routed_item = (long long)s.cpp_r * STAGE;
      int kp = 1;
      while (kp * 2 <= s.C_s && s.C_s % (kp * 2) == 0 && (long long)(s.C_s / kp) * 16 * s.cb_s * Q80_BB > routed_item)
        kp *= 2;
      s.kp_s = kp;
    } else {
      // a shared tile spans all of K (a routed row group only a few blocks): two K parts keep its
      // items from outlasting the routed work
      s.kp_s = (s.C_s % 2 == 0) ? 2 : 1;
    }
    s.cpp_s = s.C_s / s.kp_s;
  }
  return s;
}

}  // namespace

// Leading bytes of the FFN workspace that hold the decode path's item counters (the packing
// kernel of every decode call clears them behind its wait) and the first pair of the gate/up
// launch's tail experts (written by that launch, read by the finishing launch).
size_t ffn_reserved_bytes(int k, int d, int F, int Fs) {
  (void)k, (void)d, (void)F, (void)Fs;
  return 1024;
}

namespace {

// Workspace of the decode path, in order.
struct DecWs {
  size_t pkg, hf, hl, hS16, HQ, part_r, part_s, total;
};

// A fixed warp count for the split plan (the actual launch may run fewer warps a CTA): keeps the
// workspace layout independent of the device.
constexpr int PLAN_WARPS = 152 * 13;

DecWs dec_ws_layout(int T, int k, int E, int d, int F, int Fs) {
  const size_t P = (size_t)T * k;
  const Split s1 = plan_phase(1, T, k, E, d / 256, F, d / 32, Fs > 0, PLAN_WARPS);
  const size_t pr = P * (F / 16) * s1.kp_t * 2 * 16 * 4;
  const size_t ps = (size_t)T * (Fs / 16) * s1.kp_s * 2 * 16 * 4;
  auto up256 = [](size_t v) { return (v + 255) & ~(size_t)255; };
  DecWs w;
  w.pkg = ffn_reserved_bytes(k, d, F, Fs);
  w.hf = up256(w.pkg + pkg_layout(T, d).total);
  w.hl = up256(w.hf + P * (F / 256) * 256 * 2);
  w.hS16 = up256(w.hl + P * (F / 256) * 48 * 2);
  w.HQ = up256(w.hS16 + (size_t)T * Fs * 2);
  w.part_r = up256(w.HQ + (size_t)T * (Fs / 32) * 8);
  w.part_s = up256(w.part_r + pr);
  w.total = up256(w.part_s + (Fs > 0 ? ps : 0));
  return w;
}

}  // namespace

size_t ffn_ws_bytes(int T, int k, int E, int d, int F, int Fs) {
  // monotone in T: a workspace sized for T also serves every smaller batch (either path)
  size_t m = 0;
  for (int t = 1; t <= std::min(T, DECODE_T_MAX); ++t) m = std::max(m, dec_ws_layout(t, k, E, d, F, Fs).total);
  if (T > DECODE_T_MAX) m = std::max(m, ffn_gemm_ws_bytes(T, k, d, F, Fs));
  return m;
}

bre_status ffn_check_shapes(const bre_ffn_weights* r, const bre_ffn_weights* sh, int T) {
  (void)T;
  const int d = r->d, F = r->d_ff;
  if (d <= 0 || F <= 0 || d % 256 || F % 256) return BRE_ERR_UNSUPPORTED;
  if (sh && (sh->d != d || sh->d_ff <= 0 || sh->d_ff % 256)) return BRE_ERR_UNSUPPORTED;
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
  const DecWs L = dec_ws_layout(a.T, a.k, p.E, p.d, p.F, p.Fs);
  p.counters = reinterpret_cast<int*>(w);
  p.pkg = reinterpret_cast<const unsigned char*>(w + L.pkg);
  unsigned char* pkg_w = reinterpret_cast<unsigned char*>(w + L.pkg);
  p.hf = reinterpret_cast<uint16_t*>(w + L.hf);
  p.hl = reinterpret_cast<uint16_t*>(w + L.hl);
  p.hS16 = reinterpret_cast<uint16_t*>(w + L.hS16);
  p.HQ = reinterpret_cast<float2*>(w + L.HQ);
  p.part_r = reinterpret_cast<float*>(w + L.part_r);
  p.part_s = reinterpret_cast<float*>(w + L.part_s);
  p.xstride = x_stride(p.d);
  p.xlstride = xl_stride(p.d);
  p.kc = DecConst{0x43004300u, 0xC300C300u, 0x46804680u, 0x43434343u, 0x64646464u};
  p.wait = ffn_wait_budget(WAIT_LIMIT);

  const int sms = device_sm_count();
  const int smem_max = device_max_smem_optin();
  {
    const cudaError_t le =
        launch_k(ffn_prep_kernel, dim3(p.d / 256, a.T), dim3(256), 0, s, a.x, a.T, p.d, pkg_w, p.counters);
    if (le != cudaSuccess) return le;
  }
  int kp_r1 = 1, kp_s1 = 1, kp_t1 = 1;
  for (int phase = 1; phase <= 2; ++phase) {
    const int RT = phase == 1 ? RT1 : RT2;
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
      p.n_mat = 2;
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
      p.n_mat = 1;
    }
    const Split sp = plan_phase(phase, a.T, a.k, p.E, p.nb_r, p.rows_r, p.nb_s, S != nullptr, PLAN_WARPS);
    p.bps = sp.bps;
    p.kp_r = sp.kp_r;
    p.cpp_r = sp.cpp_r;
    p.kp_t = sp.kp_t;
    p.cpp_t = sp.cpp_t;
    p.cb_s = sp.cb_s;
    p.whole_s = sp.whole_s;
    p.kp_s = sp.kp_s;
    p.cpp_s = sp.cpp_s;
    if (S && p.cb_s <= 0) return cudaErrorInvalidValue;
    p.rg_r = p.rows_r / (16 * RT);
    p.tiles_s = S ? p.rows_s / 16 : 0;
    p.red_r = (phase == 2 && p.kp_r == 2) ? 1 : 0;
    p.red_s = (phase == 2 && S && p.kp_s == 2) ? 1 : 0;
    if (phase == 2 && (p.kp_r > 2 || p.kp_s > 2)) return cudaErrorInvalidValue;
    p.fd_kps = make_fdiv((unsigned)p.kp_s);
    p.fd_tkps = make_fdiv((unsigned)std::max(1, p.tiles_s * p.kp_s));
    p.fd_kpr = make_fdiv((unsigned)p.kp_r);
    p.fd_rgkpr = make_fdiv((unsigned)(p.rg_r * p.kp_r));
    p.fd_per_exp = make_fdiv((unsigned)(p.n_mat * p.rg_r * p.kp_r));
    p.fd_kpt = make_fdiv((unsigned)p.kp_t);
    p.fd_rgkpt = make_fdiv((unsigned)(p.rg_r * p.kp_t));
    p.fd_per_exp_t = make_fdiv((unsigned)(p.n_mat * p.rg_r * p.kp_t));
    p.fd_k = make_fdiv((unsigned)a.k);
    // tensor maps for the shared expert's chunked rows (unused when whole tiles fit a stage)
    CUtensorMap ms0{}, ms1{};
    if (S && !p.whole_s) {
      if (!weight_map(&ms0, p.sw0, 1, 0, p.rows_s, p.nb_s * Q80_BB, p.cb_s * Q80_BB)) return cudaErrorInvalidValue;
      if (phase == 1 && !weight_map(&ms1, p.sw1, 1, 0, p.rows_s, p.nb_s * Q80_BB, p.cb_s * Q80_BB))
        return cudaErrorInvalidValue;
    }
    const size_t xbytes = (phase == 1) ? (size_t)pkg_layout(a.T, p.d).smem : 0;   // shared-memory part
    int nc = MAX_CONS;
    while (nc > 1 && (size_t)nc * NS * STAGE + BAR_BYTES + DESC_BYTES + xbytes > (size_t)smem_max) --nc;
    const size_t smem = (size_t)nc * NS * STAGE + BAR_BYTES + DESC_BYTES + xbytes;
    if (smem > (size_t)smem_max) return cudaErrorInvalidValue;
    const int nw = nc + 1;   // consumers and the producer warp
    cudaError_t e;
    if (phase == 1) {
      kp_r1 = p.kp_r;
      kp_s1 = p.kp_s;
      kp_t1 = p.kp_t;
      p.tail_items = TAIL_ROUNDS * sms * nc;   // about one item per consumer warp
      e = cudaFuncSetAttribute(ffn_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      e = launch_k(ffn_decode_kernel<1>, dim3(sms), dim3(nw * 32), smem, s, p, ms0, ms1);
      if (e != cudaSuccess) return e;
    } else {
      FinishParams fp;
      fp.part_r = p.part_r;
      fp.part_s = p.part_s;
      fp.kp_r = kp_r1;
      fp.kp_s = kp_s1;
      fp.kp_t = kp_t1;
      fp.tail_pos = p.counters + 2;
      fp.F = p.F;
      fp.Fs = p.Fs;
      fp.P = (int)((size_t)a.T * a.k);
      fp.T = a.T;
      fp.E = p.E;
      fp.d = p.d;
      fp.offsets = a.offsets;
      fp.hf = const_cast<uint16_t*>(p.hf);
      fp.hl = const_cast<uint16_t*>(p.hl);
      fp.hS16 = const_cast<uint16_t*>(p.hS16);
      fp.HQ = const_cast<float2*>(p.HQ);
      fp.y_pairs = p.y_pairs;
      fp.y_shared = p.y_shared;
      fp.red_r = p.red_r;
      fp.red_s = p.red_s;
      const long long warps = (long long)fp.P * (p.F / 32) + (S ? (long long)a.T * (p.Fs / 32) : 0);
      e = launch_k(ffn_finish_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, fp);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(ffn_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      e = launch_k(ffn_decode_kernel<2>, dim3(sms), dim3(nw * 32), smem, s, p, ms0, ms1);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaGetLastError();
}

cudaError_t launch_ffn(const FfnArgs& a, cudaStream_t s) {
  if (a.T <= DECODE_T_MAX) return launch_decode(a, s);
  return launch_gemm(a, s);
}

}  // namespace bre
