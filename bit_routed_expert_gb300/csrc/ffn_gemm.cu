// Expert FFN for prefill-sized batches: a grouped GEMM on the 5th-generation tensor cores.
//
// Strata-DSV4.1 README, "Results" / "How it works" (chunked prefill runs each layer's
// experts once per chunk as grouped expert products) and "Verifying it" (the expert tier
// against a dequantised F32 reference).  Each expert's weight tile is dequantised to
// BF16 (w = d*sc*q - dmin*m exactly in FP32, then rounded to nearest even) straight into
// shared memory and multiplied on tcgen05 with FP32 accumulators in tensor memory.
//
// Per CTA (persistent, one per SM), 16 warps (128 registers a thread):
//   warps 0-3, 12-15  epilogue: tensor memory -> registers -> SwiGLU (gate/up) or FP32 rows
//               (down); warps w and w+12 share tensor-memory lanes 32w .. +31 and take one half
//               of the columns each; warp 0 also allocates tensor memory and its lane 0 issues
//               the MMAs of a tile before the warp turns to that tile's epilogue
//   warps 4-11  B producers: Q2_K / Q8_0 rows -> BF16, 128-byte swizzled K-major tiles, one
//               row per thread per K step; the first producer thread also issues the TMA 2-D
//               loads of the gathered activations (128-byte swizzle) for each stage
// Tile: M = 256 tokens (two 128-row accumulators), N = 256 weight rows, K step = 64.
// Phase 1: the 256 rows are 128 gate rows + the same 128 up rows, so the epilogue forms
// h = silu(g) * u for 128 columns of the intermediate.  Phase 2: 256 down rows.
#include <cuda.h>

#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

namespace {

constexpr int G_STAGES = 3;
constexpr int G_BM = 256, G_BN = 256, G_BK = 64;
constexpr int G_A_BYTES = G_BM * G_BK * 2;   // 32 KB
constexpr int G_B_BYTES = G_BN * G_BK * 2;   // 32 KB
constexpr int G_THREADS = 512;
constexpr int G_PRODUCERS = 256;   // B-producer threads (warps 4-11)
constexpr int G_MAX_GROUPS = 1025;
constexpr int R16_BYTES = 1344;   // one Q2_K_R16 tile: 16 rows x one 256-weight block
constexpr long long G_WAIT = 4000000000LL;   // cycles before a wait gives up (~2 s)

// plan: per group g (routed active experts in order, then the shared expert):
//   a_row0 (first A row), n (rows), expert (-1 shared), tile0 phase 1, tile0 phase 2
struct Plan {
  int n_groups;
  int tiles1, tiles2;
  int pad;
  int a_row0[G_MAX_GROUPS];
  int n[G_MAX_GROUPS];
  int expert[G_MAX_GROUPS];
  int tile1[G_MAX_GROUPS + 1];
  int tile2[G_MAX_GROUPS + 1];
};

__global__ void plan_kernel(const int32_t* __restrict__ offsets, const int32_t* __restrict__ active,
                            const int32_t* __restrict__ n_active, int has_shared, int T, int P, int nt1_r, int nt1_s,
                            int nt2, int E, int32_t* err, Plan* plan) {
  pdl_wait();
  if (threadIdx.x != 0) return;
  const int na = min(*n_active, G_MAX_GROUPS - 1);
  int g = 0, t1 = 0, t2 = 0;
  for (int a = 0; a < na; ++a) {
    const int e = active[a];
    if ((unsigned)e >= (unsigned)E) {   // an expert the weights do not hold: its pairs stay zero
      set_err(err, BRE_DEVERR_EXPERT_ID);
      continue;
    }
    const int off = offsets[e], n = offsets[e + 1] - off;
    const int mt = (n + G_BM - 1) / G_BM;
    plan->a_row0[g] = off;
    plan->n[g] = n;
    plan->expert[g] = e;
    plan->tile1[g] = t1;
    plan->tile2[g] = t2;
    t1 += mt * nt1_r;
    t2 += mt * nt2;
    ++g;
  }
  if (has_shared) {
    const int mt = (T + G_BM - 1) / G_BM;
    plan->a_row0[g] = P;
    plan->n[g] = T;
    plan->expert[g] = -1;
    plan->tile1[g] = t1;
    plan->tile2[g] = t2;
    t1 += mt * nt1_s;
    t2 += mt * nt2;
    ++g;
  }
  plan->tile1[g] = t1;
  plan->tile2[g] = t2;
  plan->n_groups = g;
  plan->tiles1 = t1;
  plan->tiles2 = t2;
}

// X_perm[q] = x[perm[q] / k] for valid pairs q < offsets[E]; X_perm[P + t] = x[t].  One warp per
// row, eight 16-byte loads in flight per lane before their stores.
__global__ void gather_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm,
                              const int32_t* __restrict__ offsets, int E, int k, int T, int P, int d,
                              uint16_t* __restrict__ xp, int has_shared) {
  pdl_wait();
  const int per_row = d / 8;
  const int nvalid = __ldg(offsets + E);
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  for (int q = blockIdx.x * wpb + (threadIdx.x >> 5); q < P + T; q += gridDim.x * wpb) {
    int src = -1;
    if (q < nvalid)
      src = __ldg(perm + q) / k;
    else if (q >= P && has_shared)
      src = q - P;
    if (src < 0) continue;
    const uint4* in = reinterpret_cast<const uint4*>(x + (size_t)src * d);
    uint4* out = reinterpret_cast<uint4*>(xp + (size_t)q * d);
    for (int c0 = 0; c0 < per_row; c0 += 8 * 32) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < per_row) v[u] = __ldg(in + c);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < per_row) out[c] = v[u];
      }
    }
  }
}

// ---------------------------------------------------------------------------
// tcgen05 / TMA wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mma_f16_ss(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 32 consecutive FP32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------
// B producers: one weight row, one K step (64 values) -> 8 swizzled 16-byte chunks
// ---------------------------------------------------------------------------
// One row's quarter (64 values, sub-blocks 4kq .. 4kq+3) of a Q2_K_R16 block: the scale and
// min nibble words of the lane that holds these sub-blocks (shifted so that sub-block
// 4kq + 2p + h sits at bit 16h + 4p), d | dmin << 16, and the codes in the Q2_K order (word jj:
// the 16 codes of sub-block 4kq + jj, code c at bits 2c).
struct RawQ2K {
  uint32_t s, m, dd, q[4];
};

// A whole Q2_K_R16 block of one row as the producers hold it (25 words): the codes of the row's
// four lanes (words 4kq .. 4kq+3: lane 4g + kq's words W(p, w) at 2p + w), the lanes' scale and
// min words (2kq, 2kq + 1 at 16 + ...), and d | dmin << 16.  The producers hold the next block
// while dequantising the current one, so the load has four K steps to land.
struct RawBlk {
  uint32_t c[16];
  uint32_t sm[8];
  uint32_t dd;
};

// The quarter kq of a held block of row 8 rr + g.
__device__ __forceinline__ RawQ2K quarter(const RawBlk& b, int kq, int rr) {
  RawQ2K r;
  r.s = b.sm[2 * kq] >> (8 * rr);
  r.m = b.sm[2 * kq + 1] >> (8 * rr);
  r.dd = b.dd;
#pragma unroll
  for (int pp = 0; pp < 2; ++pp) {
    // W(p, 0) holds codes 0..7 and W(p, 1) codes 8..15 of sub-blocks 4kq + 2p (low halves) and
    // 4kq + 2p + 1 (high halves)
    const uint32_t w0 = b.c[4 * kq + 2 * pp], w1 = b.c[4 * kq + 2 * pp + 1];
    r.q[2 * pp] = prmt(w0, w1, 0x5410u);
    r.q[2 * pp + 1] = prmt(w0, w1, 0x7632u);
  }
  return r;
}

// 4-entry BF16 table of one sub-block: value of code q is bf16_rne((d*sc)*q - dmin*m).
__device__ __forceinline__ void q2k_lut(float d, float dmin, uint32_t sc, uint32_t m, uint32_t& lo, uint32_t& hi) {
  const float dsc = __fmul_rn(d, (float)sc);
  const float dmm = __fmul_rn(dmin, (float)m);
  const float w0 = -dmm;
  const float w1 = __fsub_rn(dsc, dmm);
  const float w2 = __fmaf_rn(2.0f, dsc, -dmm);   // 2*dsc is exact: one rounding
  const float w3 = __fmaf_rn(3.0f, dsc, -dmm);   // 3*dsc is exact: one rounding
  lo = pack_bf16x2(w0, w1);
  hi = pack_bf16x2(w2, w3);
}

__device__ __forceinline__ void store_q2k_row(const RawQ2K& r, unsigned char* b_stage, int row) {
  const float d = f16_bits_to_f32(r.dd & 0xFFFFu), dmin = f16_bits_to_f32(r.dd >> 16);
  unsigned char* rowp = b_stage + (row >> 3) * 1024 + (row & 7) * 128;
  const int sw = row & 7;
#pragma unroll
  for (int jj = 0; jj < 4; ++jj) {
    const int sh = 16 * (jj & 1) + 4 * (jj >> 1);
    uint32_t lo, hi;
    q2k_lut(d, dmin, (r.s >> sh) & 15u, (r.m >> sh) & 15u, lo, hi);
    const uint32_t w = r.q[jj];
    const uint32_t c0 = w & 0x03030303u, c1 = (w >> 2) & 0x03030303u;
    const uint32_t c2 = (w >> 4) & 0x03030303u, c3 = (w >> 6) & 0x03030303u;
    uint32_t o[8];
#pragma unroll
    for (int B = 0; B < 4; ++B) {
      const uint32_t u01 = prmt(c0, c1, (uint32_t)(B | ((4 + B) << 4)));
      const uint32_t u23 = prmt(c2, c3, (uint32_t)(B | ((4 + B) << 4)));
      o[2 * B] = prmt(lo, hi, u01 * 0x22u + 0x1010u);
      o[2 * B + 1] = prmt(lo, hi, u23 * 0x22u + 0x1010u);
    }
    // codes 16jj .. 16jj+7 -> chunk 2jj, 16jj+8 .. +15 -> chunk 2jj+1
    *reinterpret_cast<uint4*>(rowp + (((2 * jj) ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<uint4*>(rowp + (((2 * jj + 1) ^ sw) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

struct RawQ80 {
  uint32_t w[17];   // two 34-byte blocks (68 bytes, 4-byte aligned)
};


__device__ __forceinline__ uint32_t byte_at(const RawQ80& r, int b) {  // byte b of the 68
  return (r.w[b >> 2] >> (8 * (b & 3))) & 0xFFu;
}

__device__ __forceinline__ void store_q80_row(const RawQ80& r, unsigned char* b_stage, int row) {
  unsigned char* rowp = b_stage + (row >> 3) * 1024 + (row & 7) * 128;
  const int sw = row & 7;
#pragma unroll
  for (int blk = 0; blk < 2; ++blk) {
    const int base = blk * Q80_BB;
    const float d = f16_bits_to_f32(byte_at(r, base) | (byte_at(r, base + 1) << 8));
#pragma unroll
    for (int ch = 0; ch < 4; ++ch) {
      uint32_t o[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int i0 = ch * 8 + 2 * p;
        const float a = __fmul_rn(d, (float)(int8_t)byte_at(r, base + 2 + i0));
        const float b = __fmul_rn(d, (float)(int8_t)byte_at(r, base + 3 + i0));
        o[p] = pack_bf16x2(a, b);
      }
      const int chunk = blk * 4 + ch;
      *reinterpret_cast<uint4*>(rowp + ((chunk ^ sw) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

// silu(g) * u with the hardware exponential and a fast divide (relative error ~1e-6, far below
// the BF16 rounding of h that follows; for g below about -88 the quotient is 0)
__device__ __forceinline__ float silu_mul(float gv, float uv) { return __fdividef(gv, 1.0f + __expf(-gv)) * uv; }

// Within each group of four lanes (rows 4q .. 4q+3 of the warp's 32 accumulator rows), a 4 x 4
// transpose of NW-word blocks: lane 4q+p enters with the four blocks of its own row (block b =
// v[b*NW .. b*NW+NW-1], columns b*NW ..) and leaves with block p of row 4q+k in slot k.  Two
// exchange rounds (lane ^ 2, then lane ^ 1), each moving half of the words.  Four lanes then
// write one row's consecutive columns, so a store instruction touches 8 rows, not 32.
template <int NW, typename V>
__device__ __forceinline__ void quad_transpose(V (&v)[4 * NW], int lane) {
  const bool hi = (lane & 2) != 0;
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      V& lo_s = v[j * NW + w];
      V& hi_s = v[(2 + j) * NW + w];
      const V recv = __shfl_xor_sync(0xffffffffu, hi ? lo_s : hi_s, 2);
      if (hi) lo_s = recv; else hi_s = recv;
    }
  const bool pl = (lane & 1) != 0;
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      V& s0 = v[(2 * a) * NW + w];
      V& s1 = v[(2 * a + 1) * NW + w];
      const V recv = __shfl_xor_sync(0xffffffffu, pl ? s0 : s1, 1);
      if (pl) s0 = recv; else s1 = recv;
    }
}

__device__ __forceinline__ void st_v8(float* dst, const float* v) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "f"(v[0]), "f"(v[1]),
               "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

struct GemmParams {
  const Plan* plan;
  // routed (Q2_K) and shared (Q8_0) weights of this phase: m0 = gate / down, m1 = up
  const uint8_t* r0;
  const uint8_t* r1;
  long long rs0, rs1;
  const uint8_t* s0;
  const uint8_t* s1;
  int K_r, K_s;          // contraction length (routed, shared)
  int rows_r, rows_s;    // output rows of the weight matrices
  int nt_r, nt_s;        // N tiles per M tile
  uint16_t* h_r;         // phase 1 outputs [P][F], [T][Fs]
  uint16_t* h_s;
  float* y_r;            // phase 2 outputs [P][d], [T][d]
  float* y_s;
  int out_ld_r, out_ld_s;
  int out_v8;            // phase 2 outputs 32-byte aligned: 32-byte stores
  int32_t* err;
  long long wait;        // budget (cycles) of the pipeline's waits; the drains at exit use G_WAIT
};

struct TileInfo {
  int g, mt, nt, a_row0, n, expert, K;
};

template <int PHASE>
__device__ __forceinline__ TileInfo find_tile(const GemmParams& p, int tile) {
  const Plan* pl = p.plan;
  const int* t0 = (PHASE == 1) ? pl->tile1 : pl->tile2;
  int lo = 0, hi = pl->n_groups - 1;
  while (lo < hi) {   // last group with t0[g] <= tile
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(t0 + mid) <= tile) lo = mid; else hi = mid - 1;
  }
  TileInfo ti;
  ti.g = lo;
  ti.expert = __ldg(pl->expert + lo);
  const int ntn = (ti.expert < 0) ? p.nt_s : p.nt_r;
  const int r = tile - __ldg(t0 + lo);
  ti.mt = r / ntn;
  ti.nt = r % ntn;
  ti.a_row0 = __ldg(pl->a_row0 + lo);
  ti.n = __ldg(pl->n + lo);
  ti.K = (ti.expert < 0) ? p.K_s : p.K_r;
  return ti;
}

template <int PHASE>
__global__ void __launch_bounds__(G_THREADS, 1)
    ffn_gemm_kernel(const __grid_constant__ CUtensorMap map_r, const __grid_constant__ CUtensorMap map_s,
                    const GemmParams p) {
  extern __shared__ __align__(1024) unsigned char gsm_raw[];
  // 1024-byte alignment for the swizzled tiles
  unsigned char* gsm = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(gsm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char* a_st = gsm;                                   // [G_STAGES][32 KB]
  unsigned char* b_st = gsm + G_STAGES * G_A_BYTES;            // [G_STAGES][32 KB]
  uint64_t* full = reinterpret_cast<uint64_t*>(b_st + G_STAGES * G_B_BYTES);   // B rows stored (producers)
  uint64_t* empty = full + G_STAGES;
  uint64_t* tfull = empty + G_STAGES;
  uint64_t* tempty = tfull + 1;
  uint64_t* aful = tempty + 1;             // A tile landed (the TMA alone completes it)
  uint64_t* drain = aful + G_STAGES;       // every MMA issued so far has completed
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_holder + 1);
  unsigned char* stage_raw = reinterpret_cast<unsigned char*>(full) + 256;   // [8 warps][32 rows][84 B]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  if (threadIdx.x == 0) {
    for (int s = 0; s < G_STAGES; ++s) {
      mbar_init(&full[s], G_PRODUCERS);
      mbar_init(&aful[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 256);
    mbar_init(drain, 1);
    *abort_flag = 0;
  }
  fence_mbar_init();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(tmem_holder))
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int n_tiles = (PHASE == 1) ? p.plan->tiles1 : p.plan->tiles2;
  auto fail = [&]() {
    set_err(p.err, BRE_DEVERR_TIMEOUT);
    atomicExch(abort_flag, 1);
  };
  auto aborted = [&]() { return *reinterpret_cast<volatile int*>(abort_flag) != 0; };

  if (warp >= 4 && warp < 12) {
    // ---------------- B producers (dequantise into swizzled shared memory); thread i owns row i
    // of the B tile.  The first producer thread also loads the A tile of every stage it opens.
    const int i = threadIdx.x - 128;
    const bool a_loader = (i == 0);
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles && !aborted(); tile += gridDim.x) {
      const TileInfo ti = find_tile<PHASE>(p, tile);
      const int KS = ti.K / G_BK;
      const CUtensorMap* amap = (ti.expert < 0) ? &map_s : &map_r;
      const int arow = (PHASE == 1) ? ti.a_row0 + ti.mt * G_BM : (ti.expert < 0 ? 0 : ti.a_row0) + ti.mt * G_BM;
      // wait until stage s is free, then (first thread) start its A tile
      auto open_stage = [&](int s, int ks) -> bool {
        if (!mbar_wait_bounded(&empty[s], ((it / G_STAGES) & 1) ^ 1, p.wait)) {
          fail();
          return false;
        }
        if (a_loader) {
          mbar_arrive_expect_tx(&aful[s], G_A_BYTES);
          tma_load_2d(a_st + s * G_A_BYTES, amap, ks * G_BK, arow, &aful[s]);
          tma_load_2d(a_st + s * G_A_BYTES + G_A_BYTES / 2, amap, ks * G_BK, arow + 128, &aful[s]);
        }
        return true;
      };
      const int pw = warp - 4;
      unsigned char* stg = stage_raw + pw * 32 * Q2K_BB;
      if (ti.expert >= 0) {
        // Q2_K_R16: the warp's 32 rows are two 16-row tiles; each block of them is two
        // 1344-byte tiles, copied whole into the warp's staging area by 16-byte cp.async
        // (84 pieces a tile), then each thread takes its row's words
        const int nb = p.K_r / 256;
        const uint8_t* mat;
        int r_mat;   // this thread's row within its matrix
        if (PHASE == 1) {
          mat = (i < 128) ? p.r0 + (long long)ti.expert * p.rs0 : p.r1 + (long long)ti.expert * p.rs1;
          r_mat = ti.nt * 128 + (i & 127);
        } else {
          mat = p.r0 + (long long)ti.expert * p.rs0;
          r_mat = ti.nt * 256 + i;
        }
        const long long rt0 = (r_mat - lane) >> 4;   // the warp's first row tile
        const int tau = lane >> 4, R = lane & 15, g8 = R & 7, rr = R >> 3;
        const int NBK = KS / 4;
        auto stage_copy = [&](int blk) {
#pragma unroll
          for (int c = lane; c < 2 * (R16_BYTES / 16); c += 32) {
            const int tt = c >= R16_BYTES / 16 ? 1 : 0;
            const int off = (c - tt * (R16_BYTES / 16)) * 16;
            cp_async16(stg + tt * R16_BYTES + off, mat + ((rt0 + tt) * nb + blk) * R16_BYTES + off, 16);
          }
          cp_async_commit();
        };
        auto stage_read = [&](RawBlk& a) {
          cp_async_wait<0>();
          __syncwarp();
          const unsigned char* u = stg + tau * R16_BYTES;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint4 cw = *reinterpret_cast<const uint4*>(u + rr * 512 + 64 * g8 + 16 * v);
            a.c[4 * v] = cw.x;
            a.c[4 * v + 1] = cw.y;
            a.c[4 * v + 2] = cw.z;
            a.c[4 * v + 3] = cw.w;
          }
#pragma unroll
          for (int v = 0; v < 2; ++v) {
            const uint4 sw4 = *reinterpret_cast<const uint4*>(u + 1024 + 32 * g8 + 16 * v);
            a.sm[4 * v] = sw4.x;
            a.sm[4 * v + 1] = sw4.y;
            a.sm[4 * v + 2] = sw4.z;
            a.sm[4 * v + 3] = sw4.w;
          }
          a.dd = *reinterpret_cast<const uint32_t*>(u + 1280 + 8 * g8 + 4 * rr);
          __syncwarp();
        };
        RawBlk ca;
        stage_copy(0);
        bool ok = true;
        for (int bk = 0; bk < NBK && ok; ++bk) {
          stage_read(ca);
          if (bk + 1 < NBK) stage_copy(bk + 1);
#pragma unroll
          for (int kq = 0; kq < 4; ++kq, ++it) {
            const int s = it % G_STAGES;
            if (!open_stage(s, bk * 4 + kq)) {
              ok = false;
              break;
            }
            store_q2k_row(quarter(ca, kq, rr), b_st + s * G_B_BYTES, i);
            fence_proxy_async_smem();
            mbar_arrive(&full[s]);
          }
        }
        cp_async_wait<0>();   // no copy stays in flight past the tile
      } else {
        const int rb = (p.K_s / 32) * Q80_BB;
        const uint8_t* row;
        if (PHASE == 1)
          row = (i < 128) ? p.s0 + (long long)(ti.nt * 128 + i) * rb : p.s1 + (long long)(ti.nt * 128 + i - 128) * rb;
        else
          row = p.s0 + (long long)(ti.nt * 256 + i) * rb;
        // The two Q8_0 blocks (68 bytes) of each row for a K step reach the warp's staging area
        // by coalesced copies (lanes 0..16 copy one row's 17 words per instruction); the copy of
        // the next K step runs while this one is dequantised.
        const uint8_t* pr0 = row - (long long)lane * rb + 4 * lane;
        auto stage_copy = [&](int ks) {
          if (lane < 17) {
            const uint8_t* pr = pr0 + ks * 2 * Q80_BB;
            unsigned char* dst = stg + 4 * lane;
#pragma unroll 8
            for (int r = 0; r < 32; ++r) cp_async4(dst + r * 68, pr + (long long)r * rb, 4);
          }
          cp_async_commit();
        };
        auto stage_read = [&](RawQ80& a) {
          cp_async_wait<0>();
          __syncwarp();
#pragma unroll
          for (int w = 0; w < 17; ++w) a.w[w] = *reinterpret_cast<const uint32_t*>(stg + lane * 68 + 4 * w);
          __syncwarp();
        };
        RawQ80 ca;
        stage_copy(0);
        for (int ks = 0; ks < KS; ++ks, ++it) {
          stage_read(ca);
          if (ks + 1 < KS) stage_copy(ks + 1);
          const int s = it % G_STAGES;
          if (!open_stage(s, ks)) break;
          store_q80_row(ca, b_st + s * G_B_BYTES, i);
          fence_proxy_async_smem();
          mbar_arrive(&full[s]);
        }
        cp_async_wait<0>();   // no copy stays in flight past the tile
      }
    }
    // the A tiles this thread started have landed before the CTA can exit (after an abort the
    // MMA thread may not have consumed the last ones): the last phase armed on each stage
    if (a_loader) {
      for (int q = it - G_STAGES < 0 ? 0 : it - G_STAGES; q < it; ++q)
        mbar_wait_bounded(&aful[q % G_STAGES], (q / G_STAGES) & 1, G_WAIT);
    }
  } else {
    // ---------------- MMA issue (warp 0, lane 0) and epilogue (warps 0-3 and 12-15: tensor-memory
    // lanes 32*(warp & 3) .. +31, column half warp >= 12)
    // kind::f16, D = F32, A = B = BF16, both K-major, M = 128, N = 256
    const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(G_BN >> 3) << 17) |
                           ((uint32_t)(128 >> 4) << 24);
    int it = 0, tcount = 0;
    for (int tile = blockIdx.x; tile < n_tiles && !aborted(); tile += gridDim.x, ++tcount) {
      const TileInfo ti = find_tile<PHASE>(p, tile);
      if (warp == 0 && lane == 0) {
        const int KS = ti.K / G_BK;
        // the previous tile's epilogue has drained the accumulators
        if (!mbar_wait_bounded(tempty, (tcount & 1) ^ 1, p.wait)) {
          fail();
        } else {
          tc_fence_after();
          for (int ks = 0; ks < KS; ++ks, ++it) {
            const int s = it % G_STAGES;
            if (!mbar_wait_bounded(&full[s], (it / G_STAGES) & 1, p.wait) ||
                !mbar_wait_bounded(&aful[s], (it / G_STAGES) & 1, p.wait)) {
              fail();
              break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(a_st + s * G_A_BYTES);
            const uint32_t b0 = smem_u32(b_st + s * G_B_BYTES);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int kk = 0; kk < G_BK / 16; ++kk) {
                const uint64_t ad = smem_desc_sw128(a0 + h * (G_A_BYTES / 2) + kk * 32);
                const uint64_t bd = smem_desc_sw128(b0 + kk * 32);
                mma_f16_ss(tmem + h * 256, ad, bd, idesc, (ks > 0 || kk > 0) ? 1u : 0u);
              }
            mma_commit(&empty[s]);
          }
          mma_commit(tfull);
        }
      }
      __syncwarp();
      if (!mbar_wait_bounded(tfull, tcount & 1, p.wait)) { fail(); break; }
      tc_fence_after();
      if (aborted()) break;   // the accumulators may hold a partial sum: nothing is stored
      const int q4 = lane >> 2, p4 = lane & 3;
      const int eq = warp & 3, part = warp >> 3;   // lane quarter, column half
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        // after the quad transpose this lane writes rows 4*q4 + k (k = 0..3) of the warp's 32
        const int mrow0 = ti.mt * G_BM + h * 128 + eq * 32 + 4 * q4;   // row within the group
        const uint32_t tbase = tmem + ((uint32_t)(eq * 32) << 16) + h * 256;
        if (PHASE == 1) {
          uint16_t* out0 = (ti.expert < 0) ? p.h_s + (size_t)mrow0 * p.out_ld_s
                                           : p.h_r + (size_t)(ti.a_row0 + mrow0) * p.out_ld_r;
          const int ld = (ti.expert < 0) ? p.out_ld_s : p.out_ld_r;
#pragma unroll 1
          for (int c = part * 64; c < part * 64 + 64; c += 32) {
            float gv[32], uv[32];
            tmem_ld32(tbase + c, gv);
            tmem_ld32(tbase + 128 + c, uv);
            uint32_t o[16];
#pragma unroll
            for (int q = 0; q < 16; ++q)
              o[q] = pack_bf16x2(silu_mul(gv[2 * q], uv[2 * q]), silu_mul(gv[2 * q + 1], uv[2 * q + 1]));
            quad_transpose<4>(o, lane);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (mrow0 + k < ti.n)
                *reinterpret_cast<uint4*>(out0 + (size_t)k * ld + ti.nt * 128 + c + 8 * p4) =
                    make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
          }
        } else {
          float* out0 = (ti.expert < 0) ? p.y_s + (size_t)mrow0 * p.out_ld_s
                                        : p.y_r + (size_t)(ti.a_row0 + mrow0) * p.out_ld_r;
          const int ld = (ti.expert < 0) ? p.out_ld_s : p.out_ld_r;
#pragma unroll 1
          for (int c = part * 128; c < part * 128 + 128; c += 32) {
            float v[32];
            tmem_ld32(tbase + c, v);
            quad_transpose<8>(v, lane);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (mrow0 + k < ti.n) {
                float* dst = out0 + (size_t)k * ld + ti.nt * 256 + c + 8 * p4;
                if (p.out_v8) {
                  st_v8(dst, v + 8 * k);
                } else {
                  reinterpret_cast<float4*>(dst)[0] = make_float4(v[8 * k], v[8 * k + 1], v[8 * k + 2], v[8 * k + 3]);
                  reinterpret_cast<float4*>(dst)[1] =
                      make_float4(v[8 * k + 4], v[8 * k + 5], v[8 * k + 6], v[8 * k + 7]);
                }
              }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty);
    }
    // every MMA this CTA issued has completed before its tensor memory is freed
    if (warp == 0 && lane == 0) {
      mma_commit(drain);
      mbar_wait_bounded(drain, 0, G_WAIT);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem) : "memory");
  }
}

// 2-D BF16 tensor [rows][K], box 64 x 128, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, long long rows, int K) {
  const uint64_t dims[2] = {(uint64_t)K, (uint64_t)(rows > 0 ? rows : 1)};
  const uint64_t strides[1] = {(uint64_t)K * 2};
  const uint32_t box[2] = {64, 128};
  return encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

size_t ffn_gemm_ws_bytes(int T, int k, int d, int F, int Fs) {
  const size_t P = (size_t)T * k;
  // the reserved prefix stays with the decode path's item counters (each decode call clears them)
  size_t s = ffn_reserved_bytes(k, d, F, Fs) + ((sizeof(Plan) + 1023) & ~(size_t)1023);
  s += ((P + T) * d * 2 + 1023) & ~(size_t)1023;     // gathered activations
  s += (P * F * 2 + 1023) & ~(size_t)1023;           // routed intermediate
  s += ((size_t)T * Fs * 2 + 1023) & ~(size_t)1023;  // shared intermediate
  return s;
}

cudaError_t launch_gemm(const FfnArgs& a, cudaStream_t s) {
  const bre_ffn_weights* R = a.routed;
  const bre_ffn_weights* S = a.shared;
  const int T = a.T, k = a.k, d = R->d, F = R->d_ff, Fs = S ? S->d_ff : 0, E = R->n_experts;
  const size_t P = (size_t)T * k;
  char* w = static_cast<char*>(a.ws) + ffn_reserved_bytes(k, d, F, Fs);
  Plan* plan = reinterpret_cast<Plan*>(w);
  w += (sizeof(Plan) + 1023) & ~(size_t)1023;
  uint16_t* xp = reinterpret_cast<uint16_t*>(w);
  w += ((P + T) * d * 2 + 1023) & ~(size_t)1023;
  uint16_t* h_r = reinterpret_cast<uint16_t*>(w);
  w += (P * F * 2 + 1023) & ~(size_t)1023;
  uint16_t* h_s = reinterpret_cast<uint16_t*>(w);

  {
    const cudaError_t le = launch_k(plan_kernel, dim3(1), dim3(32), 0, s, a.offsets, a.active, a.n_active,
                                    S ? 1 : 0, T, (int)P, F / 128, Fs / 128, d / 256, E, a.err, plan);
    if (le != cudaSuccess) return le;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  {
    const cudaError_t le = launch_k(gather_kernel, dim3(sms * 4), dim3(256), 0, s, a.x, a.perm, a.offsets, E, k, T,
                                    (int)P, d, xp, S ? 1 : 0);
    if (le != cudaSuccess) return le;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  const size_t smem = G_STAGES * (G_A_BYTES + G_B_BYTES) + 1024 + 256 + 8 * 32 * Q2K_BB;
  static int configured = -1;
  int dev;
  cudaGetDevice(&dev);
  if (configured != dev) {
    if ((e = cudaFuncSetAttribute(ffn_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    if ((e = cudaFuncSetAttribute(ffn_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) !=
        cudaSuccess)
      return e;
    configured = dev;
  }
  CUtensorMap m_x, m_hr, m_hs;
  if (!make_map(&m_x, xp, (long long)(P + T), d)) return cudaErrorInvalidValue;
  if (!make_map(&m_hr, h_r, (long long)P, F)) return cudaErrorInvalidValue;
  if (!make_map(&m_hs, S ? (const void*)h_s : (const void*)h_r, S ? T : (long long)P, S ? Fs : F))
    return cudaErrorInvalidValue;

  GemmParams g{};
  g.wait = ffn_wait_budget(G_WAIT);
  g.plan = plan;
  g.err = a.err;
  // phase 1: gate/up -> h
  g.r0 = static_cast<const uint8_t*>(R->gate);
  g.r1 = static_cast<const uint8_t*>(R->up);
  g.rs0 = R->expert_stride_gate;
  g.rs1 = R->expert_stride_up;
  g.s0 = S ? static_cast<const uint8_t*>(S->gate) : nullptr;
  g.s1 = S ? static_cast<const uint8_t*>(S->up) : nullptr;
  g.K_r = d;
  g.K_s = d;
  g.rows_r = F;
  g.rows_s = Fs;
  g.nt_r = F / 128;
  g.nt_s = Fs / 128;
  g.h_r = h_r;
  g.h_s = h_s;
  g.out_ld_r = F;
  g.out_ld_s = Fs;
  {
    const cudaError_t le = launch_k(ffn_gemm_kernel<1>, dim3(sms), dim3(G_THREADS), smem, s, m_x, m_x, g);
    if (le != cudaSuccess) return le;
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // phase 2: down -> y
  g.r0 = static_cast<const uint8_t*>(R->down);
  g.r1 = nullptr;
  g.rs0 = R->expert_stride_down;
  g.rs1 = 0;
  g.s0 = S ? static_cast<const uint8_t*>(S->down) : nullptr;
  g.s1 = nullptr;
  g.K_r = F;
  g.K_s = Fs;
  g.rows_r = d;
  g.rows_s = d;
  g.nt_r = d / 256;
  g.nt_s = d / 256;
  g.y_r = a.y_pairs;
  g.y_s = a.y_shared;
  g.out_ld_r = d;
  g.out_ld_s = d;
  g.out_v8 = ((reinterpret_cast<uintptr_t>(a.y_pairs) | reinterpret_cast<uintptr_t>(a.y_shared)) & 31) == 0 &&
             (d % 8) == 0;
  {
    const cudaError_t le = launch_k(ffn_gemm_kernel<2>, dim3(sms), dim3(G_THREADS), smem, s, m_hr, m_hs, g);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace bre
