// Router (score, selection-only bias, top-k, renormalised weights) and the stable
// expert permutation.
//
// Strata-DSV4.1 README, "Results": the route bias changes which experts are
// selected, while the mixing weights stay exact.  vllm.cpp PR (DeepSeek-V4-Flash-
// Vision), device router notes: top-k on the biased score, weights gathered from
// the unbiased scores, one warp per row.  strix-llama.cpp issue, "Stack progress":
// request-union planning (each selected expert runs once for all its tokens).
//
// The logit of (t, e) is accumulated in a fixed order so that it is reproducible
// bit for bit: 32 partial sums, partial j takes fmaf over rows c = j, j+32, ... in
// ascending order starting from +0, then a butterfly p_j + p_(j^o) for
// o = 16, 8, 4, 2, 1.  Any thread mapping computes exactly this.
#include <algorithm>
#include <mutex>

#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

namespace {

constexpr int SMALL_TT = 8;      // tokens per token group, small-batch logits
constexpr int TILE_T = 32;       // tokens per CTA, tiled logits
constexpr int TILE_E = 32;       // experts per CTA, tiled logits
constexpr int SMALL_T_MAX = 32;  // up to this many tokens use the small-batch kernel

// s = 1 / (1 + exp(-z)) in float, every step one IEEE operation so that any conforming
// machine gets the same bits: Cody-Waite range reduction n = rint(x log2 e), r = x - n ln2
// (ln 2 split in two float parts, the first with few enough bits that n * LN2_HI is exact),
// exp(r) by its degree-7 Taylor polynomial in Horner form, scaled by 2^n.  x = -z is clamped
// below at -30 (there 1 + exp(x) == 1 in float); x > 88 gives 0.
__device__ __forceinline__ float sigmoid_ref(float z) {
  const float LOG2E = 1.44269504088896341f;
  const float LN2_HI = 0.693359375f;
  const float LN2_LO = -2.12194440054690583e-4f;
  float x = -z;
  if (isnan(x)) return x;
  if (x > 88.0f) return 0.0f;
  x = fmaxf(x, -30.0f);
  const float n = rintf(__fmul_rn(x, LOG2E));
  float r = __fmaf_rn(-n, LN2_HI, x);
  r = __fmaf_rn(-n, LN2_LO, r);
  float p = 1.0f / 5040.0f;
  p = __fmaf_rn(p, r, 1.0f / 720.0f);
  p = __fmaf_rn(p, r, 1.0f / 120.0f);
  p = __fmaf_rn(p, r, 1.0f / 24.0f);
  p = __fmaf_rn(p, r, 1.0f / 6.0f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  // p * 2^n with n in [-44, 128): exact scaling (two steps so that 2^n itself never overflows)
  const int ni = (int)n;
  const int n1 = ni / 2, n2 = ni - n1;
  const float e = __fmul_rn(__fmul_rn(p, __int_as_float((127 + n1) << 23)), __int_as_float((127 + n2) << 23));
  return __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
}

// exp(x) for -87 <= x <= 0 with the same steps as sigmoid_ref (n >= -126: 2^n is a normal
// number and the scaling is exact).
__device__ __forceinline__ float exp_neg_ref(float x) {
  const float LOG2E = 1.44269504088896341f;
  const float LN2_HI = 0.693359375f;
  const float LN2_LO = -2.12194440054690583e-4f;
  const float n = rintf(__fmul_rn(x, LOG2E));
  float r = __fmaf_rn(-n, LN2_HI, x);
  r = __fmaf_rn(-n, LN2_LO, r);
  float p = 1.0f / 5040.0f;
  p = __fmaf_rn(p, r, 1.0f / 720.0f);
  p = __fmaf_rn(p, r, 1.0f / 120.0f);
  p = __fmaf_rn(p, r, 1.0f / 24.0f);
  p = __fmaf_rn(p, r, 1.0f / 6.0f);
  p = __fmaf_rn(p, r, 0.5f);
  p = __fmaf_rn(p, r, 1.0f);
  p = __fmaf_rn(p, r, 1.0f);
  return __fmul_rn(p, __int_as_float((127 + (int)n) << 23));
}

// s = sqrt(softplus(z)) in float (the vllm.cpp device router notes' SqrtSoftplusRouteTopk
// score): softplus(z) = max(z, 0) + log1p(exp(-|z|)), exp(-|z|) as above (0 for |z| > 87),
// log1p(e) = 2 atanh(u), u = e / (2 + e) <= 1/3, as 2u (1 + v/3 + ... + v^7/15), v = u^2, in
// Horner form; every step one IEEE operation, so any conforming machine gets the same bits.
__device__ __forceinline__ float sqrt_softplus_ref(float z) {
  if (isnan(z)) return z;
  const float a = fabsf(z);
  const float e = a > 87.0f ? 0.0f : exp_neg_ref(-a);
  const float u = __fdiv_rn(e, __fadd_rn(2.0f, e));
  const float v = __fmul_rn(u, u);
  float q = 1.0f / 15.0f;
  q = __fmaf_rn(q, v, 1.0f / 13.0f);
  q = __fmaf_rn(q, v, 1.0f / 11.0f);
  q = __fmaf_rn(q, v, 1.0f / 9.0f);
  q = __fmaf_rn(q, v, 1.0f / 7.0f);
  q = __fmaf_rn(q, v, 1.0f / 5.0f);
  q = __fmaf_rn(q, v, 1.0f / 3.0f);
  q = __fmaf_rn(q, v, 1.0f);
  const float l = __fmul_rn(2.0f, __fmul_rn(u, q));
  return __fsqrt_rn(__fadd_rn(z > 0.0f ? z : 0.0f, l));
}

__device__ __forceinline__ float score_ref(float z, int fn) { return fn == 1 ? sqrt_softplus_ref(z) : sigmoid_ref(z); }

// The per-row rule of the device router notes (SqrtSoftplusRouteTopk): row t is media when a
// vision bias and a media mask are given and media[t] != 0; a media row's key is s + vbias and
// it selects the top k; a text row's key is s + bias, and on a hash layer (tid2eid given) its
// ids are tid2eid[tok[t]][0..k) instead.  Weights come from the unbiased s.  A token id outside
// [0, vocab) sets BRE_DEVERR_ROW_ID (ids -1, weights 0); a table id outside [0, E) sets
// BRE_DEVERR_EXPERT_ID, is passed on, and counts s = 0.
struct RouteVar {
  int score;               // 0 sigmoid, 1 sqrt(softplus)
  const float* vbias;      // [E] or null
  const uint8_t* media;    // [T] or null
  const int32_t* tid2eid;  // [vocab][k] or null
  const int32_t* tok;      // [T]
  int vocab;
  float* hash_s;           // [T][k] scratch (small-batch kernel): s of each hash row's table ids
  int32_t* err;            // error word or null
};

__device__ __forceinline__ bool row_media(const RouteVar& rv, int t) {
  return rv.vbias != nullptr && rv.media != nullptr && rv.media[t] != 0;
}

// Does (ka, ia) rank before (kb, ib)?  Larger key first, then lower id; NaN last.
__device__ __forceinline__ bool ranks_before(float ka, int ia, float kb, int ib) {
  const bool na = isnan(ka), nb = isnan(kb);
  if (na != nb) return !na;
  if (!na && ka != kb) return ka > kb;
  return ia < ib;
}

// One warp writes a hash row's ids (tid2eid[tok[t]] in table order) and weights (its unbiased
// scores, S in slot order).  s_src: the row's E scores (from_slots = false) or its k table
// scores in slot order (from_slots = true, the small-batch kernel's hash_s).
__device__ void hash_row(const float* __restrict__ s_src, int E, int k, const RouteVar& rv, int t,
                         int32_t* __restrict__ ids_t, float* __restrict__ w_t, bool from_slots) {
  const int lane = threadIdx.x & 31;
  const int tk = __ldg(rv.tok + t);
  if (tk < 0 || tk >= rv.vocab) {
    if (lane < k) {
      ids_t[lane] = -1;
      w_t[lane] = 0.0f;
    }
    if (lane == 0 && rv.err) atomicOr(rv.err, BRE_DEVERR_ROW_ID);
    return;
  }
  int id = 0;
  float sj = 0.0f;
  bool bad = false;
  if (lane < k) {
    id = __ldg(rv.tid2eid + (size_t)tk * k + lane);
    bad = id < 0 || id >= E;
    if (!bad) sj = from_slots ? __ldcg(s_src + lane) : __ldcg(s_src + id);
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && rv.err) atomicOr(rv.err, BRE_DEVERR_EXPERT_ID);
  float S = 0.0f;
  for (int j = 0; j < k; ++j) {
    const float v = __shfl_sync(0xffffffffu, sj, j);
    S = (j == 0) ? v : __fadd_rn(S, v);
  }
  if (lane < k) {
    ids_t[lane] = id;
    w_t[lane] = __fdiv_rn(sj, S);
  }
}

// One warp selects the top k of the E scores of one token and writes ids and weights; lane l
// holds scores l, l+32, ... (NI >= ceil(E/32) of them, a compile-time count).
template <int NI>
__device__ void topk_warp(const float* __restrict__ s_row, const float* __restrict__ bias, int E, int k,
                          int32_t* __restrict__ ids_out, float* __restrict__ w_out) {
  const int lane = threadIdx.x & 31;
  float sv[NI];
  // selection code of each candidate, ordered as the selection order (larger key first, NaN
  // last, -0 equal to +0; ties go to the lower id): finite and infinite keys map monotonically
  // to codes >= 0x007FFFFF, NaN to 1, a slot past E to 0 (never selected)
  uint32_t kc[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    sv[i] = 0.0f;
    kc[i] = 0u;
    if (e < E) {
      sv[i] = __ldcg(s_row + e);
      const float key = __fadd_rn(__fadd_rn(sv[i], bias ? __ldg(bias + e) : 0.0f), 0.0f);   // -0 -> +0
      const uint32_t b = __float_as_uint(key);
      kc[i] = isnan(key) ? 1u : ((b & 0x80000000u) ? ~b : (b | 0x80000000u));
    }
  }
  uint32_t used = 0;
  float my_sel_s = 0.0f;
  int my_sel_id = 0;
  for (int j = 0; j < k; ++j) {
    // lane-local best (the first of equal codes is the lowest id), then the warp's: the largest
    // code, and among the lanes holding it the lowest id
    uint32_t bc = 0u;
    int bi = -1;
    float bs = 0.0f;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (!((used >> i) & 1u) && kc[i] > bc) {
        bc = kc[i];
        bi = i;
        bs = sv[i];
      }
    const uint32_t wc = __reduce_max_sync(0xffffffffu, bc);
    const uint32_t wid = __reduce_min_sync(0xffffffffu, (bi >= 0 && bc == wc) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu);
    const int owner = (int)(wid & 31u);
    const float ws = __shfl_sync(0xffffffffu, bs, owner);
    if (lane == owner) used |= 1u << (wid >> 5);
    if (lane == j) {
      my_sel_s = ws;
      my_sel_id = (int)wid;
    }
  }
  float S = 0.0f;
  for (int j = 0; j < k; ++j) {
    const float sj = __shfl_sync(0xffffffffu, my_sel_s, j);
    S = (j == 0) ? sj : __fadd_rn(S, sj);
  }
  if (lane < k) {
    ids_out[lane] = my_sel_id;
    w_out[lane] = __fdiv_rn(my_sel_s, S);
  }
}

// Small batches (decode): one warp per (partial j, block of 32 experts), lane = expert.  A
// CTA holds four consecutive j; the eight CTAs that hold j = 0..31 of one expert block form
// a cluster and add their partials in the butterfly order through distributed shared memory.
// The CTA's W_r slice (rows c = j (mod 32) of its 32 experts) is copied to shared memory
// with cp.async (coalesced 128-byte rows, all in flight at once, issued before the wait on
// the producing kernel: W_r is a weight); x is staged once as FP32 in [j][i][token] order.
// Every loop stays rolled: each SM runs this code once, so its size, not its arithmetic,
// would set the time.  Each cluster then selects a local top k of its 32 experts per token;
// the CTA that makes the last delivery (one ticket for all tokens) merges every token's block
// lists (the global top k of a token is contained in the union of the per-block top k) and,
// for moe_route_permute, builds the permutation from the ids it holds.
constexpr int RC_J = 4;                   // partials (warps) per CTA
constexpr int RC_CLUSTER = 32 / RC_J;     // CTAs per cluster
constexpr int RC_THREADS = RC_J * 32;

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
  uint32_t a = (uint32_t)__cvta_generic_to_shared(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// Selection order as an unsigned code: (code, id) ascending = key descending, then id ascending,
// NaN keys last (an exact restatement of ranks_before for keys that are never -0; -0 is mapped
// to +0).
__device__ __forceinline__ uint32_t key_code(float k) {
  if (isnan(k)) return 0xFFFFFFFFu;
  uint32_t u = __float_as_uint(k);
  if ((u << 1) == 0u) u = 0u;                                   // -0 -> +0
  const uint32_t asc = (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // float order as unsigned order
  return ~asc;
}
__device__ __forceinline__ bool code_before(uint32_t ca, int ia, uint32_t cb, int ib) {
  return ca < cb || (ca == cb && ia < ib);
}

// Candidates of one token: kc slots per expert block, (code, s, id), sorted by rank within the
// block; id = -1 for an empty slot (a block with fewer than kc experts).
__host__ __device__ __forceinline__ int rc_slots(int E, int k) { return ((E + 31) / 32) * (k < 32 ? k : 32); }

// Outputs of the permutation when the router kernel also permutes (offsets == nullptr: it does not).
struct PermOut {
  int32_t* offsets;
  int32_t* perm;
  int32_t* inv;
  int32_t* active;
  int32_t* n_active;
};
constexpr long long RC_WAIT_LIMIT = 2000000000LL;   // cycles (~1 s) before the W wait gives up

// A group of W lanes (W = 32, or 16: two tokens per warp) merges the candidate lists of one
// token: list b (lane b of the group, b < nblk <= W) holds the block's top kc in rank order, so
// the token's top k are k rounds of "take the best list head".  Writes ids / weights (weights
// from the unbiased s, S summed in slot order) and keeps the ids in ids_s for the permutation.
// lane is the lane inside the group; every lane of the warp calls it (W = 16: each half-warp
// with its own token, or with active = false for a half that has none).
template <int W>
__device__ __forceinline__ void merge_token(const uint32_t* mc, const int* mid, const float* ms, int nblk, int kc,
                                            int k, int lane, bool active, int32_t* __restrict__ ids_t,
                                            float* __restrict__ w_t, int* ids_s) {
  int h = 0;
  uint32_t hc = 0xFFFFFFFFu;
  int hid = 0x7FFFFFFF;
  float hs = 0.0f;
  auto load_head = [&]() {
    hc = 0xFFFFFFFFu;
    hid = 0x7FFFFFFF;
    if (active && lane < nblk && h < kc) {
      const int id = mid[lane * kc + h];
      if (id >= 0) {
        hc = mc[lane * kc + h];
        hid = id;
        hs = ms[lane * kc + h];
      }
    }
  };
  load_head();
  float my_s = 0.0f;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    uint32_t bc = hc;
    int bid = hid;
#pragma unroll
    for (int o = W / 2; o >= 1; o >>= 1) {
      const uint32_t oc = __shfl_xor_sync(0xffffffffu, bc, o, W);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, o, W);
      if (code_before(oc, oid, bc, bid)) {
        bc = oc;
        bid = oid;
      }
    }
    // ids are distinct across lists, so exactly one lane of the group holds the winner
    const bool mine = hid == bid && hid != 0x7FFFFFFF;
    const unsigned gm = __ballot_sync(0xffffffffu, mine) >> ((threadIdx.x & 31) & ~(W - 1) & 31);
    const unsigned wmask = W == 32 ? gm : (gm & 0xFFFFu);
    const float ws = __shfl_sync(0xffffffffu, hs, wmask ? __ffs(wmask) - 1 : 0, W);
    if (lane == j) {
      my_s = ws;
      my_id = bid;
    }
    if (mine) {
      ++h;
      load_head();
    }
  }
  float S = 0.0f;
  for (int j = 0; j < k; ++j) {
    const float sj = __shfl_sync(0xffffffffu, my_s, j, W);
    S = (j == 0) ? sj : __fadd_rn(S, sj);
  }
  if (active && lane < k) {
    ids_t[lane] = my_id;
    w_t[lane] = __fdiv_rn(my_s, S);
    ids_s[lane] = my_id;
  }
}

// The W_r slice of a CTA arrives by one tensor copy when W_r allows (E % 4 == 0, d / 32 <= 256,
// 16-byte aligned): a map over W_r viewed as [d/32][32][E] (innermost E) with box
// {32 experts, RC_J rows j, d/32 groups} lands as [i][jj][e], the layout the FMA loop reads.
struct RouteMap {
  CUtensorMap map;
  int use;
};

__global__ void __cluster_dims__(1, RC_CLUSTER, 1) __launch_bounds__(RC_THREADS)
    route_cluster_kernel(const uint16_t* __restrict__ x, const float* __restrict__ w_r,
                         const float* __restrict__ bias, int T, int d, int E, int k, uint32_t* __restrict__ cand_c,
                         float* __restrict__ cand_s, int* __restrict__ cand_id, int* tickets,
                         int32_t* __restrict__ ids, float* __restrict__ wts, const PermOut po, int merge_group,
                         int32_t* err, const __grid_constant__ RouteMap wm, const RouteVar rv) {
  extern __shared__ __align__(128) float rc_smem[];
  __shared__ float part[SMALL_TT][RC_J][33];     // partial sums of this CTA's j, padded
  __shared__ __align__(8) uint64_t wbar;
  __shared__ int s_last;
  __shared__ int s_scan[2][RC_J];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n = d / 32;
  float* Ws = rc_smem;                           // [n][RC_J][32]
  float* xs = rc_smem + (size_t)n * RC_J * 32;   // [RC_J][n][SMALL_TT]
  const int e = blockIdx.x * 32 + lane;
  const int jb = blockIdx.y;                     // j block = rank in the cluster
  const int j = jb * RC_J + warp;
  const int t0 = blockIdx.z * SMALL_TT;
  const int nt = min(SMALL_TT, T - t0);
  const int kc = min(k, 32);
  const int slots = rc_slots(E, k);
  if (wm.use) {
    if (tid == 0) {
      mbar_init(&wbar, 1);
      fence_mbar_init();
      mbar_arrive_expect_tx(&wbar, (uint32_t)(n * RC_J * 32 * 4));
      tma_load_3d(Ws, &wm.map, blockIdx.x * 32, jb * RC_J, 0, &wbar);
    }
  } else if ((E & 3) == 0) {
    // 16-byte pieces: slice row (i, jj) is 8 pieces of W_r row 32 i + RC_J jb + jj; thread tid
    // copies piece tid % 8 of jj = (tid / 8) % 4 for i = tid / 32, +4, +8, ...
    const int pc = tid & 7, jj = (tid >> 3) & 3, i0 = tid >> 5;
    const int ee = blockIdx.x * 32 + pc * 4;
    const bool ok = ee < E;
    const float* src = w_r + (size_t)(32 * i0 + jb * RC_J + jj) * E + (ok ? ee : 0);
    float* dst = Ws + (size_t)(i0 * RC_J + jj) * 32 + pc * 4;
    const size_t sstep = (size_t)128 * E;
#pragma unroll 4
    for (int i = i0; i < n; i += 4, src += sstep, dst += 4 * RC_J * 32) cp_async16(dst, src, ok ? 16 : 0);
  } else {
    const float* src = w_r + (size_t)j * E + (e < E ? e : 0);
    const size_t rstride = (size_t)32 * E;
    float* dst = Ws + warp * 32 + lane;
    for (int i = 0; i < n; ++i) cp_async4(dst + (size_t)i * RC_J * 32, src + i * rstride, e < E ? 4 : 0);
  }
  pdl_wait();
  // the next launch may start now: every kernel that follows waits for this grid before it uses
  // anything this grid writes (the decode FFN's prep reads only x, which the wait above covers)
  pdl_launch_dependents();
  // stage x: item q = (i, tt) reads the RC_J values x[t0+tt][32 i + RC_J jb ...] (8 bytes); a
  // thread's loads (eight at a time) are all issued before their stores, so their latencies
  // overlap instead of adding up
  for (int q0 = 0; q0 < n * SMALL_TT; q0 += 8 * RC_THREADS) {
    uint2 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + u * RC_THREADS + tid;
      const int tt = q & (SMALL_TT - 1), i = q / SMALL_TT;
      v[u] = make_uint2(0u, 0u);
      if (q < n * SMALL_TT && tt < nt)
        v[u] = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t0 + tt) * d + 32 * i + RC_J * jb));
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int q = q0 + u * RC_THREADS + tid;
      if (q < n * SMALL_TT) {
        const int tt = q & (SMALL_TT - 1), i = q / SMALL_TT;
        xs[(0 * n + i) * SMALL_TT + tt] = bf16_bits_to_f32(v[u].x & 0xFFFFu);
        xs[(1 * n + i) * SMALL_TT + tt] = bf16_bits_to_f32(v[u].x >> 16);
        xs[(2 * n + i) * SMALL_TT + tt] = bf16_bits_to_f32(v[u].y & 0xFFFFu);
        xs[(3 * n + i) * SMALL_TT + tt] = bf16_bits_to_f32(v[u].y >> 16);
      }
    }
  }
  if (!wm.use) cp_async_wait_all();
  __syncthreads();   // x staged; the slice barrier's initialisation is visible to every thread
  if (wm.use) {
    // bounded: on a timeout the error word is set and the CTA carries on (it must still reach
    // the cluster barriers its peers wait on)
    if (!mbar_wait_bounded(&wbar, 0, RC_WAIT_LIMIT) && err && tid == 0) atomicOr(err, BRE_DEVERR_TIMEOUT);
  }
  // partial j of expert e: rows c = j + 32 i in ascending i, fmaf from +0; the operands of eight
  // rows are loaded before their FMAs (one warp per scheduler: the loads' latency is not hidden
  // by other warps)
  float acc[SMALL_TT];
#pragma unroll
  for (int tt = 0; tt < SMALL_TT; ++tt) acc[tt] = 0.0f;
  const float4* xw = reinterpret_cast<const float4*>(xs + (size_t)warp * n * SMALL_TT);
  const float* wp = Ws + warp * 32 + lane;
  auto fma_row = [&](float wgt, float4 a, float4 b) {
    acc[0] = fmaf(a.x, wgt, acc[0]);
    acc[1] = fmaf(a.y, wgt, acc[1]);
    acc[2] = fmaf(a.z, wgt, acc[2]);
    acc[3] = fmaf(a.w, wgt, acc[3]);
    acc[4] = fmaf(b.x, wgt, acc[4]);
    acc[5] = fmaf(b.y, wgt, acc[5]);
    acc[6] = fmaf(b.z, wgt, acc[6]);
    acc[7] = fmaf(b.w, wgt, acc[7]);
  };
  int i = 0;
  for (; i + 8 <= n; i += 8) {
    float wv[8];
    float4 xa[8], xb[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      wv[u] = wp[(size_t)(i + u) * RC_J * 32];
      xa[u] = xw[2 * (i + u)];
      xb[u] = xw[2 * (i + u) + 1];
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) fma_row(wv[u], xa[u], xb[u]);
  }
  for (; i < n; ++i) fma_row(wp[(size_t)i * RC_J * 32], xw[2 * i], xw[2 * i + 1]);
#pragma unroll
  for (int tt = 0; tt < SMALL_TT; ++tt) part[tt][warp][lane] = acc[tt];
  cluster_sync_all();
  // CTA of rank r adds the 32 partials of token t0 + r for the 32 experts of the block, then
  // writes the block's top kc of that token in rank order (rank = number of the block's experts
  // that come first).  One ticket counts the deliveries of all tokens; the CTA that makes the
  // last one merges every token and, when asked, permutes.
  const uint32_t r = cluster_ctarank();
  if (warp == 0 && (int)r < nt) {
    float v[32];
#pragma unroll
    for (int b = 0; b < RC_CLUSTER; ++b)
#pragma unroll
      for (int w = 0; w < RC_J; ++w) v[b * RC_J + w] = ld_cluster_f32(&part[r][w][lane], (uint32_t)b);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
      for (int q = 0; q < o; ++q) v[q] = __fadd_rn(v[q], v[q + o]);
    const bool valid = e < E;
    const int t = t0 + (int)r;
    const bool media = row_media(rv, t);
    const float* rb = media ? rv.vbias : bias;
    const float sv = valid ? score_ref(v[0], rv.score) : 0.0f;
    const float key = __fadd_rn(sv, (rb && valid) ? __ldg(rb + e) : 0.0f);
    if (rv.tid2eid != nullptr && !media) {
      // a hash row: the expert's score goes to every slot of the row's table that names it
      const int tk = __ldg(rv.tok + t);
      if (valid && tk >= 0 && tk < rv.vocab)
        for (int q = 0; q < k; ++q)
          if (__ldg(rv.tid2eid + (size_t)tk * k + q) == e) rv.hash_s[(size_t)t * k + q] = sv;
    }
    const uint32_t code = valid ? key_code(key) : 0xFFFFFFFFu;   // absent experts: last (id >= E)
    int rank = 0;
#pragma unroll 8
    for (int src = 0; src < 32; ++src) {
      const uint32_t c2 = __shfl_sync(0xffffffffu, code, src);
      rank += (src != lane && code_before(c2, blockIdx.x * 32 + src, code, e)) ? 1 : 0;
    }
    const size_t cbase = (size_t)(t0 + r) * slots + (size_t)blockIdx.x * kc;
    if (rank < kc) {
      cand_c[cbase + rank] = code;
      cand_s[cbase + rank] = sv;
      cand_id[cbase + rank] = valid ? e : -1;
    }
    // the warp barrier orders the lanes' candidate stores before lane 0's release
    __syncwarp();
    if (lane == 0) {
      int prev;
      asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(tickets) : "memory");
      const int last = prev == (int)gridDim.x * T - 1;
      if (last) tickets[0] = 0;   // every delivery is counted: ready for the next call
      s_last = last;
    }
  } else if (tid == 0) {
    s_last = 0;
  }
  cluster_sync_all();  // no CTA leaves while another reads its partials; s_last is visible
  if (!s_last) return;
  // ---- the last CTA: merge every token (one warp per token, token groups that fit the shared
  // memory), then the permutation from the ids kept in shared memory
  const int nblk = (E + 31) / 32;
  const int P = T * k;
  int* ids_s = reinterpret_cast<int*>(rc_smem);   // [T * k]
  int* cnt = ids_s + P;                            // [E + 1], then run [E + 1] (permutation)
  int* run = cnt + (E + 1);
  uint32_t* mc = reinterpret_cast<uint32_t*>(run + (E + 1));   // [merge_group * slots] x 3
  int* mid = reinterpret_cast<int*>(mc + (size_t)merge_group * slots);
  float* ms = reinterpret_cast<float*>(mid + (size_t)merge_group * slots);
  for (int g0 = 0; g0 < T; g0 += merge_group) {
    const int ng = min(merge_group, T - g0);
    // the acquire of the last ticket precedes this barrier-ordered read of every delivery; a
    // thread's loads (eight slots at a time) are issued before their stores
    for (int c0 = 0; c0 < ng * slots; c0 += 8 * RC_THREADS) {
      uint32_t vc[8];
      int vi[8];
      float vs[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * RC_THREADS + tid;
        if (c < ng * slots) {
          const size_t gi = (size_t)g0 * slots + c;
          vc[u] = __ldcg(cand_c + gi);
          vi[u] = __ldcg(cand_id + gi);
          vs[u] = __ldcg(cand_s + gi);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int c = c0 + u * RC_THREADS + tid;
        if (c < ng * slots) {
          mc[c] = vc[u];
          mid[c] = vi[u];
          ms[c] = vs[u];
        }
      }
    }
    __syncthreads();
    // hash rows (text rows of a hash layer) take their table instead of a merge
    auto hash_t = [&](int t) { return rv.tid2eid != nullptr && !row_media(rv, t); };
    if (nblk <= 16 && k <= 16) {
      // two tokens per warp, one per half-warp
      for (int p0 = 2 * warp; p0 < ng; p0 += 2 * RC_J) {
        const int tt = p0 + (lane >> 4);
        const bool act = tt < ng;
        const int ts = act ? tt : p0;
        const int t = g0 + ts;
        merge_token<16>(mc + (size_t)ts * slots, mid + (size_t)ts * slots, ms + (size_t)ts * slots, nblk, kc, k,
                        lane & 15, act && !hash_t(t), ids + (size_t)t * k, wts + (size_t)t * k,
                        ids_s + (size_t)t * k);
      }
    } else {
      for (int tt = warp; tt < ng; tt += RC_J) {
        const int t = g0 + tt;
        merge_token<32>(mc + (size_t)tt * slots, mid + (size_t)tt * slots, ms + (size_t)tt * slots, nblk, kc, k,
                        lane, !hash_t(t), ids + (size_t)t * k, wts + (size_t)t * k, ids_s + (size_t)t * k);
      }
    }
    if (rv.tid2eid != nullptr)
      for (int tt = warp; tt < ng; tt += RC_J) {
        const int t = g0 + tt;
        if (hash_t(t)) hash_row(rv.hash_s + (size_t)t * k, E, k, rv, t, ids + (size_t)t * k, wts + (size_t)t * k, true);
      }
    __syncthreads();
  }
  if (po.offsets == nullptr) return;
  // stable counting sort of the T * k pairs by expert id (ids are in [0, E) by construction)
  for (int q = tid; q <= E; q += RC_THREADS) {
    cnt[q] = 0;
    run[q] = 0;
  }
  __syncthreads();
  for (int q = tid; q < P; q += RC_THREADS) atomicAdd(&cnt[ids_s[q]], 1);
  __syncthreads();
  // exclusive scan of the counts (and of the active flags): thread i takes experts
  // [i * per, (i + 1) * per)
  const int per = (E + RC_THREADS - 1) / RC_THREADS, a0 = min(E, tid * per), a1 = min(E, a0 + per);
  int sum = 0, nact = 0;
  for (int q = a0; q < a1; ++q) {
    sum += cnt[q];
    nact += cnt[q] > 0 ? 1 : 0;
  }
  int ps = sum, pa = nact;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ys = __shfl_up_sync(0xffffffffu, ps, o), ya = __shfl_up_sync(0xffffffffu, pa, o);
    if (lane >= o) {
      ps += ys;
      pa += ya;
    }
  }
  if (lane == 31) {
    s_scan[0][warp] = ps;
    s_scan[1][warp] = pa;
  }
  __syncthreads();
  int ws0 = 0, wa0 = 0, tot_s = 0, tot_a = 0;
#pragma unroll
  for (int w = 0; w < RC_J; ++w) {
    if (w < warp) {
      ws0 += s_scan[0][w];
      wa0 += s_scan[1][w];
    }
    tot_s += s_scan[0][w];
    tot_a += s_scan[1][w];
  }
  int base = ws0 + ps - sum, abase = wa0 + pa - nact;
  for (int q = a0; q < a1; ++q) {
    const int c = cnt[q];
    po.offsets[q] = base;
    cnt[q] = base;
    if (c > 0) po.active[abase++] = q;
    base += c;
  }
  if (tid == 0) {
    po.offsets[E] = tot_s;
    *po.n_active = tot_a;
  }
  for (int q = tot_a + tid; q < E; q += RC_THREADS) po.active[q] = -1;
  __syncthreads();
  if (warp != 0) return;
  // pairs in chunks of 32, in order; rank among equal ids from a warp match
  const unsigned lt = (1u << lane) - 1u;
  for (int c0 = 0; c0 < P; c0 += 32) {
    const int q = c0 + lane;
    const int key = q < P ? ids_s[q] : E;
    const unsigned m = __match_any_sync(0xffffffffu, key);
    const int lr = __popc(m & lt);
    if (q < P) {
      const int pos = cnt[key] + run[key] + lr;
      po.perm[pos] = q;
      po.inv[q] = pos;
    }
    __syncwarp();
    if (q < P && lr == 0) run[key] += __popc(m);
    __syncwarp();
  }
}

// Large batches: CTA = TILE_T tokens x TILE_E experts, 16 warps.  Lane = partial j; warp q
// owns tokens 8*(q/4) .. +8 and experts 8*(q%4) .. +8 of the tile.  Rows arrive TR at a time
// through a TSTAGES-deep cp.async ring: W_r rows as FP32 (padded to 36 words so that the 32
// lanes' 16-byte loads of 32 different rows spread over the banks), x as the raw BF16 tile
// [token][row], which lane j reads at row c0 + j (consecutive lanes, consecutive addresses)
// and widens in registers.  One barrier per stage.  (Measured on GB300: an 8-token x 16-expert
// tile per thread with 8 warps, and widening x once per stage into a transposed FP32 tile, were
// both slower than this.)
constexpr int TR = 512;
constexpr int TSTAGES = 2;
constexpr int TTHREADS = 512;
constexpr int TW = TILE_E + 4;   // padded W row (words)
constexpr size_t TILED_SMEM = (size_t)TSTAGES * (TR * TW * 4 + TILE_T * TR * 2);


__global__ void __launch_bounds__(TTHREADS, 1) route_tiled_kernel(const uint16_t* __restrict__ x,
                                                                  const float* __restrict__ w_r, int T, int d,
                                                                  int E, float* __restrict__ S, int score_fn) {
  extern __shared__ __align__(16) unsigned char tsm[];
  float* Wst = reinterpret_cast<float*>(tsm);                                          // [TSTAGES][TR][TW]
  uint16_t* Xst = reinterpret_cast<uint16_t*>(tsm + (size_t)TSTAGES * TR * TW * 4);    // [TSTAGES][TILE_T][TR]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * TILE_T, e0 = blockIdx.y * TILE_E;
  const int tsub = (warp >> 2) * 8, esub = (warp & 3) * 8;
  const int nst = (d + TR - 1) / TR;
  // accumulators of experts (2q, 2q+1) in one 64-bit register pair: fma.rn.f32x2 performs the two
  // IEEE fmaf of each row in one instruction (the same bits as two fmaf)
  unsigned long long acc2[8][4];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int q = 0; q < 4; ++q) acc2[a][q] = 0ull;
  auto row_fma = [&](const uint16_t* X, const float* W, int c) {
    unsigned long long xx[8], ww[4];
#pragma unroll
    for (int a = 0; a < 8; ++a) {
      // BF16 -> FP32 by one byte permute (integer pipe; the FMA pipe is the busy one)
      uint32_t xf;
      asm("prmt.b32 %0, %1, 0, 0x1044;" : "=r"(xf) : "r"((uint32_t)X[(tsub + a) * TR + c]));
      const float xv = __uint_as_float(xf);
      asm("mov.b64 %0, {%1, %1};" : "=l"(xx[a]) : "f"(xv));
    }
    const float4 w4 = *reinterpret_cast<const float4*>(W + c * TW + esub);
    const float4 v4 = *reinterpret_cast<const float4*>(W + c * TW + esub + 4);
    asm("mov.b64 %0, {%1, %2};" : "=l"(ww[0]) : "f"(w4.x), "f"(w4.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(ww[1]) : "f"(w4.z), "f"(w4.w));
    asm("mov.b64 %0, {%1, %2};" : "=l"(ww[2]) : "f"(v4.x), "f"(v4.y));
    asm("mov.b64 %0, {%1, %2};" : "=l"(ww[3]) : "f"(v4.z), "f"(v4.w));
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int q = 0; q < 4; ++q) asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[a][q]) : "l"(xx[a]), "l"(ww[q]));
  };

  // full tile (every token, expert and row in range, 16-byte W rows): each thread copies the
  // same pieces of every stage, so their addresses are set up once
  constexpr int NWP = TR * (TILE_E / 4) / TTHREADS, NXP = TILE_T * (TR / 8) / TTHREADS;
  static_assert(NWP * TTHREADS == TR * (TILE_E / 4) && NXP * TTHREADS == TILE_T * (TR / 8), "piece split");
  const bool full = (t0 + TILE_T <= T) && (e0 + TILE_E <= E) && ((E & 3) == 0) && (d % TR == 0);
  const float* gW = w_r + (size_t)(tid >> 3) * E + e0 + (tid & 7) * 4;
  const int sW = (tid >> 3) * TW + (tid & 7) * 4;
  const uint16_t* gX = x + (size_t)(t0 + tid / (TR / 8)) * d + (tid % (TR / 8)) * 8;
  const int sX = (tid / (TR / 8)) * TR + (tid % (TR / 8)) * 8;
  auto issue_full = [&](int st, int slot) {
    float* W = Wst + slot * TR * TW;
    uint16_t* X = Xst + slot * TILE_T * TR;
    const float* gw = gW + (size_t)st * TR * E;
#pragma unroll
    for (int i = 0; i < NWP; ++i)
      cp_async16(W + sW + i * (TTHREADS / 8) * TW, gw + (size_t)i * (TTHREADS / 8) * E, 16);
    const uint16_t* gx = gX + (size_t)st * TR;
#pragma unroll
    for (int i = 0; i < NXP; ++i)
      cp_async16(X + sX + i * (TTHREADS / (TR / 8)) * TR, gx + (size_t)i * (TTHREADS / (TR / 8)) * d, 16);
  };

  auto issue = [&](int st) {
    if (full) {
      issue_full(st, st % TSTAGES);
      return;
    }
    const int c0 = st * TR;
    float* W = Wst + (size_t)(st % TSTAGES) * TR * TW;
    uint16_t* X = Xst + (size_t)(st % TSTAGES) * TILE_T * TR;
    // W: TR rows x 32 experts (zeros past E or d); 16-byte pieces when rows are 16-byte aligned
    if ((E & 3) == 0) {
      for (int q = tid; q < TR * (TILE_E / 4); q += TTHREADS) {
        const int r = q >> 3, ee = (q & 7) * 4;
        const bool ok = (c0 + r < d) && (e0 + ee < E);
        const float* src = ok ? w_r + (size_t)(c0 + r) * E + e0 + ee : w_r;
        cp_async16(W + r * TW + ee, src, ok ? 16 : 0);
      }
    } else {
      for (int q = tid; q < TR * TILE_E; q += TTHREADS) {
        const int r = q >> 5, ee = q & 31;
        const bool ok = (c0 + r < d) && (e0 + ee < E);
        const float* src = ok ? w_r + (size_t)(c0 + r) * E + e0 + ee : w_r;
        cp_async4(W + r * TW + ee, src, ok ? 4 : 0);
      }
    }
    // x: TILE_T tokens x TR values, 16-byte pieces (zeros past T or d)
    for (int q = tid; q < TILE_T * (TR / 8); q += TTHREADS) {
      const int tt = q / (TR / 8), pc = (q % (TR / 8)) * 8;
      const bool ok = (t0 + tt < T) && (c0 + pc < d);
      const uint16_t* src = ok ? x + (size_t)(t0 + tt) * d + c0 + pc : x;
      cp_async16(X + tt * TR + pc, src, ok ? 16 : 0);
    }
  };

  pdl_wait();
#pragma unroll
  for (int st = 0; st < TSTAGES - 1; ++st) {
    if (st < nst) issue(st);
    cp_async_commit();
  }
  for (int st = 0; st < nst; ++st) {
    cp_async_wait<TSTAGES - 2>();
    __syncthreads();   // stage st landed for every thread; stage st-1 is no longer read
    if (st + TSTAGES - 1 < nst) issue(st + TSTAGES - 1);
    cp_async_commit();
    const float* W = Wst + (size_t)(st % TSTAGES) * TR * TW;
    const uint16_t* X = Xst + (size_t)(st % TSTAGES) * TILE_T * TR;
    const int rows = min(TR, d - st * TR);
    if (rows == TR) {
#pragma unroll
      for (int u = 0; u < TR; u += 32) row_fma(X, W, u + lane);
    } else {
      for (int u = 0; u < rows; u += 32) row_fma(X, W, u + lane);
    }
  }
  float v[64];   // v[a*8 + b]
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int q = 0; q < 4; ++q) asm("mov.b64 {%0, %1}, %2;" : "=f"(v[a * 8 + 2 * q]), "=f"(v[a * 8 + 2 * q + 1]) : "l"(acc2[a][q]));
  // the butterfly over the 32 partials (xor 16, 8, 4, 2, 1) as a reduce-scatter: at each level a
  // lane keeps the half of its sums selected by that lane bit and adds its partner's copy of them
  // (the same pairs as the full butterfly, so the same bits); lane L ends with sums 2L and 2L+1
#pragma unroll
  for (int lvl = 0; lvl < 5; ++lvl) {
    const int m = 16 >> lvl, h = 32 >> lvl;
    const bool up = (lane & m) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = up ? v[i] : v[i + h];
      const float keep = up ? v[i + h] : v[i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, m));
    }
  }
  const int t = t0 + tsub + (lane >> 2), e = e0 + esub + (lane & 3) * 2;
  if (t < T) {
    float* dst = S + (size_t)t * E + e;
    if (e + 1 < E && (E & 1) == 0) {
      *reinterpret_cast<float2*>(dst) = make_float2(score_ref(v[0], score_fn), score_ref(v[1], score_fn));
    } else {
      if (e < E) dst[0] = score_ref(v[0], score_fn);
      if (e + 1 < E) dst[1] = score_ref(v[1], score_fn);
    }
  }
}

template <int NI>
__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ S, const float* __restrict__ bias,
                                                   int T, int E, int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ wts, const RouteVar rv) {
  pdl_wait();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const bool media = row_media(rv, t);
  if (rv.tid2eid != nullptr && !media) {
    hash_row(S + (size_t)t * E, E, k, rv, t, ids + (size_t)t * k, wts + (size_t)t * k, false);
    return;
  }
  topk_warp<NI>(S + (size_t)t * E, media ? rv.vbias : bias, E, k, ids + (size_t)t * k, wts + (size_t)t * k);
}

// Stable counting sort of pair ids by expert, one CTA of 1024 threads.  Pairs are taken
// in chunks of 1024 in order; within a chunk a pair's rank among equal ids comes from a
// warp match (lower lanes) plus the per-warp counts of lower warps.
constexpr int PERM_THREADS = 1024;
constexpr int PERM_EMAX = 1024;

__global__ void __launch_bounds__(PERM_THREADS, 1) permute_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                                  int32_t* __restrict__ offsets,
                                                                  int32_t* __restrict__ perm,
                                                                  int32_t* __restrict__ inv,
                                                                  int32_t* __restrict__ active,
                                                                  int32_t* __restrict__ n_active, int32_t* err) {
  extern __shared__ __align__(16) int perm_smem[];
  int* cnt = perm_smem;                                   // [E+1]
  int* base = cnt + (E + 1);                              // [E+1]
  int* running = base + (E + 1);                          // [E+1]
  unsigned short* wcnt = reinterpret_cast<unsigned short*>(running + (E + 1));  // [32][E+1]
  __shared__ int wsum[32];
  __shared__ int wflag[32];
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i <= E; i += PERM_THREADS) {
    cnt[i] = 0;
    running[i] = 0;
  }
  for (int i = tid; i < 32 * (E + 1); i += PERM_THREADS) wcnt[i] = 0;
  __syncthreads();
  bool bad = false;
  for (int p = tid; p < P; p += PERM_THREADS) {
    const int e = ids[p];
    if (e >= 0 && e < E)
      atomicAdd(&cnt[e], 1);
    else {
      atomicAdd(&cnt[E], 1);
      bad = true;
    }
  }
  if (bad) set_err(err, BRE_DEVERR_EXPERT_ID);
  __syncthreads();
  // exclusive scan of cnt[0..E) -> base; active flags scan -> active list (E <= 1024: one per thread)
  {
    const int c = (tid < E) ? cnt[tid] : 0;
    const int f = (tid < E && c > 0) ? 1 : 0;
    int ic = c, iff = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, ic, o);
      const int b = __shfl_up_sync(0xffffffffu, iff, o);
      if (lane >= o) {
        ic += a;
        iff += b;
      }
    }
    if (lane == 31) {
      wsum[warp] = ic;
      wflag[warp] = iff;
    }
    __syncthreads();
    if (warp == 0) {
      int s = wsum[lane], g = wflag[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, s, o);
        const int b = __shfl_up_sync(0xffffffffu, g, o);
        if (lane >= o) {
          s += a;
          g += b;
        }
      }
      wsum[lane] = s;   // inclusive over warps
      wflag[lane] = g;
    }
    __syncthreads();
    const int prev_c = (warp > 0 ? wsum[warp - 1] : 0) + ic - c;
    const int prev_f = (warp > 0 ? wflag[warp - 1] : 0) + iff - f;
    if (tid < E) {
      base[tid] = prev_c;
      offsets[tid] = prev_c;
      if (f) active[prev_f] = tid;
    }
    const int total_valid = wsum[31];
    const int total_active = wflag[31];
    if (tid == 0) {
      base[E] = total_valid;
      offsets[E] = total_valid;
      *n_active = total_active;
    }
    for (int i = total_active + tid; i < E; i += PERM_THREADS) active[i] = -1;
  }
  __syncthreads();
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int c0 = 0; c0 < P; c0 += PERM_THREADS) {
    const int p = c0 + tid;
    int key = -1;
    if (p < P) {
      const int e = ids[p];
      key = (e >= 0 && e < E) ? e : E;
    }
    const unsigned m = __match_any_sync(0xffffffffu, key);
    const int lrank = __popc(m & lt_mask);
    const bool leader = (lrank == 0);
    if (p < P && leader) wcnt[warp * (E + 1) + key] = (unsigned short)__popc(m);
    __syncthreads();
    int pos = 0;
    if (p < P) {
      int pre = 0;
      for (int w2 = 0; w2 < warp; ++w2) pre += wcnt[w2 * (E + 1) + key];
      pos = base[key] + running[key] + pre + lrank;
    }
    __syncthreads();
    if (p < P) {
      perm[pos] = p;
      inv[p] = pos;
      if (leader) {
        atomicAdd(&running[key], __popc(m));
        wcnt[warp * (E + 1) + key] = 0;
      }
    }
    __syncthreads();
  }
}

// Large P: the same stable order from three launches over chunks of PERM_THREADS pairs (the
// one-CTA kernel's chunks): per-chunk histograms; one CTA turns each key's counts into the
// counts of earlier chunks and writes the offsets (the keys' global bases) and the active list;
// then every chunk places its pairs at offset + earlier-chunk count + warp-match rank.
__global__ void __launch_bounds__(PERM_THREADS) perm_count_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                                  int32_t* __restrict__ counts, int32_t* err) {
  extern __shared__ __align__(16) int hist[];   // [E+1]
  pdl_wait();
  const int tid = threadIdx.x;
  for (int i = tid; i <= E; i += PERM_THREADS) hist[i] = 0;
  __syncthreads();
  const int p = blockIdx.x * PERM_THREADS + tid;
  if (p < P) {
    const int e = ids[p];
    const bool ok = (e >= 0 && e < E);
    if (!ok) set_err(err, BRE_DEVERR_EXPERT_ID);
    atomicAdd(&hist[ok ? e : E], 1);
  }
  __syncthreads();
  for (int i = tid; i <= E; i += PERM_THREADS) counts[(size_t)blockIdx.x * (E + 1) + i] = hist[i];
}

__global__ void __launch_bounds__(PERM_THREADS, 1) perm_scan_kernel(int32_t* __restrict__ counts, int nch, int E,
                                                                    int32_t* __restrict__ offsets,
                                                                    int32_t* __restrict__ active,
                                                                    int32_t* __restrict__ n_active) {
  __shared__ int tot[PERM_EMAX + 1];
  __shared__ int wsum[32];
  __shared__ int wflag[32];
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // per key: counts of earlier chunks (in place), and the key's total; twelve chunks' counts
  // are loaded before any is rewritten
  for (int e = tid; e <= E; e += PERM_THREADS) {
    int run = 0;
    for (int c0 = 0; c0 < nch; c0 += 12) {
      int v[12];
#pragma unroll
      for (int u = 0; u < 12; ++u) v[u] = (c0 + u < nch) ? counts[(size_t)(c0 + u) * (E + 1) + e] : 0;
#pragma unroll
      for (int u = 0; u < 12; ++u)
        if (c0 + u < nch) {
          counts[(size_t)(c0 + u) * (E + 1) + e] = run;
          run += v[u];
        }
    }
    tot[e] = run;
  }
  __syncthreads();
  // exclusive scan of tot[0..E) -> base; active flags scan -> active list (E <= 1024: one per thread)
  const int c = (tid < E) ? tot[tid] : 0;
  const int f = (tid < E && c > 0) ? 1 : 0;
  int ic = c, iff = f;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, o);
    const int b = __shfl_up_sync(0xffffffffu, iff, o);
    if (lane >= o) {
      ic += a;
      iff += b;
    }
  }
  if (lane == 31) {
    wsum[warp] = ic;
    wflag[warp] = iff;
  }
  __syncthreads();
  if (warp == 0) {
    int sm = wsum[lane], g = wflag[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, sm, o);
      const int b = __shfl_up_sync(0xffffffffu, g, o);
      if (lane >= o) {
        sm += a;
        g += b;
      }
    }
    wsum[lane] = sm;   // inclusive over warps
    wflag[lane] = g;
  }
  __syncthreads();
  const int prev_c = (warp > 0 ? wsum[warp - 1] : 0) + ic - c;
  const int prev_f = (warp > 0 ? wflag[warp - 1] : 0) + iff - f;
  const int total_valid = wsum[31], total_active = wflag[31];
  if (tid < E) {
    offsets[tid] = prev_c;
    if (f) active[prev_f] = tid;
  }
  if (tid == 0) {
    offsets[E] = total_valid;   // invalid ids go after every valid pair
    *n_active = total_active;
  }
  for (int i = total_active + tid; i < E; i += PERM_THREADS) active[i] = -1;
}

__global__ void __launch_bounds__(PERM_THREADS) perm_place_kernel(const int32_t* __restrict__ ids, int P, int E,
                                                                  const int32_t* __restrict__ earlier,
                                                                  const int32_t* __restrict__ offsets,
                                                                  int32_t* __restrict__ perm,
                                                                  int32_t* __restrict__ inv) {
  extern __shared__ __align__(16) int place_smem[];
  int* base = place_smem;                                                       // [E+1]
  unsigned short* wcnt = reinterpret_cast<unsigned short*>(base + (E + 1));     // [32][E+1]
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i <= E; i += PERM_THREADS) base[i] = offsets[i] + earlier[(size_t)blockIdx.x * (E + 1) + i];
  for (int i = tid; i < 32 * (E + 1); i += PERM_THREADS) wcnt[i] = 0;
  __syncthreads();
  const int p = blockIdx.x * PERM_THREADS + tid;
  int key = -1;
  if (p < P) {
    const int e = ids[p];
    key = (e >= 0 && e < E) ? e : E;
  }
  const unsigned m = __match_any_sync(0xffffffffu, key);
  const int lrank = __popc(m & ((1u << lane) - 1u));
  if (p < P && lrank == 0) wcnt[warp * (E + 1) + key] = (unsigned short)__popc(m);
  __syncthreads();
  if (p < P) {
    int pre = 0;
    for (int w2 = 0; w2 < warp; ++w2) pre += wcnt[w2 * (E + 1) + key];
    const int pos = base[key] + pre + lrank;
    perm[pos] = p;
    inv[p] = pos;
  }
}

}  // namespace

size_t route_ws_bytes(int T, int E) {
  // scores (T x E) for the large-batch path; candidates (s, id) for the small-batch path
  size_t s = (size_t)T * E * sizeof(float);
  // small batches: candidates (12 bytes a slot), then the hash rows' table scores [T][32]
  if (T <= SMALL_T_MAX) s = std::max(s, (size_t)T * rc_slots(E, 32) * 12 + (size_t)T * 32 * 4);
  s = (s + 255) & ~(size_t)255;
  return s + 256;
}

namespace {
cudaError_t route_impl(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                       int32_t* ids, float* w, void* ws, const PermOut& po, const RouteVar& rv, bool* permuted,
                       cudaStream_t s);
}

cudaError_t launch_route(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                         int32_t* ids, float* w, void* ws, cudaStream_t s) {
  bool permuted = false;
  return route_impl(x, w_r, bias, T, d, E, k, ids, w, ws, PermOut{}, RouteVar{}, &permuted, s);
}

cudaError_t launch_route_ex(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                            int score, const float* vision_bias, const uint8_t* is_media, const int32_t* tid2eid,
                            const int32_t* token_ids, int vocab, int32_t* ids, float* w, int32_t* err, void* ws,
                            cudaStream_t s) {
  bool permuted = false;
  RouteVar rv{};
  rv.score = score;
  rv.vbias = vision_bias;
  rv.media = is_media;
  rv.tid2eid = tid2eid;
  rv.tok = token_ids;
  rv.vocab = vocab;
  rv.err = err;
  return route_impl(x, w_r, bias, T, d, E, k, ids, w, ws, PermOut{}, rv, &permuted, s);
}

cudaError_t launch_route_permute(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                                 int32_t* ids, float* w, int32_t* offsets, int32_t* perm, int32_t* inv,
                                 int32_t* active, int32_t* n_active, int32_t* err, void* ws, cudaStream_t s) {
  bool permuted = false;
  RouteVar rv{};
  rv.err = err;
  const cudaError_t e =
      route_impl(x, w_r, bias, T, d, E, k, ids, w, ws, PermOut{offsets, perm, inv, active, n_active}, rv, &permuted,
                 s);
  if (e != cudaSuccess || permuted) return e;
  // the score buffer is dead once the top k are chosen: it holds the chunk counts
  return launch_permute(ids, T, k, E, offsets, perm, inv, active, n_active, err, s,
                        static_cast<char*>(ws) + 256, route_ws_bytes(T, E) - 256);
}

namespace {
// Tensor map of W_r for the small-batch router's slice copies (RouteMap), cached per (W_r, d, E):
// decode calls repeat the same few, and an encode costs host time on every call.  use = 0 when
// W_r does not meet the copy's rules (then the kernel copies with cp.async).
bool route_map(RouteMap* rm, const float* w_r, int d, int E) {
  rm->use = 0;
  const int n = d / 32;
  if ((E & 3) != 0 || n < 1 || n > 256 || (reinterpret_cast<uintptr_t>(w_r) & 15) != 0) return true;
  struct Entry {
    const float* w;
    int d, E;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[32];
  static int n_cached = 0, next = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cached; ++i) {
    if (cache[i].w == w_r && cache[i].d == d && cache[i].E == E) {
      rm->map = cache[i].map;
      rm->use = 1;
      return true;
    }
  }
  const uint64_t dims[3] = {(uint64_t)E, 32u, (uint64_t)n};
  const uint64_t strides[2] = {(uint64_t)E * 4u, (uint64_t)E * 128u};
  const uint32_t box[3] = {32u, (uint32_t)RC_J, (uint32_t)n};
  if (!encode_tiled(&rm->map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, w_r, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return false;
  cache[next] = Entry{w_r, d, E, rm->map};
  next = (next + 1) % 32;
  if (n_cached < 32) ++n_cached;
  rm->use = 1;
  return true;
}

cudaError_t route_impl(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                       int32_t* ids, float* w, void* ws, const PermOut& po, const RouteVar& rv_in, bool* permuted,
                       cudaStream_t s) {
  RouteVar rv = rv_in;
  int32_t* err = rv.err;
  // the small-batch kernel's ticket sits at a fixed offset, so that calls with different T share it
  int* ticket = reinterpret_cast<int*>(ws);
  float* S = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + 256);
  const size_t small_smem = (size_t)(d / 32) * (RC_J * 32 + RC_J * SMALL_TT) * sizeof(float);
  // the merging CTA's shared memory (words): ids [T k], two count arrays [E + 1], and the
  // candidates of at least one token (3 words a slot)
  const int slots = rc_slots(E, k);
  const size_t fixed_words = (size_t)T * k + 2 * (size_t)(E + 1);
  const size_t avail_words = small_smem / 4;
  if (T <= SMALL_T_MAX && small_smem <= (size_t)device_max_smem_optin() &&
      avail_words >= fixed_words + 3 * (size_t)slots) {
    const int merge_group = (int)std::min<size_t>((size_t)T, (avail_words - fixed_words) / (3 * (size_t)slots));
    RouteMap rm;
    if (!route_map(&rm, w_r, d, E)) return cudaErrorInvalidValue;
    const size_t smem = small_smem;
    static int configured_dev = -1;
    static size_t configured_smem = 0;
    int dev;
    cudaGetDevice(&dev);
    if (dev != configured_dev || smem > configured_smem) {
      cudaError_t e = cudaFuncSetAttribute(route_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
      configured_dev = dev;
      configured_smem = smem;
    }
    uint32_t* cand_c = reinterpret_cast<uint32_t*>(S);
    float* cand_s = S + (size_t)T * slots;
    int* cand_id = reinterpret_cast<int*>(S + (size_t)2 * T * slots);
    rv.hash_s = S + (size_t)3 * T * rc_slots(E, 32);   // after the largest candidate area
    dim3 grid((E + 31) / 32, RC_CLUSTER, (T + SMALL_TT - 1) / SMALL_TT);
    {
      const cudaError_t le = launch_k(route_cluster_kernel, dim3(grid), dim3(RC_THREADS), smem, s, x, w_r, bias, T,
                                      d, E, k, cand_c, cand_s, cand_id, ticket, ids, w, po, merge_group, err, rm, rv);
      if (le != cudaSuccess) return le;
    }
    *permuted = po.offsets != nullptr;
    return cudaGetLastError();
  }
  static int tiled_dev = -1;
  int dev;
  cudaGetDevice(&dev);
  if (dev != tiled_dev) {
    cudaError_t e = cudaFuncSetAttribute(route_tiled_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)TILED_SMEM);
    if (e != cudaSuccess) return e;
    tiled_dev = dev;
  }
  dim3 grid((T + TILE_T - 1) / TILE_T, (E + TILE_E - 1) / TILE_E);
  {
    const cudaError_t le =
        launch_k(route_tiled_kernel, dim3(grid), dim3(TTHREADS), TILED_SMEM, s, x, w_r, T, d, E, S, rv.score);
    if (le != cudaSuccess) return le;
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    auto kern = E <= 32 ? topk_kernel<1> : E <= 128 ? topk_kernel<4> : E <= 384 ? topk_kernel<12> : topk_kernel<32>;
    const cudaError_t le = launch_k(kern, dim3((T + 7) / 8), dim3(256), 0, s, S, bias, T, E, k, ids, w, rv);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* perm, int32_t* inv,
                           int32_t* active, int32_t* n_active, int32_t* err, cudaStream_t s, void* scratch,
                           size_t scratch_bytes) {
  const int P = T * k;
  const int nch = (P + PERM_THREADS - 1) / PERM_THREADS;
  if (nch > 1 && scratch != nullptr && (size_t)nch * (E + 1) * sizeof(int32_t) <= scratch_bytes) {
    int32_t* counts = static_cast<int32_t*>(scratch);
    const size_t place_smem = (size_t)(E + 1) * sizeof(int) + (size_t)32 * (E + 1) * sizeof(unsigned short);
    static int place_dev = -1;
    int dev;
    cudaGetDevice(&dev);
    if (dev != place_dev) {
      const int max_smem = (int)((size_t)(PERM_EMAX + 1) * sizeof(int) + (size_t)32 * (PERM_EMAX + 1) * 2);
      cudaError_t e = cudaFuncSetAttribute(perm_place_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
      if (e != cudaSuccess) return e;
      place_dev = dev;
    }
    cudaError_t le = launch_k(perm_count_kernel, dim3(nch), dim3(PERM_THREADS), (size_t)(E + 1) * sizeof(int), s, ids,
                              P, E, counts, err);
    if (le != cudaSuccess) return le;
    le = launch_k(perm_scan_kernel, dim3(1), dim3(PERM_THREADS), 0, s, counts, nch, E, offsets, active, n_active);
    if (le != cudaSuccess) return le;
    le = launch_k(perm_place_kernel, dim3(nch), dim3(PERM_THREADS), place_smem, s, ids, P, E,
                  static_cast<const int32_t*>(counts), static_cast<const int32_t*>(offsets), perm, inv);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
  }
  const size_t smem = (size_t)3 * (E + 1) * sizeof(int) + (size_t)32 * (E + 1) * sizeof(unsigned short);
  static int configured_dev = -1;
  int dev;
  cudaGetDevice(&dev);
  if (dev != configured_dev) {
    const int max_smem = (int)((size_t)3 * (PERM_EMAX + 1) * sizeof(int) + (size_t)32 * (PERM_EMAX + 1) * 2);
    cudaError_t e = cudaFuncSetAttribute(permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  {
    const cudaError_t le = launch_k(permute_kernel, dim3(1), dim3(PERM_THREADS), smem, s, ids, T * k, E, offsets,
                                    perm, inv, active, n_active, err);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace bre
