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
#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

namespace {

constexpr int SMALL_TT = 8;      // tokens per CTA, small-batch logits
constexpr int SMALL_ET = 4;      // experts per CTA, small-batch logits
constexpr int SMALL_THREADS = SMALL_ET * 32;
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

// Does (ka, ia) rank before (kb, ib)?  Larger key first, then lower id; NaN last.
__device__ __forceinline__ bool ranks_before(float ka, int ia, float kb, int ib) {
  const bool na = isnan(ka), nb = isnan(kb);
  if (na != nb) return !na;
  if (!na && ka != kb) return ka > kb;
  return ia < ib;
}

// One warp selects the top k of the E scores of one token and writes ids and weights.
__device__ void topk_warp(const float* __restrict__ s_row, const float* __restrict__ bias, int E, int k,
                          int32_t* __restrict__ ids_out, float* __restrict__ w_out) {
  const int lane = threadIdx.x & 31;
  float sv[32], kv[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = lane + 32 * i;
    if (e < E) {
      sv[i] = __ldcg(s_row + e);
      kv[i] = __fadd_rn(sv[i], bias ? __ldg(bias + e) : 0.0f);
    } else {
      sv[i] = 0.0f;
      kv[i] = 0.0f;
    }
  }
  uint32_t used = 0;
  float my_sel_s = 0.0f;
  int my_sel_id = 0;
  for (int j = 0; j < k; ++j) {
    float bk = 0.0f, bs = 0.0f;
    int bid = -1;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((used >> i) & 1u)) {
        if (bid < 0 || ranks_before(kv[i], e, bk, bid)) {
          bk = kv[i];
          bid = e;
          bs = sv[i];
        }
      }
    }
    // warp arg-best; lanes with no candidate carry id = INT_MAX and rank last
    float wk = bk;
    int wid = bid < 0 ? 0x7FFFFFFF : bid;
    bool has = bid >= 0;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
      const float ok = __shfl_xor_sync(0xffffffffu, wk, o);
      const int oid = __shfl_xor_sync(0xffffffffu, wid, o);
      const bool ohas = __shfl_xor_sync(0xffffffffu, (int)has, o) != 0;
      bool take;
      if (has != ohas)
        take = ohas;
      else if (!has)
        take = oid < wid;
      else
        take = ranks_before(ok, oid, wk, wid);
      if (take) {
        wk = ok;
        wid = oid;
        has = ohas;
      }
    }
    const int owner = wid & 31;
    const float ws = __shfl_sync(0xffffffffu, bs, owner);
    if (lane == owner) used |= 1u << (wid >> 5);
    if (lane == j) {
      my_sel_s = ws;
      my_sel_id = wid;
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

// Small batches: CTA = up to SMALL_TT tokens x SMALL_ET experts, all 32 partials.
// Thread (e_l = tid % SMALL_ET, j = tid / SMALL_ET) runs the fmaf chain of partial j of expert e_l
// for every token of the CTA.  With NI = d/32 known at compile time every W_r load of the
// thread is issued before the first FMA (one memory round trip); x is staged once as FP32,
// transposed to [c][token], so one row costs two 16-byte shared loads.  The last CTA to
// finish selects the top k of every token.
template <int NI>
__global__ void __launch_bounds__(SMALL_THREADS) route_small_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ w_r,
                                                          const float* __restrict__ bias, int T, int d, int E,
                                                          int k, float* __restrict__ S, int* ticket,
                                                          int32_t* __restrict__ ids, float* __restrict__ wts) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* xs = reinterpret_cast<float*>(smem_raw);                                    // [d][TT]
  float* part = reinterpret_cast<float*>(smem_raw + (size_t)SMALL_TT * d * 4);      // [TT][32][ET]
  __shared__ int is_last;
  pdl_wait();
  const int tid = threadIdx.x;
  const int e0 = blockIdx.x * SMALL_ET;
  const int t0 = blockIdx.y * SMALL_TT;
  const int nt = min(SMALL_TT, T - t0);
  const int e_l = tid % SMALL_ET, j = tid / SMALL_ET;
  const int e = e0 + e_l;
  const float* wcol = w_r + (e < E ? e : 0);
  float wv[NI > 0 ? NI : 1];
  if (NI > 0) {
#pragma unroll
    for (int i = 0; i < NI; ++i) wv[i] = (e < E) ? __ldg(wcol + (size_t)(j + 32 * i) * E) : 0.0f;
  }
  // token index fastest across threads: the eight stores of a row land in eight consecutive words
#pragma unroll 8
  for (int i = tid; i < SMALL_TT * d / 8; i += SMALL_THREADS) {
    const int tt = i % SMALL_TT, c = (i / SMALL_TT) * 8;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (tt < nt) v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * d + c));
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      xs[(c + 2 * q) * SMALL_TT + tt] = bf16_bits_to_f32(w4[q] & 0xFFFFu);
      xs[(c + 2 * q + 1) * SMALL_TT + tt] = bf16_bits_to_f32(w4[q] >> 16);
    }
  }
  __syncthreads();
  float acc[SMALL_TT];
#pragma unroll
  for (int tt = 0; tt < SMALL_TT; ++tt) acc[tt] = 0.0f;
  auto fma_row = [&](int c, float wgt) {
    const float4* xp = reinterpret_cast<const float4*>(xs + c * SMALL_TT);
    const float4 a = xp[0], b = xp[1];
    const float xv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int tt = 0; tt < SMALL_TT; ++tt) acc[tt] = fmaf(xv[tt], wgt, acc[tt]);
  };
  if (NI > 0) {
#pragma unroll
    for (int i = 0; i < NI; ++i) fma_row(j + 32 * i, wv[i]);
  } else {
    const int n = d / 32;
    constexpr int B = 16;
    for (int i0 = 0; i0 < n; i0 += B) {
      float wb[B];
#pragma unroll
      for (int u = 0; u < B; ++u) wb[u] = (e < E && i0 + u < n) ? __ldg(wcol + (size_t)(j + 32 * (i0 + u)) * E) : 0.0f;
#pragma unroll
      for (int u = 0; u < B; ++u)
        if (i0 + u < n) fma_row(j + 32 * (i0 + u), wb[u]);
    }
  }
#pragma unroll
  for (int tt = 0; tt < SMALL_TT; ++tt) part[(tt * 32 + j) * SMALL_ET + e_l] = acc[tt];
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int q = warp; q < SMALL_TT * SMALL_ET; q += SMALL_THREADS / 32) {
    const int tt = q / SMALL_ET, el = q % SMALL_ET;
    float v = part[(tt * 32 + lane) * SMALL_ET + el];
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0 && tt < nt && e0 + el < E) S[(size_t)(t0 + tt) * E + e0 + el] = sigmoid_ref(v);
  }
  // the last CTA selects
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int total = gridDim.x * gridDim.y;
    is_last = (atomicAdd(ticket, 1) == total - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int t = warp; t < T; t += SMALL_THREADS / 32)
    topk_warp(S + (size_t)t * E, bias, E, k, ids + (size_t)t * k, wts + (size_t)t * k);
  if (tid == 0) *ticket = 0;
}

// Large batches: CTA = TILE_T tokens x TILE_E experts, 16 warps.  Lane = partial j; warp q
// owns tokens 8*(q/4) .. +8 and experts 8*(q%4) .. +8 of the tile.  Rows are staged 32 at a
// time through shared memory (lane j uses row c0 + j).
__global__ void __launch_bounds__(512, 1) route_tiled_kernel(const uint16_t* __restrict__ x,
                                                             const float* __restrict__ w_r, int T, int d, int E,
                                                             float* __restrict__ S) {
  __shared__ __align__(16) float Wt[32][TILE_E + 4];
  __shared__ __align__(16) float Xt[32][TILE_T + 4];
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int t0 = blockIdx.x * TILE_T, e0 = blockIdx.y * TILE_E;
  const int tsub = (warp >> 2) * 8, esub = (warp & 3) * 8;
  float acc[8][8];
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) acc[a][b] = 0.0f;

  // register staging: W 32x32 floats = 2 per thread; X 32 tokens x 32 values = 2 per thread
  const int wr_r = tid >> 4, wr_c = (tid & 15) * 2;
  const int xr_t = tid >> 4, xr_c = (tid & 15) * 2;
  float2 wreg;
  uint32_t xreg;
  auto load = [&](int c0) {
    const int e = e0 + wr_c;
    const float* wp = w_r + (size_t)(c0 + wr_r) * E + e;
    wreg.x = (e < E) ? __ldg(wp) : 0.0f;
    wreg.y = (e + 1 < E) ? __ldg(wp + 1) : 0.0f;
    const int t = t0 + xr_t;
    xreg = (t < T) ? __ldg(reinterpret_cast<const uint32_t*>(x + (size_t)t * d + c0 + xr_c)) : 0u;
  };
  load(0);
  for (int c0 = 0; c0 < d; c0 += 32) {
    __syncthreads();
    Wt[wr_r][wr_c] = wreg.x;
    Wt[wr_r][wr_c + 1] = wreg.y;
    Xt[xr_c + 0][xr_t] = bf16_bits_to_f32(xreg & 0xFFFFu);
    Xt[xr_c + 1][xr_t] = bf16_bits_to_f32(xreg >> 16);
    __syncthreads();
    if (c0 + 32 < d) load(c0 + 32);
    float xv[8], wv[8];
    const float4* xp = reinterpret_cast<const float4*>(&Xt[lane][tsub]);
    const float4* wp = reinterpret_cast<const float4*>(&Wt[lane][esub]);
    float4 t4 = xp[0], u4 = xp[1];
    xv[0] = t4.x; xv[1] = t4.y; xv[2] = t4.z; xv[3] = t4.w;
    xv[4] = u4.x; xv[5] = u4.y; xv[6] = u4.z; xv[7] = u4.w;
    float4 w4 = wp[0], v4 = wp[1];
    wv[0] = w4.x; wv[1] = w4.y; wv[2] = w4.z; wv[3] = w4.w;
    wv[4] = v4.x; wv[5] = v4.y; wv[6] = v4.z; wv[7] = v4.w;
#pragma unroll
    for (int a = 0; a < 8; ++a)
#pragma unroll
      for (int b = 0; b < 8; ++b) acc[a][b] = fmaf(xv[a], wv[b], acc[a][b]);
  }
  // butterfly over the 32 partials (lanes); every lane ends with the same sums
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      float v = acc[a][b];
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
      acc[a][b] = v;
    }
#pragma unroll
  for (int a = 0; a < 8; ++a)
#pragma unroll
    for (int b = 0; b < 8; ++b) {
      if (lane == ((a * 8 + b) & 31)) {
        const int t = t0 + tsub + a, e = e0 + esub + b;
        if (t < T && e < E) S[(size_t)t * E + e] = sigmoid_ref(acc[a][b]);
      }
    }
}

__global__ void __launch_bounds__(256) topk_kernel(const float* __restrict__ S, const float* __restrict__ bias,
                                                   int T, int E, int k, int32_t* __restrict__ ids,
                                                   float* __restrict__ wts) {
  pdl_wait();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_warp(S + (size_t)t * E, bias, E, k, ids + (size_t)t * k, wts + (size_t)t * k);
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

}  // namespace

size_t route_ws_bytes(int T, int E) {
  size_t s = (size_t)T * E * sizeof(float);
  s = (s + 255) & ~(size_t)255;
  return s + 256;
}

cudaError_t launch_route(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                         int32_t* ids, float* w, void* ws, cudaStream_t s) {
  // the ticket sits at a fixed offset so that calls with different T share it
  int* ticket = reinterpret_cast<int*>(ws);
  float* S = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + 256);
  const size_t small_smem = (size_t)SMALL_TT * d * 4 + SMALL_TT * 32 * SMALL_ET * sizeof(float);
  if (T <= SMALL_T_MAX && small_smem <= (size_t)device_max_smem_optin()) {
    const size_t smem = small_smem;
    dim3 grid((E + SMALL_ET - 1) / SMALL_ET, (T + SMALL_TT - 1) / SMALL_TT);
    auto launch = [&](auto kern) -> cudaError_t {
      static int configured_dev = -1;
      static size_t configured_smem = 0;
      int dev;
      cudaGetDevice(&dev);
      if (dev != configured_dev || smem > configured_smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
        configured_smem = smem;
      }
      kern<<<grid, SMALL_THREADS, smem, s>>>(x, w_r, bias, T, d, E, k, S, ticket, ids, w);
      return cudaGetLastError();
    };
    if (d == 4096) return launch(route_small_kernel<128>);
    if (d == 512) return launch(route_small_kernel<16>);
    return launch(route_small_kernel<0>);
  }
  dim3 grid((T + TILE_T - 1) / TILE_T, (E + TILE_E - 1) / TILE_E);
  route_tiled_kernel<<<grid, 512, 0, s>>>(x, w_r, T, d, E, S);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  topk_kernel<<<(T + 7) / 8, 256, 0, s>>>(S, bias, T, E, k, ids, w);
  return cudaGetLastError();
}

cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* perm, int32_t* inv,
                           int32_t* active, int32_t* n_active, int32_t* err, cudaStream_t s) {
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
  permute_kernel<<<1, PERM_THREADS, smem, s>>>(ids, T * k, E, offsets, perm, inv, active, n_active, err);
  return cudaGetLastError();
}

}  // namespace bre
