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
constexpr int SMALL_ET = 8;      // experts per CTA, small-batch logits
constexpr int TILE_T = 32;       // tokens per CTA, tiled logits
constexpr int TILE_E = 32;       // experts per CTA, tiled logits
constexpr int SMALL_T_MAX = 32;  // up to this many tokens use the small-batch kernel

__device__ __forceinline__ float sigmoid_ref(float z) {
  return (float)(1.0 / (1.0 + exp(-(double)z)));
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
// Thread (e_l = tid & 7, j = tid >> 3) runs the fmaf chain of partial j of expert e_l
// for every token of the CTA.  The last CTA to finish selects the top k of every token.
__global__ void __launch_bounds__(256) route_small_kernel(const uint16_t* __restrict__ x,
                                                          const float* __restrict__ w_r,
                                                          const float* __restrict__ bias, int T, int d, int E,
                                                          int k, float* __restrict__ S, int* ticket,
                                                          int32_t* __restrict__ ids, float* __restrict__ wts) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem_raw);                             // [TT][d]
  float* part = reinterpret_cast<float*>(smem_raw + (size_t)SMALL_TT * d * 2);      // [TT][32][8]
  __shared__ int is_last;
  pdl_wait();
  const int tid = threadIdx.x;
  const int e0 = blockIdx.x * SMALL_ET;
  const int t0 = blockIdx.y * SMALL_TT;
  const int nt = min(SMALL_TT, T - t0);
  for (int i = tid; i < SMALL_TT * d / 8; i += 256) {
    const int tt = i / (d / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (tt < nt) v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t0 + tt) * d) + (i % (d / 8)));
    reinterpret_cast<uint4*>(xs)[i] = v;
  }
  __syncthreads();
  const int e_l = tid & 7, j = tid >> 3;
  const int e = e0 + e_l;
  float acc[SMALL_TT];
#pragma unroll
  for (int tt = 0; tt < SMALL_TT; ++tt) acc[tt] = 0.0f;
  const int n = d / 32;
  const float* wcol = w_r + e;
  constexpr int B = 16;
  for (int i0 = 0; i0 < n; i0 += B) {
    float wv[B];
#pragma unroll
    for (int u = 0; u < B; ++u) {
      const int c = j + 32 * (i0 + u);
      wv[u] = (e < E && i0 + u < n) ? __ldg(wcol + (size_t)c * E) : 0.0f;
    }
#pragma unroll
    for (int u = 0; u < B; ++u) {
      if (i0 + u < n) {
        const int c = j + 32 * (i0 + u);
#pragma unroll
        for (int tt = 0; tt < SMALL_TT; ++tt) acc[tt] = fmaf(bf16_bits_to_f32(xs[tt * d + c]), wv[u], acc[tt]);
      }
    }
  }
#pragma unroll
  for (int tt = 0; tt < SMALL_TT; ++tt) part[(tt * 32 + j) * 8 + e_l] = acc[tt];
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int q = warp; q < SMALL_TT * SMALL_ET; q += 8) {
    const int tt = q / SMALL_ET, el = q % SMALL_ET;
    float v = part[(tt * 32 + lane) * 8 + el];
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
  for (int t = warp; t < T; t += 8) topk_warp(S + (size_t)t * E, bias, E, k, ids + (size_t)t * k, wts + (size_t)t * k);
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
  if (T <= SMALL_T_MAX) {
    const size_t smem = (size_t)SMALL_TT * d * 2 + SMALL_TT * 32 * 8 * sizeof(float);
    static int configured_dev = -1;
    static size_t configured_smem = 0;
    int dev;
    cudaGetDevice(&dev);
    if (dev != configured_dev || smem > configured_smem) {
      cudaError_t e = cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
      if (e != cudaSuccess) return e;
      configured_dev = dev;
      configured_smem = smem;
    }
    dim3 grid((E + SMALL_ET - 1) / SMALL_ET, (T + SMALL_TT - 1) / SMALL_TT);
    route_small_kernel<<<grid, 256, smem, s>>>(x, w_r, bias, T, d, E, k, S, ticket, ids, w);
    return cudaGetLastError();
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
