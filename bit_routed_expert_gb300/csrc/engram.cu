// Engram gather-decode: 264-byte rows (256 E4M3 values + 8 E8M0 scales) gathered by
// row id, decoded to FP32, summed over heads in order and rounded to BF16.
// (strix-llama.cpp issue, "Feature Description" and "DeepSeek V4.1 Engram graph
// integration".)
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

// Two E4M3 bytes (low byte -> low half) to two floats; exact (E4M3 is a subset of f16).
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_bytes) {
  uint32_t h2;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.rn.f16x2.e4m3x2 %0, t; }" : "=r"(h2) : "r"(two_bytes));
  return make_float2(f16_bits_to_f32(h2 & 0xFFFFu), f16_bits_to_f32(h2 >> 16));
}

// 2^(e-127) for an E8M0 byte, NaN for 0xFF (exact).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) {
  if (e == 255u) return __uint_as_float(0x7FC00000u);
  if (e == 0u) return __uint_as_float(0x00400000u);  // 2^-127, subnormal
  return __uint_as_float(e << 23);
}

// Decode one 8-value slice of a row (lane l owns values 8l .. 8l+7 and scale byte l/4).
__device__ __forceinline__ void decode8(uint2 v, uint32_t sb, float (&val)[8]) {
  const float sc = e8m0_to_f32(sb);
  const float2 f01 = e4m3x2_to_f32x2(v.x & 0xFFFFu), f23 = e4m3x2_to_f32x2(v.x >> 16);
  const float2 f45 = e4m3x2_to_f32x2(v.y & 0xFFFFu), f67 = e4m3x2_to_f32x2(v.y >> 16);
  val[0] = __fmul_rn(f01.x, sc); val[1] = __fmul_rn(f01.y, sc);   // exact, or +-inf / NaN
  val[2] = __fmul_rn(f23.x, sc); val[3] = __fmul_rn(f23.y, sc);
  val[4] = __fmul_rn(f45.x, sc); val[5] = __fmul_rn(f45.y, sc);
  val[6] = __fmul_rn(f67.x, sc); val[7] = __fmul_rn(f67.y, sc);
}

// Eight E4M3 bytes (values 8l .. 8l+7 of lane l) as four float pairs, unscaled (exact).
__device__ __forceinline__ void e4m3x8_f32(uint2 v, float2 (&o)[4]) {
  const uint32_t w[2] = {v.x, v.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w[i] >> 16), __NV_E4M3);
    o[2 * i] = __half22float2(__half2(lo));
    o[2 * i + 1] = __half22float2(__half2(hi));
  }
}

// Scale bytes below this make value * 2^(e-127) exact and finite for every E4M3 value (|v| <=
// 448 < 2^9, and no E4M3 bit falls below FP32's subnormal floor).
constexpr uint32_t E8M0_NO_OVERFLOW = 246;

// Eight heads (the configuration's H): one warp per (token, table); lanes 0..7 load the eight
// row ids with one instruction and check them with one unsigned compare; every row's loads are
// issued before any decode; the E8M0 scales come from a 256-entry table in shared memory; the
// first head starts the sum.  Same arithmetic as the general kernel below.
__global__ void __launch_bounds__(256) engram_gather8_kernel(EngramTables tabs, int n_tables,
                                                             const int64_t* __restrict__ ids, int T,
                                                             uint16_t* __restrict__ out, int32_t* err) {
  __shared__ float sc_tab[256];
  sc_tab[threadIdx.x] = e8m0_to_f32(threadIdx.x);   // blockDim.x == 256
  __syncthreads();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= (long long)T * n_tables) return;
  const int tau = (int)(w % n_tables);
  const uint8_t* table = tabs.ptr[0];
  long long nrows = tabs.n_rows[0];
#pragma unroll
  for (int q = 1; q < 8; ++q)
    if (tau == q) {
      table = tabs.ptr[q];
      nrows = tabs.n_rows[q];
    }
  const long long myid = lane < 8 ? __ldg(ids + w * 8 + lane) : 0;
  const unsigned okm = __ballot_sync(0xffffffffu, (unsigned long long)myid < (unsigned long long)nrows);
  if ((okm & 0xFFu) != 0xFFu && lane == 0) set_err(err, BRE_DEVERR_ROW_ID);
  uint2 v[8];
  uint32_t sb[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) {
    const long long r = __shfl_sync(0xffffffffu, myid, h);
    const bool ok = (okm >> h) & 1u;
    const uint8_t* row = table + (ok ? r : 0) * ENGRAM_ROW;
    v[h] = ok ? __ldg(reinterpret_cast<const uint2*>(row) + lane) : make_uint2(0u, 0u);
    sb[h] = ok ? __ldg(row + 256 + (lane >> 2)) : 127u;
  }
  // the head sum in head order, two values per packed FP32 instruction.  The result is defined
  // as acc + (value * scale) with the product rounded first.  While the product is exact and
  // finite (scale byte below E8M0_NO_OVERFLOW) a fused multiply-add rounds the same sum once, so
  // a packed FMA does each step; a larger scale may overflow the product, which must then be
  // infinite before the add, so it is formed by scalar multiplies (the compiler fuses a packed
  // multiply into a following packed add, but never a scalar __fmul_rn).
  float2 acc[4];
  uint32_t sb_max = 0;
#pragma unroll
  for (int h = 0; h < 8; ++h) sb_max = max(sb_max, sb[h]);
  if (sb_max < E8M0_NO_OVERFLOW) {   // the lane's eight heads (the common case)
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float sc = sc_tab[sb[h]];
      const float2 s2 = make_float2(sc, sc);
      float2 raw[4];
      e4m3x8_f32(v[h], raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = (h == 0) ? __fmul2_rn(raw[i], s2) : __ffma2_rn(raw[i], s2, acc[i]);
    }
  } else {
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float sc = sc_tab[sb[h]];
      float2 raw[4];
      e4m3x8_f32(v[h], raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 pr = make_float2(__fmul_rn(raw[i].x, sc), __fmul_rn(raw[i].y, sc));
        acc[i] = (h == 0) ? pr : __fadd2_rn(acc[i], pr);
      }
    }
  }
  uint4 o;
  o.x = f32_to_bf16_rne(acc[0].x) | (f32_to_bf16_rne(acc[0].y) << 16);
  o.y = f32_to_bf16_rne(acc[1].x) | (f32_to_bf16_rne(acc[1].y) << 16);
  o.z = f32_to_bf16_rne(acc[2].x) | (f32_to_bf16_rne(acc[2].y) << 16);
  o.w = f32_to_bf16_rne(acc[3].x) | (f32_to_bf16_rne(acc[3].y) << 16);
  reinterpret_cast<uint4*>(out + w * 256)[lane] = o;
}

// One warp per (token, table); HC heads per pass with every row load of the pass issued
// before any decode.  HC is a compile-time count so that the row registers stay registers.
template <int HC>
__global__ void __launch_bounds__(256) engram_gather_kernel(EngramTables tabs, int n_tables,
                                                            const int64_t* __restrict__ ids, int T, int H,
                                                            uint16_t* __restrict__ out, int32_t* err) {
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (w >= (long long)T * n_tables) return;
  const int tau = (int)(w % n_tables);
  // select the table without indexing the parameter array dynamically (that would copy it to local memory)
  const uint8_t* table = tabs.ptr[0];
  long long nrows = tabs.n_rows[0];
#pragma unroll
  for (int q = 1; q < 8; ++q)
    if (tau == q) {
      table = tabs.ptr[q];
      nrows = tabs.n_rows[q];
    }
  const int64_t* idp = ids + w * H;

  float acc[8];
  bool bad = false;
  for (int h0 = 0; h0 < H; h0 += HC) {
    const long long myid = (h0 + lane < H && lane < HC) ? __ldg(idp + h0 + lane) : 0;
    uint2 v[HC];
    uint32_t sb[HC];
#pragma unroll
    for (int h = 0; h < HC; ++h) {
      const long long r = __shfl_sync(0xffffffffu, myid, h);
      const bool ok = (h0 + h < H) && r >= 0 && r < nrows;
      bad |= (h0 + h < H) && !ok;
      const uint8_t* row = table + (ok ? r : 0) * ENGRAM_ROW;
      v[h] = ok ? __ldg(reinterpret_cast<const uint2*>(row) + lane) : make_uint2(0u, 0u);
      sb[h] = ok ? __ldg(row + 256 + (lane >> 2)) : 127u;
    }
#pragma unroll
    for (int h = 0; h < HC; ++h) {
      if (h0 + h < H) {
        float val[8];
        decode8(v[h], sb[h], val);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = (h0 + h == 0) ? val[i] : __fadd_rn(acc[i], val[i]);
      }
    }
  }
  if (bad && lane == 0) set_err(err, BRE_DEVERR_ROW_ID);
  uint4 o;
  o.x = f32_to_bf16_rne(acc[0]) | (f32_to_bf16_rne(acc[1]) << 16);
  o.y = f32_to_bf16_rne(acc[2]) | (f32_to_bf16_rne(acc[3]) << 16);
  o.z = f32_to_bf16_rne(acc[4]) | (f32_to_bf16_rne(acc[5]) << 16);
  o.w = f32_to_bf16_rne(acc[6]) | (f32_to_bf16_rne(acc[7]) << 16);
  reinterpret_cast<uint4*>(out + w * 256)[lane] = o;
}

cudaError_t launch_engram(const EngramTables& tabs, int n_tables, const int64_t* ids, int T, int H, uint16_t* out,
                          int32_t* err, cudaStream_t s) {
  const long long warps = (long long)T * n_tables;
  const int threads = 256;
  const long long blocks = (warps * 32 + threads - 1) / threads;
  if (H == 8) {
    const cudaError_t le = launch_k(engram_gather8_kernel, dim3((unsigned)blocks), dim3(threads), 0, s, tabs,
                                    n_tables, ids, T, out, err);
    if (le != cudaSuccess) return le;
  } else if (H == 1)
    {
      const cudaError_t le = launch_k(engram_gather_kernel<1>, dim3((unsigned)blocks), dim3(threads), 0, s, tabs,
                                      n_tables, ids, T, H, out, err);
      if (le != cudaSuccess) return le;
    }
  else
    {
      const cudaError_t le = launch_k(engram_gather_kernel<8>, dim3((unsigned)blocks), dim3(threads), 0, s, tabs,
                                      n_tables, ids, T, H, out, err);
      if (le != cudaSuccess) return le;
    }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Engram gate and residual injection (strix-llama.cpp issue, "Placement"): the R gathered rows
// of a token, concatenated ([R * 256] BF16), times engram_kv.weight [5W][R * 256] give four keys
// and one shared value of width W; each of the four hyper-connection branches h then takes
//   dot = sum_i r[h,i] qn[h,i] kn[h,i] key[h,i] / sqrt(mean r^2 + eps) / sqrt(mean key^2 + eps)
//         / sqrt(W),
//   gate = sigmoid(copysign(sqrt(max(|dot|, 1e-6)), dot)),  r[h,i] = bf16(r[h,i] + gate bf16(v[i])).
// ---------------------------------------------------------------------------
namespace {

constexpr int KV_WARPS = 8;
constexpr int KV_NS = 4;                     // ring stages per warp (three copies in flight)
constexpr int KV_KS = 128;                   // K per stage (4 warps with 256-K stages measured slower)
constexpr int KV_STAGE = 16 * KV_KS * 2;     // 16 rows x 128 K of W (two 64-K boxes, 128-byte swizzle)
constexpr int KV_TOK = 8;                    // tokens per launch (MMA N)
constexpr long long KV_WAIT = 2000000000LL;  // cycles before a wait gives up

struct KvParams {
  const uint8_t* table;
  long long n_rows;
  const int64_t* row_ids;  // [T][R]
  int R, T, t0, tg;        // rows per token, tokens, this launch's first token and count (<= 8)
  int K, N, KP;            // K = R * 256, N = 5W, K parts
  float* part;             // [KP][T][N]
  int* counter;
  int32_t* err;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Persistent: each warp takes items (16 rows of W, one K part) from a counter and streams the
// item's W through its own ring of 4 KB stages (TMA, 128-byte swizzle so that ldmatrix reads
// are conflict-free); the launch's <= 8 tokens' rows are decoded into shared memory first (BF16,
// row pitch K + 8 elements).  MMA m16n8k16: A = W rows, B = tokens.  Each item stores FP32
// partial sums part[kp][t][n]; the gate kernel adds the parts in order.
__global__ void __launch_bounds__(KV_WARPS * 32, 1) engram_kv_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                    const KvParams p) {
  extern __shared__ __align__(1024) unsigned char kvs[];
  unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(kvs) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + KV_WARPS * KV_NS * KV_STAGE);
  int* q_ids = reinterpret_cast<int*>(bars + KV_WARPS * KV_NS);       // [KV_WARPS][4] item ids in flight
  uint16_t* xs = reinterpret_cast<uint16_t*>(q_ids + KV_WARPS * 4);   // [8][K + 8]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pitch = p.K + 8;
  if (threadIdx.x < KV_WARPS * KV_NS) mbar_init(&bars[threadIdx.x], 1);
  fence_mbar_init();
  __syncthreads();
  pdl_wait();
  const int tiles = p.N / 16, kl = p.K / p.KP, spi = kl / KV_KS;   // stages per item
  const int n_items = tiles * p.KP;
  unsigned char* my_ring = ring + warp * KV_NS * KV_STAGE;
  uint64_t* my_bar = bars + warp * KV_NS;
  int* my_q = q_ids + warp * 4;
  // producer state (lane 0 issues): item being loaded, its stage, sequence number
  int ld_item = 0, ld_c = 0, ld_seq = 0, q_tail = 0;
  auto fetch = [&]() -> int {
    int i = 0;
    if (lane == 0) i = atomicAdd(p.counter, 1);
    i = __shfl_sync(0xffffffffu, i, 0);
    return i < n_items ? i : -1;
  };
  ld_item = fetch();
  if (lane == 0) my_q[q_tail & 3] = ld_item;
  ++q_tail;
  auto issue_next = [&]() {
    if (ld_item < 0) return;
    if (lane == 0) {
      const int slot = ld_seq % KV_NS;
      unsigned char* dst = my_ring + slot * KV_STAGE;
      const int tile = ld_item / p.KP, kp = ld_item - tile * p.KP;
      const int k0 = kp * kl + ld_c * KV_KS;
      mbar_arrive_expect_tx(&my_bar[slot], KV_STAGE);
#pragma unroll
      for (int bx = 0; bx < KV_KS / 64; ++bx) tma_load_2d(dst + bx * 2048, &wmap, k0 + bx * 64, tile * 16, &my_bar[slot]);
    }
    ++ld_seq;
    if (++ld_c == spi) {
      ld_c = 0;
      ld_item = fetch();
      if (lane == 0) my_q[q_tail & 3] = ld_item;
      ++q_tail;
    }
  };
  for (int i = 0; i < KV_NS - 1; ++i) issue_next();
  // decode the launch's tokens' rows into shared memory (zeros past tg; bad ids decode as
  // zeros); a thread's loads, eight slices at a time, are issued before their decodes
  {
    const int per_tok = p.R * 32;   // 8-value slices per token
    const int total = KV_TOK * per_tok;
    bool bad = false;
    for (int q0 = 0; q0 < total; q0 += 8 * KV_WARPS * 32) {
      uint2 v[8];
      uint32_t sb[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int q = q0 + u * KV_WARPS * 32 + threadIdx.x;
        v[u] = make_uint2(0u, 0u);
        sb[u] = 127u;
        if (q < total) {
          const int tt = q / per_tok, rem = q - tt * per_tok, j = rem >> 5, l = rem & 31;
          if (tt < p.tg) {
            const long long r = __ldg(p.row_ids + (size_t)(p.t0 + tt) * p.R + j);
            const bool ok = r >= 0 && r < p.n_rows;
            bad |= !ok;
            if (ok) {
              const uint8_t* row = p.table + r * ENGRAM_ROW;
              v[u] = __ldg(reinterpret_cast<const uint2*>(row) + l);
              sb[u] = __ldg(row + 256 + (l >> 2));
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int q = q0 + u * KV_WARPS * 32 + threadIdx.x;
        if (q < total) {
          const int tt = q / per_tok, rem = q - tt * per_tok, j = rem >> 5, l = rem & 31;
          float val[8];
          decode8(v[u], sb[u], val);   // zeros for absent and bad rows
          uint4 o;
          o.x = f32_to_bf16_rne(val[0]) | (f32_to_bf16_rne(val[1]) << 16);
          o.y = f32_to_bf16_rne(val[2]) | (f32_to_bf16_rne(val[3]) << 16);
          o.z = f32_to_bf16_rne(val[4]) | (f32_to_bf16_rne(val[5]) << 16);
          o.w = f32_to_bf16_rne(val[6]) | (f32_to_bf16_rne(val[7]) << 16);
          *reinterpret_cast<uint4*>(xs + (size_t)tt * pitch + j * 256 + l * 8) = o;
        }
      }
    }
    if (bad) set_err(p.err, BRE_DEVERR_ROW_ID);
  }
  __syncthreads();
  const int g = lane >> 2, t = lane & 3;
  // ldmatrix lane addresses: A (rows (lane & 7) + 8 ((lane >> 3) & 1), 16-byte chunk + (lane >> 4));
  // B (token lane & 7, chunk + ((lane >> 3) & 1))
  const int arow = (lane & 7) + ((lane >> 3) & 1) * 8, achk = lane >> 4;
  const uint32_t xs_lane = smem_u32(xs) + (uint32_t)((lane & 7) * pitch * 2 + ((lane >> 3) & 1) * 16);
  int cs = 0, q_head = 0;
  while (true) {
    __syncwarp();   // lane 0's queue write comes first for every lane
    const int item = my_q[q_head & 3];
    if (item < 0) break;
    const int tile = item / p.KP, kp = item - tile * p.KP;
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int c = 0; c < spi; ++c) {
      const int slot = cs % KV_NS;
      if (!mbar_wait_bounded(&my_bar[slot], (cs / KV_NS) & 1, KV_WAIT)) {
        if (lane == 0) set_err(p.err, BRE_DEVERR_TIMEOUT);
        for (int q = cs + 1; q < ld_seq; ++q) mbar_wait_bounded(&my_bar[q % KV_NS], (q / KV_NS) & 1, KV_WAIT);
        return;
      }
      const uint32_t st = smem_u32(my_ring + slot * KV_STAGE);
      const int kg0 = kp * kl + c * KV_KS;
#pragma unroll
      for (int kk = 0; kk < KV_KS / 16; ++kk) {
        const int box = kk >> 2, chunk = (kk & 3) * 2 + achk;
        uint32_t a0, a1, a2, a3, b0, b1;
        ldsm_x4(st + box * 2048 + arow * 128 + ((chunk ^ (arow & 7)) << 4), a0, a1, a2, a3);
        ldsm_x2(xs_lane + (uint32_t)(kg0 + kk * 16) * 2, b0, b1);
        mma_bf16_16816(acc, a0, a1, a2, a3, b0, b1);
      }
      fence_proxy_async_smem();   // the stage's reads come before the copy that refills it
      __syncwarp();
      ++cs;
      issue_next();
    }
    ++q_head;
    // C fragment: rows tile*16 + g (+8), tokens 2t, 2t+1
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int tt = 2 * t + (i & 1), n = tile * 16 + g + 8 * (i >> 1);
      if (tt < p.tg) p.part[((size_t)kp * p.T + p.t0 + tt) * p.N + n] = acc[i];
    }
  }
}

// The gate in two fully parallel launches.  engram_reduce_kernel: one CTA per (token, 256-element
// slice of a key or of the value): adds the K parts in part order (kv), and for key slices
// forms the slice's three sums (r q_norm k_norm key, r^2, key^2) in a fixed order (thread FMA,
// warp butterfly, warps in order).  engram_apply_kernel: one CTA per (token, branch, slice):
// adds the branch's slice sums in slice order -- every CTA of a branch gets the same gate -- and
// updates its slice.  Deterministic, with no atomics.
constexpr int GATE_THREADS = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = red[0];
  for (int w = 1; w < GATE_THREADS / 32; ++w) s = __fadd_rn(s, red[w]);
  return s;
}

struct GateParams {
  const float* part;   // [KP][T][5W]
  int KP, T, W, NSL;   // NSL = slices of 256 per branch
  float* kv;           // [T][5W] (workspace, or the caller's kv_out)
  float* sums;         // [T][4][NSL][3]
  uint16_t* resid;
  const float* qn;
  const float* kn;
  const uint8_t* mask;
  float eps;
  float* gate_out;
  int* counter;
};

__global__ void __launch_bounds__(GATE_THREADS) engram_reduce_kernel(const GateParams g) {
  __shared__ float red[GATE_THREADS / 32];
  pdl_wait();
  const int t = blockIdx.x, b = blockIdx.y / g.NSL, sl = blockIdx.y % g.NSL;   // b = 0..3 keys, 4 value
  if (t == 0 && blockIdx.y == 0 && threadIdx.x == 0) *g.counter = 0;   // ready for the next projection
  const int i = sl * 256 + threadIdx.x;
  const size_t N = (size_t)5 * g.W, n = (size_t)b * g.W + i;
  float v = 0.0f;
  if (i < g.W) {
    float pv[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) pv[q] = q < g.KP ? __ldcg(g.part + ((size_t)q * g.T + t) * N + n) : 0.0f;
    v = pv[0];
#pragma unroll
    for (int q = 1; q < 8; ++q)
      if (q < g.KP) v = __fadd_rn(v, pv[q]);
    g.kv[(size_t)t * N + n] = v;
  }
  if (b == 4) return;   // value slices: the sum only
  float dot = 0.0f, rr = 0.0f, kk = 0.0f;
  if (i < g.W) {
    const float ri = bf16_bits_to_f32(g.resid[((size_t)t * 4 + b) * g.W + i]);
    const float qk = __fmul_rn(__ldg(g.qn + (size_t)b * g.W + i), __ldg(g.kn + (size_t)b * g.W + i));
    dot = __fmul_rn(__fmul_rn(ri, qk), v);
    rr = __fmul_rn(ri, ri);
    kk = __fmul_rn(v, v);
  }
  dot = block_sum(dot, red);
  rr = block_sum(rr, red);
  kk = block_sum(kk, red);
  if (threadIdx.x == 0) {
    float* s = g.sums + (((size_t)t * 4 + b) * g.NSL + sl) * 3;
    s[0] = dot;
    s[1] = rr;
    s[2] = kk;
  }
}

__global__ void __launch_bounds__(GATE_THREADS) engram_apply_kernel(const GateParams g) {
  pdl_wait();
  const int t = blockIdx.x, h = blockIdx.y / g.NSL, sl = blockIdx.y % g.NSL;
  if (g.mask && g.mask[t]) {
    if (g.gate_out && sl == 0 && threadIdx.x == 0) g.gate_out[t * 4 + h] = 0.0f;
    return;
  }
  const float* s = g.sums + ((size_t)t * 4 + h) * g.NSL * 3;
  float dot = s[0], rr = s[1], kk = s[2];
  for (int q = 1; q < g.NSL; ++q) {
    dot = __fadd_rn(dot, s[q * 3 + 0]);
    rr = __fadd_rn(rr, s[q * 3 + 1]);
    kk = __fadd_rn(kk, s[q * 3 + 2]);
  }
  const float inv_w = 1.0f / (float)g.W;
  dot = __fmul_rn(dot, 1.0f / sqrtf(__fadd_rn(__fmul_rn(rr, inv_w), g.eps)));
  dot = __fmul_rn(dot, 1.0f / sqrtf(__fadd_rn(__fmul_rn(kk, inv_w), g.eps)));
  dot = __fmul_rn(dot, 1.0f / sqrtf((float)g.W));
  const float m = sqrtf(fmaxf(fabsf(dot), 1e-6f));
  const float gate = 1.0f / (1.0f + expf(-copysignf(m, dot)));
  if (g.gate_out && sl == 0 && threadIdx.x == 0) g.gate_out[t * 4 + h] = gate;
  const int i = sl * 256 + threadIdx.x;
  if (i < g.W) {
    uint16_t* r = g.resid + ((size_t)t * 4 + h) * g.W + i;
    const float vb = bf16_bits_to_f32(f32_to_bf16_rne(__ldcg(g.kv + (size_t)t * 5 * g.W + (size_t)4 * g.W + i)));
    *r = (uint16_t)f32_to_bf16_rne(__fmaf_rn(gate, vb, bf16_bits_to_f32(*r)));
  }
}

// K parts: the largest of 8, 4, 2, 1 that leaves whole stages (at R = 24, 12,800 items of
// 24 KB: ~10 per warp, so the last wave is short); K must be a multiple of KV_KS.
int kv_parts(int K) {
  for (int kp = 8; kp >= 1; kp >>= 1)
    if (K % (KV_KS * kp) == 0) return kp;
  return 0;
}

}  // namespace

// workspace: counter | K-part sums [KP][T][5W] | kv [T][5W] | slice sums [T][4][NSL][3]
size_t engram_inject_ws_bytes(int T, int R, int W) {
  const int K = R * 256, KP = kv_parts(K);
  if (KP == 0) return 0;
  const size_t nsl = (size_t)(W + 255) / 256;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  return 256 + up((size_t)KP * T * 5 * W * 4) + up((size_t)T * 5 * W * 4) + up((size_t)T * 4 * nsl * 3 * 4);
}

cudaError_t launch_engram_inject(const uint8_t* table, long long n_rows, const int64_t* row_ids, int R,
                                 const uint16_t* w_kv, int W, uint16_t* resid, const float* q_norm,
                                 const float* k_norm, const uint8_t* mask, int T, float eps, float* kv_out,
                                 float* gate_out, int32_t* err, void* ws, cudaStream_t s) {
  const int K = R * 256, N = 5 * W, KP = kv_parts(K);
  if (KP == 0 || N % 16 != 0) return cudaErrorInvalidValue;
  int* counter = reinterpret_cast<int*>(ws);
  float* part = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + 256);
  // W_kv as [N][K] BF16, box 64 K x 16 rows, 128-byte swizzle
  struct Entry {
    const void* w;
    int K, N;
    CUtensorMap map;
  };
  static std::mutex mu;
  static Entry cache[8];
  static int n_cached = 0, next = 0;
  CUtensorMap map;
  {
    std::lock_guard<std::mutex> lock(mu);
    bool found = false;
    for (int i = 0; i < n_cached && !found; ++i)
      if (cache[i].w == w_kv && cache[i].K == K && cache[i].N == N) {
        map = cache[i].map;
        found = true;
      }
    if (!found) {
      const uint64_t dims[2] = {(uint64_t)K, (uint64_t)N};
      const uint64_t strides[1] = {(uint64_t)K * 2};
      const uint32_t box[2] = {64u, 16u};
      if (!encode_tiled(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_kv, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
      cache[next] = Entry{w_kv, K, N, map};
      next = (next + 1) % 8;
      if (n_cached < 8) ++n_cached;
    }
  }
  const size_t smem = 1024 + (size_t)KV_WARPS * KV_NS * KV_STAGE + (size_t)KV_WARPS * KV_NS * 8 + KV_WARPS * 16 +
                      (size_t)KV_TOK * (K + 8) * 2;
  if (smem > (size_t)device_max_smem_optin()) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(engram_kv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int sms = device_sm_count();
  for (int t0 = 0; t0 < T; t0 += KV_TOK) {
    KvParams p;
    p.table = table;
    p.n_rows = n_rows;
    p.row_ids = row_ids;
    p.R = R;
    p.T = T;
    p.t0 = t0;
    p.tg = T - t0 < KV_TOK ? T - t0 : KV_TOK;
    p.K = K;
    p.N = N;
    p.KP = KP;
    p.part = part;
    p.counter = counter;
    p.err = err;
    if (t0 > 0) {
      // each launch hands its items out from zero again
      const cudaError_t me = cudaMemsetAsync(counter, 0, sizeof(int), s);
      if (me != cudaSuccess) return me;
    }
    const cudaError_t le = launch_k(engram_kv_kernel, dim3(sms), dim3(KV_WARPS * 32), smem, s, map, p);
    if (le != cudaSuccess) return le;
  }
  GateParams gp;
  auto up = [](size_t v) { return (v + 255) & ~(size_t)255; };
  gp.part = part;
  gp.KP = KP;
  gp.T = T;
  gp.W = W;
  gp.NSL = (W + 255) / 256;
  gp.kv = kv_out ? kv_out : reinterpret_cast<float*>(reinterpret_cast<char*>(part) + up((size_t)KP * T * N * 4));
  gp.sums = reinterpret_cast<float*>(reinterpret_cast<char*>(part) + up((size_t)KP * T * N * 4) + up((size_t)T * N * 4));
  gp.resid = resid;
  gp.qn = q_norm;
  gp.kn = k_norm;
  gp.mask = mask;
  gp.eps = eps;
  gp.gate_out = gate_out;
  gp.counter = counter;
  {
    const cudaError_t le = launch_k(engram_reduce_kernel, dim3(T, 5 * gp.NSL), dim3(GATE_THREADS), 0, s, gp);
    if (le != cudaSuccess) return le;
  }
  {
    const cudaError_t le = launch_k(engram_apply_kernel, dim3(T, 4 * gp.NSL), dim3(GATE_THREADS), 0, s, gp);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

}  // namespace bre
