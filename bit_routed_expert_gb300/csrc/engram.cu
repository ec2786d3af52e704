// Engram gather-decode: 264-byte rows (256 E4M3 values + 8 E8M0 scales) gathered by
// row id, decoded to FP32, summed over heads in order and rounded to BF16.
// (strix-llama.cpp issue, "Feature Description" and "DeepSeek V4.1 Engram graph
// integration".)
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
  if (H == 1)
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

}  // namespace bre
