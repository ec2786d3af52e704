// Weighted combine (shared expert + routed sum, Strata-DSV4.1 README, V4-Flash "How it
// works", finish step), the residual update + RMS norm of a stack of MoE layers (verify
// batch, "Latest (2026-10-14)"), and the block dequantiser used to check the decode.
#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

namespace {

// out[t][c] = bf16(y_shared[t][c] + sum_j w[t,j] * y_pairs[inv[t*k+j]][c]), j ascending; four
// values per thread.  The routing entries of up to eight pairs, then their rows, are loaded
// before the FMAs, so that a token's loads are in flight together rather than one pair after
// another.
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y_pairs,
                                                      const float* __restrict__ topk_w,
                                                      const int32_t* __restrict__ inv,
                                                      const int32_t* __restrict__ offsets, int E,
                                                      const float* __restrict__ y_shared, int T, int k, int d,
                                                      uint16_t* __restrict__ out, float* __restrict__ out_f32) {
  pdl_wait();
  pdl_launch_dependents();   // the next launch waits for this grid before it reads anything
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int per_row = d / 4;
  if (i >= (long long)T * per_row) return;
  const int t = (int)(i / per_row), c = (int)(i % per_row) * 4;
  float4 acc = y_shared ? __ldg(reinterpret_cast<const float4*>(y_shared + (size_t)t * d + c))
                        : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  const int nvalid = __ldg(offsets + E);
  for (int j0 = 0; j0 < k; j0 += 8) {
    int pos[8];
    float w[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const bool in = j0 + q < k;
      pos[q] = in ? __ldg(inv + (size_t)t * k + j0 + q) : -1;
      w[q] = in ? __ldg(topk_w + (size_t)t * k + j0 + q) : 0.0f;
    }
    float4 y[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (pos[q] < 0 || pos[q] >= nvalid) pos[q] = -1;
      y[q] = pos[q] >= 0 ? __ldg(reinterpret_cast<const float4*>(y_pairs + (size_t)pos[q] * d + c))
                         : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (pos[q] >= 0) {
        acc.x = fmaf(w[q], y[q].x, acc.x);
        acc.y = fmaf(w[q], y[q].y, acc.y);
        acc.z = fmaf(w[q], y[q].z, acc.z);
        acc.w = fmaf(w[q], y[q].w, acc.w);
      }
    }
  }
  uint2 o;
  o.x = f32_to_bf16_rne(acc.x) | (f32_to_bf16_rne(acc.y) << 16);
  o.y = f32_to_bf16_rne(acc.z) | (f32_to_bf16_rne(acc.w) << 16);
  *reinterpret_cast<uint2*>(out + (size_t)t * d + c) = o;
  if (out_f32) *reinterpret_cast<float4*>(out_f32 + (size_t)t * d + c) = acc;
}

// One CTA per token: x_out = bf16(x + bf16(moe) * scale); the sum of squares of x_out in the
// router's 32-partial order; r = 1 / sqrtf(mean + eps); u = bf16(x_out * r).
__global__ void __launch_bounds__(256) residual_norm_kernel(const uint16_t* __restrict__ x,
                                                            const uint16_t* __restrict__ moe, int d, float scale,
                                                            float eps, uint16_t* __restrict__ x_out,
                                                            uint16_t* __restrict__ u_out) {
  extern __shared__ float xs[];  // [d]
  __shared__ float r_s;
  pdl_wait();
  pdl_launch_dependents();   // the next launch waits for this grid before it reads anything
  const int t = blockIdx.x;
  const uint16_t* xr = x + (size_t)t * d;
  const uint16_t* mr = moe + (size_t)t * d;
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    const float m = __fmul_rn(bf16_bits_to_f32(mr[c]), scale);
    const uint32_t b = f32_to_bf16_rne(__fadd_rn(bf16_bits_to_f32(xr[c]), m));
    x_out[(size_t)t * d + c] = (uint16_t)b;
    xs[c] = bf16_bits_to_f32(b);
  }
  __syncthreads();
  if (!u_out) return;
  if (threadIdx.x < 32) {
    const int j = threadIdx.x;
    float p = 0.0f;
    for (int c = j; c < d; c += 32) p = fmaf(xs[c], xs[c], p);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, o));
    if (j == 0) {
      const float mean = __fdiv_rn(p, (float)d);
      r_s = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
    }
  }
  __syncthreads();
  const float r = r_s;
  for (int c = threadIdx.x; c < d; c += blockDim.x) u_out[(size_t)t * d + c] = (uint16_t)f32_to_bf16_rne(__fmul_rn(xs[c], r));
}

__global__ void dequant_q2k_kernel(const uint8_t* __restrict__ blk, long long nblk, float* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nblk * 256) return;
  const long long b = i >> 8;
  const int w = (int)(i & 255);
  const uint8_t* p = blk + b * Q2K_BB;
  const float d = f16_bits_to_f32(p[80] | (p[81] << 8));
  const float dmin = f16_bits_to_f32(p[82] | (p[83] << 8));
  const int j = w >> 4;
  const uint32_t sc = p[j] & 15u, m = p[j] >> 4;
  const uint32_t q = (p[16 + (w >> 2)] >> (2 * (w & 3))) & 3u;
  const float a = __fmul_rn(__fmul_rn(d, (float)sc), (float)q);
  out[i] = __fsub_rn(a, __fmul_rn(dmin, (float)m));
}

__global__ void dequant_q80_kernel(const uint8_t* __restrict__ blk, long long nblk, float* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nblk * 32) return;
  const uint8_t* p = blk + (i >> 5) * Q80_BB;
  const float d = f16_bits_to_f32(p[0] | (p[1] << 8));
  out[i] = __fmul_rn(d, (float)(int8_t)p[2 + (i & 31)]);
}

}  // namespace

cudaError_t launch_combine(const float* y_pairs, const float* topk_w, const int32_t* inv, const int32_t* offsets,
                           int E, const float* y_shared, int T, int k, int d, uint16_t* out, float* out_f32,
                           cudaStream_t s) {
  const long long n = (long long)T * (d / 4);
  {
    const cudaError_t le = launch_k(combine_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, s, y_pairs,
                                    topk_w, inv, offsets, E, y_shared, T, k, d, out, out_f32);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_residual_norm(const uint16_t* x, const uint16_t* moe, int T, int d, float scale, float eps,
                                 uint16_t* x_out, uint16_t* u_out, cudaStream_t s) {
  const size_t smem = (size_t)d * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(residual_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  {
    const cudaError_t le = launch_k(residual_norm_kernel, dim3(T), dim3(256), smem, s, x, moe, d, scale, eps, x_out,
                                    u_out);
    if (le != cudaSuccess) return le;
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant(int fmt, const uint8_t* blocks, int64_t n_blocks, float* out, cudaStream_t s) {
  const long long n = n_blocks * (fmt == BRE_FMT_Q2_K ? 256 : 32);
  const unsigned grid = (unsigned)((n + 255) / 256);
  if (fmt == BRE_FMT_Q2_K)
    dequant_q2k_kernel<<<grid, 256, 0, s>>>(blocks, n_blocks, out);
  else
    dequant_q80_kernel<<<grid, 256, 0, s>>>(blocks, n_blocks, out);
  return cudaGetLastError();
}

}  // namespace bre
