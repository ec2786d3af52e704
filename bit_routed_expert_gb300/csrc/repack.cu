// Q2_K -> Q2_K_R16: the routed experts' blocks regrouped into 1344-byte tiles of 16 rows.
//
// The bytes of every block are kept (a permutation at the level of 2-bit codes and 4-bit
// nibbles; the tile is exactly the 16 blocks' 1,344 bytes), so the layout holds the same Q2_K
// weights as the block format of the strix-llama.cpp issue ("Feature Description", Q2_K experts):
// w = d * sc * q - dmin * m.  What changes is where each field sits, so that the expert FFN's
// warps read their tensor-core fragment data with one 16-byte load per lane and a row's codes
// of one sub-block pair come out of one 32-bit word with a mask.
//
// Tile of rows 16 * rt .. 16 * rt + 15 and block b (256 weights) of one matrix, at byte offset
// (rt * nb + b) * 1344; inside it, row R = 8 * rr + g (g < 8) and lane L = 4 * g + t (t < 4):
//   [rr * 512 + 16 * L, +16)  codes of row R for sub-blocks 4t .. 4t+3, as four words
//                             W(p, w), p, w in {0, 1}, at word 2p + w: bits 16h + 2s hold code
//                             8w + s of sub-block 4t + 2p + h (h in {0, 1}, s < 8)
//   [1024 + 8 * L, +8)        two words: the scales (low nibbles) then the mins (high nibbles)
//                             of rows g and g + 8 for sub-blocks 4t .. 4t+3; the nibble of
//                             (row 8 rr' + g, sub-block 4t + 2p + h) sits at bit 16h + 4(2rr' + p)
//   [1280 + 8 * g + 4 * rr, +4)  fp16 d then fp16 dmin of row R
#include <cuda_runtime.h>

#include "bre_common.cuh"
#include "kernels.h"

namespace bre {

namespace {

// One thread per (tile, block, lane): it reads rows g and g + 8 of the block and writes the
// lane's codes of both rows, its scale and min words and (t == 0) the rows' d and dmin.
__global__ void __launch_bounds__(256) repack_q2k_r16_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                                             long long n_mat, long long units, int nb,
                                                             long long row_bytes, long long src_stride,
                                                             long long dst_stride) {
  const long long gid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long ug = gid >> 5;
  if (ug >= n_mat * units) return;
  const long long mat = ug / units, unit = ug - mat * units;
  const int L = (int)(gid & 31), g = L >> 2, t = L & 3;
  const long long rt = unit / nb;
  const int b = (int)(unit - rt * nb);
  src += mat * src_stride;
  uint8_t* out = dst + mat * dst_stride + unit * 1344;
  uint32_t sc_word = 0, m_word = 0;
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const uint8_t* blk = src + (rt * 16 + 8 * rr + g) * row_bytes + (long long)b * Q2K_BB;
    uint32_t words[4];
#pragma unroll
    for (int p = 0; p < 2; ++p)
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        uint32_t v = 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = 4 * t + 2 * p + h;
          // codes 8w .. 8w+7 of sub-block j: bytes qs[4j + 2w], qs[4j + 2w + 1] (four codes each,
          // code i at bits 2 (i % 4) of qs[i / 4]) -- already the little-endian 2-bit order
          const uint32_t lo = blk[16 + 4 * j + 2 * w], hi = blk[16 + 4 * j + 2 * w + 1];
          v |= (lo | (hi << 8)) << (16 * h);
          const uint32_t sb = blk[j];
          const int pos = 16 * h + 4 * (2 * rr + p);
          if (w == 0) {
            sc_word |= (sb & 15u) << pos;
            m_word |= (sb >> 4) << pos;
          }
        }
        words[2 * p + w] = v;
      }
    *reinterpret_cast<uint4*>(out + rr * 512 + 16 * L) = make_uint4(words[0], words[1], words[2], words[3]);
    if (t == 0) {
      const uint32_t dd = blk[80] | (blk[81] << 8) | (blk[82] << 16) | ((uint32_t)blk[83] << 24);
      *reinterpret_cast<uint32_t*>(out + 1280 + 8 * g + 4 * rr) = dd;
    }
  }
  *reinterpret_cast<uint2*>(out + 1024 + 8 * L) = make_uint2(sc_word, m_word);
}

}  // namespace

cudaError_t launch_repack_q2k_r16(const uint8_t* src, uint8_t* dst, long long n_mat, int rows, int cols,
                                  long long src_stride, long long dst_stride, cudaStream_t s) {
  const int nb = cols / 256;
  const long long row_bytes = (long long)nb * Q2K_BB;
  const long long units = (long long)(rows / 16) * nb;
  const long long threads = n_mat * units * 32;
  const long long grid = (threads + 255) / 256;
  if (grid <= 0 || grid > 0x7FFFFFFFLL) return cudaErrorInvalidValue;
  repack_q2k_r16_kernel<<<(unsigned)grid, 256, 0, s>>>(src, dst, n_mat, units, nb, row_bytes, src_stride, dst_stride);
  return cudaGetLastError();
}

}  // namespace bre
