// gemm_q4.cu -- the device layout of 4-bit affine weights (groups of 64 columns, w = s * q + b
// with q in 0..15 and bf16 s, b) read by the decode projections (gemm_q4r.cu).
//
// The engine copies each matrix once, at creation, from the interchange format (uint32 words of
// eight codes, element 8j + t in bits 4t..4t+3 of word j; bf16 scales and biases
// [rows][cols / 64]) into a layout of its own: per (128-row tile, 128-column superblock) one
// contiguous 9 KB block,
//   [4 chunks][128 rows][16 bytes]  codes: chunk c of a row holds columns 32c .. 32c + 31 as
//                                   four words, word i's pair p = (bits 4p..4p+3: column 8i+2p,
//                                   bits 16+4p..19+4p: column 8i+2p+1), so one shift and one
//                                   logic op turn a pair into a 16-bit float pair with the codes
//                                   in its low mantissa bits;
//   [128 rows][s0, b0, s1, b1]      bf16 scale and bias of the block's two groups.
// SwiGLU tiles hold 64 gate rows and then the same 64 features' up rows, so one tile's
// epilogue sees a feature's gate and up values together.
//
// Prefill projections (more than 32 tokens) are dense contractions: there a matrix is expanded
// from the interchange format into bf16 hi and lo parts in engine scratch and the tensor-core
// GEMM runs over both.  w = s * q + b is formed once in fp32 (s * q is exact: 8 significant
// bits times 4; the sum rounds once), hi = bf16(w), lo = bf16(w - hi) (w - hi is exact), so
// hi + lo carries w to about 2^-17 of its magnitude.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kNK = 2;  // 64-column groups per block
constexpr int kCodeBytes = 128 * 64;

// One thread per tile row of one block; invalid rows (past the matrix) are zero codes with zero
// scale and bias, so they contribute nothing.
__global__ void k_q4_repack(const uint32_t* __restrict__ packed, const uint16_t* __restrict__ scales,
                            const uint16_t* __restrict__ biases, int M, int K, int F, int SB,
                            uint8_t* __restrict__ out) {
  const int blk = blockIdx.x, r = threadIdx.x;
  const int rb = blk / SB, sb = blk % SB;
  int src;
  bool valid;
  if (F > 0) {  // SwiGLU: gate rows, then the same features' up rows
    const int f = rb * 64 + (r & 63);
    valid = f < F;
    src = r < 64 ? f : F + f;
  } else {
    src = rb * 128 + r;
    valid = src < M;
  }
  uint8_t* dst = out + (size_t)blk * kQ4BlockBytes;
#pragma unroll 1
  for (int i = 0; i < 16; ++i) {  // word i: columns sb*128 + 8i .. + 7
    const uint32_t w = valid ? packed[(size_t)src * (K / 8) + sb * 16 + i] : 0u;
    uint32_t o = 0;
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
      o |= ((w >> (8 * pp)) & 0xFu) << (4 * pp);
      o |= ((w >> (8 * pp + 4)) & 0xFu) << (16 + 4 * pp);
    }
    // chunk i / 4 of row r, word i % 4
    reinterpret_cast<uint32_t*>(dst + (i >> 2) * 2048 + r * 16)[i & 3] = o;
  }
  uint16_t* sbd = reinterpret_cast<uint16_t*>(dst + kCodeBytes + r * 8);
#pragma unroll
  for (int jj = 0; jj < kNK; ++jj) {
    const size_t gi = (size_t)src * (K / 64) + sb * kNK + jj;
    sbd[2 * jj] = valid ? scales[gi] : (uint16_t)0;
    sbd[2 * jj + 1] = valid ? biases[gi] : (uint16_t)0;
  }
}

// One thread per word of eight codes (one row, eight consecutive columns inside one group);
// the eight hi parts and the eight lo parts leave as one 16-byte store each.
__global__ void k_q4_expand(const uint32_t* __restrict__ packed, const uint16_t* __restrict__ scales,
                            const uint16_t* __restrict__ biases, long long words, int K,
                            uint16_t* __restrict__ hi, uint16_t* __restrict__ lo) {
  const int wpr = K / 8;  // words per row
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < words;
       i += (long long)gridDim.x * blockDim.x) {
    const uint32_t w = __ldcs(packed + i);
    const long long row = i / wpr;
    const int col = (int)(i - row * wpr) * 8;
    const size_t gi = (size_t)row * (K / 64) + col / 64;
    const float sc = bf16_to_f32(scales[gi]), bi = bf16_to_f32(biases[gi]);
    uint32_t h[4], l[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const float v0 = fmaf(sc, (float)((w >> (8 * t)) & 15u), bi);
      const float v1 = fmaf(sc, (float)((w >> (8 * t + 4)) & 15u), bi);
      const uint16_t h0 = f32_to_bf16(v0), h1 = f32_to_bf16(v1);
      const uint16_t l0 = f32_to_bf16(v0 - bf16_to_f32(h0)), l1 = f32_to_bf16(v1 - bf16_to_f32(h1));
      h[t] = (uint32_t)h0 | ((uint32_t)h1 << 16);
      l[t] = (uint32_t)l0 | ((uint32_t)l1 << 16);
    }
    *reinterpret_cast<uint4*>(hi + i * 8) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + i * 8) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

}  // namespace

bool launch_q4_expand(const uint32_t* packed, const uint16_t* scales, const uint16_t* biases,
                      int M, int K, uint16_t* hi, uint16_t* lo, int num_sms, cudaStream_t s) {
  if (M <= 0 || K <= 0 || K % 64 || (reinterpret_cast<uintptr_t>(hi) & 15) ||
      (reinterpret_cast<uintptr_t>(lo) & 15))
    return false;
  const long long words = (long long)M * (K / 8);
  const long long want = (words + 255) / 256;
  const int grid = (int)std::min<long long>(want, (long long)num_sms * 16);
  k_q4_expand<<<grid, 256, 0, s>>>(packed, scales, biases, words, K, hi, lo);
  count_launch();
  return cudaGetLastError() == cudaSuccess;
}

size_t q4_native_bytes(int M, int K, int F) {
  if (K % 128) return 0;
  const int RB = F > 0 ? (F + 63) / 64 : (M + 127) / 128;
  return (size_t)RB * (K / 128) * kQ4BlockBytes;
}

bool launch_q4_repack(const uint32_t* packed, const uint16_t* scales, const uint16_t* biases,
                      int M, int K, int F, uint8_t* out, cudaStream_t s) {
  if (K % 128 || M <= 0 || (F > 0 && M != 2 * F)) return false;
  const int RB = F > 0 ? (F + 63) / 64 : (M + 127) / 128;
  const int SB = K / 128;
  k_q4_repack<<<RB * SB, 128, 0, s>>>(packed, scales, biases, M, K, F, SB, out);
  count_launch();
  return cudaGetLastError() == cudaSuccess;
}
