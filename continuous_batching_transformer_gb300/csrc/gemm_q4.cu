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

}  // namespace

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
