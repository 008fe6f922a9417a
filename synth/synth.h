/*
 * synth.h -- seeded, counter-based generator for the synthetic workloads.
 *
 * This module produces INPUTS only (weights, token ids, lengths, KV contents).
 * It holds none of the transformer's arithmetic, and both the CPU oracle and
 * the CUDA path draw their inputs from it, so that the two sides see the same
 * bits.  Every function here is pure integer / IEEE-double code that gives the
 * same result on x86_64, aarch64 and the GPU:
 *
 *   syn_u64(seed, stream, index)   splitmix64 finaliser applied three times
 *                                  (Steele, Lea & Flood, "Fast splittable
 *                                  pseudorandom number generators", 2014).
 *   syn_normal(seed, stream, index)  Irwin-Hall sum of eight 16-bit uniforms
 *                                  drawn from two syn_u64 words, centred and
 *                                  scaled to unit variance.  Support is
 *                                  +-4.9 sigma.  Only integer adds, one
 *                                  exact int->double conversion and one
 *                                  double multiply, so host and device agree
 *                                  bit for bit.
 *   syn_bf16_from_double(x)        double -> float (round to nearest even,
 *                                  IEEE) -> bf16 (round to nearest even on
 *                                  the float bits).
 *   syn_uniform_int(u, n)          multiply-shift map of the top 32 bits of a
 *                                  word to [0, n).
 */
#ifndef CBT_SYNTH_H
#define CBT_SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_FN static __host__ __device__ __forceinline__
#else
#define SYN_FN static inline
#endif

SYN_FN uint64_t syn_mix64(uint64_t z) {
  z += 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* One 64-bit word for (seed, stream, index).  Counter based: any index can be
 * generated on its own, so host and device can fill the same tensor in any
 * order or layout. */
SYN_FN uint64_t syn_u64(uint64_t seed, uint64_t stream, uint64_t index) {
  uint64_t k = syn_mix64(seed ^ 0x243F6A8885A308D3ull);
  k = syn_mix64(k ^ stream);
  return syn_mix64(k ^ (index * 0xD1B54A32D192ED03ull));
}

/* Approximately standard normal: (sum of eight U{0..65535} - 8*32767.5)
 * scaled so that the variance is 1 (a U{0..65535} has variance
 * (65536^2 - 1)/12). */
SYN_FN double syn_normal(uint64_t seed, uint64_t stream, uint64_t index) {
  uint64_t a = syn_u64(seed, stream, 2 * index);
  uint64_t b = syn_u64(seed, stream, 2 * index + 1);
  int64_t s = 0;
  for (int i = 0; i < 4; ++i) {
    s += (int64_t)((a >> (16 * i)) & 0xFFFF);
    s += (int64_t)((b >> (16 * i)) & 0xFFFF);
  }
  /* 2*s - 8*65535 is an exact even integer; divide by 2 and by the standard
   * deviation sqrt(8*(65536^2-1)/12) = 53509.92 (a double constant). */
  double c = (double)(2 * s - 8 * 65535);
  return c * (0.5 / 53509.91992145008);
}

SYN_FN uint16_t syn_bf16_from_float_bits(uint32_t u) {
  if ((u & 0x7F800000u) == 0x7F800000u) {       /* inf or nan */
    return (uint16_t)((u >> 16) | ((u & 0x007FFFFFu) ? 0x40u : 0u));
  }
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;                            /* round to nearest even */
  return (uint16_t)(u >> 16);
}

SYN_FN uint16_t syn_bf16_from_double(double x) {
  float f = (float)x;
  union { float f; uint32_t u; } cv;
  cv.f = f;
  return syn_bf16_from_float_bits(cv.u);
}

SYN_FN uint32_t syn_uniform_int(uint64_t word, uint32_t n) {
  return (uint32_t)(((word >> 32) * (uint64_t)n) >> 32);
}

/* ---- stream ids: which tensor of which config a draw belongs to ---------- */
enum {
  SYN_EMBED = 1,
  SYN_LM_HEAD = 2,
  SYN_FINAL_NORM = 3,
  SYN_WQ = 16, SYN_WK, SYN_WV, SYN_WO, SYN_WG, SYN_WU, SYN_WD,
  SYN_ATTN_NORM, SYN_FFN_NORM
};

/* weight tensors: kind for the model-level tensors, (layer+1)<<8 | kind for
 * per-layer tensors */
SYN_FN uint64_t syn_stream_weight(int layer, int kind) {
  return layer < 0 ? (uint64_t)kind : (((uint64_t)(layer + 1)) << 8) | (uint64_t)kind;
}

/* synthetic KV contents of row `row`, layer, kv (0 = K, 1 = V), kv head;
 * index = pos * head_dim + dim */
SYN_FN uint64_t syn_stream_kv(int row, int layer, int kv, int head) {
  return (1ull << 48) | ((uint64_t)row << 24) | ((uint64_t)layer << 12) |
         ((uint64_t)kv << 8) | (uint64_t)head;
}

/* token ids of row `row` (index = position) */
SYN_FN uint64_t syn_stream_tokens(int row) { return (2ull << 48) | (uint64_t)row; }

/* scalar draws of a workload (lengths, arrival gaps): index = item number */
SYN_FN uint64_t syn_stream_misc(int what) { return (3ull << 48) | (uint64_t)what; }

#endif
