/*
 * synth_host.c -- host-side fills for the seeded synthetic inputs.
 * Inputs only: no transformer arithmetic lives here.  Built with
 * -ffp-contract=off so that mean + sigma*z rounds twice on every machine,
 * exactly as the device fill does with __dmul_rn/__dadd_rn.
 */
#include "synth.h"
#include <stddef.h>

static uint16_t affine_bf16(double mean, double sigma, double z) {
  double p = sigma * z;
  double s = mean + p;
  return syn_bf16_from_double(s);
}

/* out[i] = bf16(mean + sigma * normal(seed, stream, first + i)), i < n */
void syn_fill_normal_bf16(uint16_t* out, uint64_t n, uint64_t seed, uint64_t stream,
                          uint64_t first, double mean, double sigma) {
#pragma omp parallel for schedule(static)
  for (long long i = 0; i < (long long)n; ++i)
    out[i] = affine_bf16(mean, sigma, syn_normal(seed, stream, first + (uint64_t)i));
}

/* KV of one sequence in the layout [L][Hkv][n_tok][hd]; kv = 0 for K, 1 for V;
 * value = bf16(sigma * normal(seed, syn_stream_kv(row, l, kv, h), pos*hd + d)) */
void syn_fill_kv(uint16_t* out, int row, int kv, int L, int Hkv, int n_tok, int hd,
                 uint64_t seed, double sigma) {
  long long blocks = (long long)L * Hkv;
  long long per = (long long)n_tok * hd;
#pragma omp parallel for schedule(static)
  for (long long blk = 0; blk < blocks; ++blk) {
    int l = (int)(blk / Hkv), h = (int)(blk % Hkv);
    uint64_t st = syn_stream_kv(row, l, kv, h);
    uint16_t* o = out + blk * per;
    for (long long i = 0; i < per; ++i) o[i] = affine_bf16(0.0, sigma, syn_normal(seed, st, (uint64_t)i));
  }
}

/* token ids uniform in [0, vocab) */
void syn_fill_tokens(int32_t* out, uint64_t n, uint64_t seed, uint64_t stream, uint64_t first,
                     uint32_t vocab) {
  for (uint64_t i = 0; i < n; ++i)
    out[i] = (int32_t)syn_uniform_int(syn_u64(seed, stream, first + i), vocab);
}

/* integers uniform in [lo, hi] inclusive */
void syn_fill_uniform_int(int32_t* out, uint64_t n, uint64_t seed, uint64_t stream, int32_t lo,
                          int32_t hi) {
  for (uint64_t i = 0; i < n; ++i)
    out[i] = lo + (int32_t)syn_uniform_int(syn_u64(seed, stream, i), (uint32_t)(hi - lo + 1));
}

/* raw 64-bit words (for workload draws such as arrival gaps) */
void syn_fill_u64(uint64_t* out, uint64_t n, uint64_t seed, uint64_t stream) {
  for (uint64_t i = 0; i < n; ++i) out[i] = syn_u64(seed, stream, i);
}
