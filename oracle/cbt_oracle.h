/*
 * cbt_oracle.h -- plain CPU oracle of the continuous-batching decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link or call
 * this library: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code with the CUDA path.
 *
 * What it computes, and where the pages define it (gnosis "Continuous Decode
 * Batching -- the transformer capture", sections "REVISED: the hard kernel
 * already exists -- forward_batch_segmented" and "decode_step_batch --
 * paint-by-numbers"):
 *   - a pre-norm decoder: embed; per layer RMSNorm, Q/K/V projections, RoPE of
 *     q and k at the token's own position, K/V saved into the sequence's own
 *     cache at that position, causal softmax attention over positions [0, pos]
 *     of the sequence's own cache (grouped-query: q head j reads kv head
 *     j / (n_heads / n_kv_heads)), output projection + residual, RMSNorm,
 *     SwiGLU FFN + residual; final RMSNorm and lm_head.
 *   - decode_step_batch(seq_ids, last_tokens) -> logits[B]: one token per
 *     sequence at that sequence's position t_s, attending [0, t_s], appending
 *     K/V at t_s and bumping t_s ("Delta 1..3" of the same page).
 *   - forward_batch_segmented(tokens, seg_lens): K prompts packed in one pass;
 *     token g of a segment starting at seg_start attends only [seg_start, g],
 *     i.e. positions [0, g - seg_start] of its own sequence, RoPE at the
 *     segment-local position.
 *   - greedy argmax with the lowest vocabulary id winning ties (mlx-bun
 *     batching.md v0.4.0 campaign notes: "lowest vocabulary ID among tied
 *     candidate scores").
 *
 * Precision: activations are stored in fp32 (the page's "f32-act precision
 * discipline"); every dot product, norm, softmax and rotation is evaluated
 * in double and rounded to fp32 when stored.  K and V are rounded to bf16
 * when appended (the KV cache holds bf16).  Weights are bf16 values (or the
 * exact affine dequantisation scale*q + bias of 4-bit codes).
 */
#ifndef CBT_ORACLE_H
#define CBT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int n_layers, d_model, n_heads, n_kv_heads, head_dim, d_ff, vocab;
  double rms_eps, rope_theta;
  int weight_format; /* 0 = bf16 [out][in]; 1 = 4-bit affine, groups along `in` */
  int group_size;    /* 4-bit affine only */
} orc_config;

typedef struct {
  const uint16_t* w;      /* bf16 bits [out][in]                         (format 0) */
  const uint32_t* packed; /* [out][in/8], element 8j+k in bits 4k..4k+3  (format 1) */
  const uint16_t* scales; /* bf16 [out][in/group]                        (format 1) */
  const uint16_t* biases; /* bf16 [out][in/group]                        (format 1) */
} orc_linear;

typedef struct {
  orc_linear wq, wk, wv, wo, wg, wu, wd;
  const uint16_t* attn_norm; /* bf16 [d_model] */
  const uint16_t* ffn_norm;  /* bf16 [d_model] */
} orc_layer;

typedef struct {
  orc_config cfg;
  const uint16_t* embed;      /* bf16 [vocab][d_model] */
  orc_linear lm_head;         /* [vocab][d_model] */
  const uint16_t* final_norm; /* bf16 [d_model] */
  const orc_layer* layers;    /* [n_layers] */
} orc_model;

/* One sequence's KV cache: bf16 bits, layout [n_layers][n_kv_heads][capacity][head_dim]. */
typedef struct {
  int capacity;
  int len; /* positions [0, len) hold valid K/V */
  uint16_t* k;
  uint16_t* v;
  /* Affine KV of `bits` = 8 or 4 bits (the mlx-bun batching design's quantised KV, "--kv-quant
   * 4|8": affine groups of 64 along head_dim, as its weights).  kq == NULL: a plain bf16
   * cache.  Otherwise codes [n_layers][n_kv_heads][capacity][head_dim * bits / 8] and bf16
   * scale/bias [n_layers][n_kv_heads][capacity][head_dim/64] for K and V.  A sequence's first
   * call runs on its bf16 K/V and is then converted (the design's "prefill bf16, then to
   * quantized"); from then on (qlen > 0) every appended position is quantised at once and
   * attention reads every position through its codes.  Positions [0, qlen) hold codes. */
  uint8_t* kq;
  uint8_t* vq;
  uint16_t* ks;
  uint16_t* kb;
  uint16_t* vs;
  uint16_t* vb;
  int qlen;
  int bits;
} orc_kv;

/* status codes */
#define ORC_OK 0
#define ORC_EINVAL -1

/* ---- building blocks (exported so tests can pin each one) -------------------- */
float orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f); /* round to nearest even */
void orc_rmsnorm(const float* x, const uint16_t* gain, int n, double eps, float* out);
void orc_rope(float* vec, int head_dim, int pos, double theta);
void orc_attention(const float* q, const uint16_t* k, const uint16_t* v, int n_keys,
                   int head_dim, float* out);
double orc_silu(double z);
void orc_linear_apply(const orc_config* cfg, const orc_linear* lin, int out_dim, int in_dim,
                      const float* x, int n, float* y);
int orc_argmax(const float* logits, int vocab);
int orc_quantize_affine4(const uint16_t* w, int rows, int cols, int group, uint32_t* packed,
                         uint16_t* scales, uint16_t* biases);
void orc_dequantize_affine4(const uint32_t* packed, const uint16_t* scales,
                            const uint16_t* biases, int rows, int cols, int group, double* out);
/* Affine KV rows of `bits` = 8 or 4: per group of 64 values of a row, L = 2^bits - 1,
 * scale = bf16((max - min) / L), bias = bf16(min), q = clamp(rint((x - bias) / scale), 0, L)
 * (q = 0 when scale = 0); the value read back is scale * q + bias.  cols must be a multiple of
 * 64; a row's codes take cols * bits / 8 bytes (4 bits: element 2i in the low nibble of byte i,
 * 2i + 1 in its high nibble). */
int orc_quantize_kv(const uint16_t* x, int rows, int cols, int bits, uint8_t* codes,
                    uint16_t* scales, uint16_t* biases);
int orc_quantize_kv8(const uint16_t* x, int rows, int cols, uint8_t* codes, uint16_t* scales,
                     uint16_t* biases);
/* attention of one query over n_keys quantised K/V rows (codes [n][hd * bits / 8],
 * scale/bias [n][hd/64]) */
void orc_attention_kvq(const float* q, const uint8_t* kq, const uint16_t* ks, const uint16_t* kb,
                       const uint8_t* vq, const uint16_t* vs, const uint16_t* vb, int n_keys,
                       int head_dim, int bits, float* out);
void orc_attention_kv8(const float* q, const uint8_t* kq, const uint16_t* ks, const uint16_t* kb,
                       const uint8_t* vq, const uint16_t* vs, const uint16_t* vb, int n_keys,
                       int head_dim, float* out);
/* quantise positions [qlen, len) of a quantised cache from its bf16 rows; qlen becomes len */
int orc_kv_convert(const orc_config* cfg, orc_kv* kv);
/* What export gives for a quantised position (a reading of the pages, which define no export):
 * scale * code + bias in double, rounded to fp32 and then to bf16. */
uint16_t orc_kvq_export_value(uint16_t scale, uint16_t bias, int code);

/* ---- the model ------------------------------------------------------------------ */
/* General forward: n tokens; token i belongs to cache kv[seq[i]] at position pos[i] and
 * attends to positions [0, pos[i]] of that cache.  The tokens of one sequence must appear
 * in increasing, consecutive positions starting at that cache's len.  Logits are written
 * for tokens with want[i] != 0, one row of `vocab` floats each, in token order. */
int orc_forward(const orc_model* m, orc_kv* kv, int n_kv, int n, const int* seq, const int* pos,
                const int* tok, const int* want, float* logits);

/* decode_step_batch: one token per row at the row's current length; logits [B][vocab] */
int orc_decode_step_batch(const orc_model* m, orc_kv* kv, int B, const int* last_tokens,
                          float* logits);

/* forward_batch_segmented: K prompts packed back to back (tokens[sum seg_lens]); every cache
 * must be empty; logits of each segment's last token, [K][vocab] */
int orc_prefill_segmented(const orc_model* m, orc_kv* kv, int K, const int* seg_lens,
                          const int* tokens, float* logits);

/* one sequence alone: prompt prefill (len tokens from position kv->len) */
int orc_prefill_sequence(const orc_model* m, orc_kv* kv, int len, const int* tokens,
                         float* logits_last);

/* threads the oracle's OpenMP loops use */
int orc_num_threads(void);
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
