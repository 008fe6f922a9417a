/*
 * cbt_oracle.c -- plain CPU oracle of the continuous-batching decode step.
 *
 * TEST INFRASTRUCTURE ONLY (see cbt_oracle.h): called by the test suite, the
 * smoke check and the benchmark's CPU-baseline leg, never by the product.
 *
 * Written for obviousness, not speed: every reduction is a straight loop in
 * double, in index order.  The only parallelism is OpenMP over independent
 * output elements (rows of a projection, heads of an attention), which does
 * not change any result.  Built with -ffp-contract=off so no multiply-add is
 * fused and results are identical on x86_64 and aarch64.
 */
#include "cbt_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- bf16 <-> fp32 ------------------------------------------------------------- */
float orc_bf16_to_f32(uint16_t b) {
  union { uint32_t u; float f; } c;
  c.u = ((uint32_t)b) << 16;
  return c.f;
}

uint16_t orc_f32_to_bf16(float f) {
  union { uint32_t u; float f; } c;
  c.f = f;
  uint32_t u = c.u;
  if ((u & 0x7F800000u) == 0x7F800000u) return (uint16_t)((u >> 16) | ((u & 0x7FFFFFu) ? 0x40u : 0u));
  /* round to nearest, ties to even, on the 16 discarded bits */
  uint32_t keep = u >> 16, rest = u & 0xFFFFu;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
  return (uint16_t)keep;
}

/* ---- RMSNorm: x / sqrt(mean(x^2) + eps) * gain --------------------------------- */
void orc_rmsnorm(const float* x, const uint16_t* gain, int n, double eps, float* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += (double)x[i] * (double)x[i];
  double r = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; ++i) out[i] = (float)((double)x[i] * r * (double)orc_bf16_to_f32(gain[i]));
}

/* ---- RoPE, rotate-half form: pair (i, i + hd/2) rotated by pos * theta^(-2i/hd) ---- */
void orc_rope(float* vec, int head_dim, int pos, double theta) {
  int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    double freq = pow(theta, -2.0 * (double)i / (double)head_dim);
    double ang = (double)pos * freq;
    double c = cos(ang), s = sin(ang);
    double a = vec[i], b = vec[i + half];
    vec[i] = (float)(a * c - b * s);
    vec[i + half] = (float)(a * s + b * c);
  }
}

/* ---- softmax attention of one query over n_keys cached keys/values ----------------- */
/* softmax(q.K^T / sqrt(hd)) V over n_keys rows of K and V given as doubles */
static void attention_values(const float* q, const double* k, const double* v, int n_keys,
                             int head_dim, float* out) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
  double inv_sqrt = 1.0 / sqrt((double)head_dim);
  double mx = -INFINITY;
  for (int t = 0; t < n_keys; ++t) {
    double dot = 0.0;
    for (int d = 0; d < head_dim; ++d) dot += (double)q[d] * k[(size_t)t * head_dim + d];
    s[t] = dot * inv_sqrt;
    if (s[t] > mx) mx = s[t];
  }
  double z = 0.0;
  for (int t = 0; t < n_keys; ++t) {
    s[t] = exp(s[t] - mx);
    z += s[t];
  }
  for (int d = 0; d < head_dim; ++d) {
    double acc = 0.0;
    for (int t = 0; t < n_keys; ++t) acc += s[t] * v[(size_t)t * head_dim + d];
    out[d] = (float)(acc / z);
  }
  free(s);
}

void orc_attention(const float* q, const uint16_t* k, const uint16_t* v, int n_keys,
                   int head_dim, float* out) {
  size_t n = (size_t)(n_keys > 0 ? n_keys : 1) * head_dim;
  double* kd = (double*)malloc(sizeof(double) * n);
  double* vd = (double*)malloc(sizeof(double) * n);
  for (size_t i = 0; i < (size_t)n_keys * head_dim; ++i) {
    kd[i] = orc_bf16_to_f32(k[i]);
    vd[i] = orc_bf16_to_f32(v[i]);
  }
  attention_values(q, kd, vd, n_keys, head_dim, out);
  free(kd);
  free(vd);
}

/* ---- affine KV, 8 or 4 bits: x^ = scale * q + bias per group of 64 along head_dim ------ */
/* Codes of a row of `cols` values take cols * bits / 8 bytes; at 4 bits element 2i sits in the
 * low nibble of byte i and element 2i + 1 in its high nibble (the weights' packing order). */
static int kv_code(const uint8_t* codes, int cols, int bits, size_t row, int i) {
  if (bits == 8) return codes[row * (size_t)cols + i];
  const uint8_t byte = codes[row * (size_t)(cols / 2) + i / 2];
  return (i & 1) ? (byte >> 4) : (byte & 0xF);
}

int orc_quantize_kv(const uint16_t* x, int rows, int cols, int bits, uint8_t* codes,
                    uint16_t* scales, uint16_t* biases) {
  if (rows < 0 || cols <= 0 || cols % 64 != 0 || (bits != 8 && bits != 4)) return ORC_EINVAL;
  const int ng = cols / 64;
  const int levels = (1 << bits) - 1;
  const size_t row_bytes = (size_t)cols * bits / 8;
  for (int r = 0; r < rows; ++r) {
    memset(codes + (size_t)r * row_bytes, 0, row_bytes);
    for (int g = 0; g < ng; ++g) {
      const uint16_t* src = x + (size_t)r * cols + (size_t)g * 64;
      double mn = orc_bf16_to_f32(src[0]), mx = mn;
      for (int i = 1; i < 64; ++i) {
        double v = orc_bf16_to_f32(src[i]);
        if (v < mn) mn = v;
        if (v > mx) mx = v;
      }
      uint16_t sb = orc_f32_to_bf16((float)((mx - mn) / (double)levels));
      uint16_t bb = orc_f32_to_bf16((float)mn);
      double sc = orc_bf16_to_f32(sb), bi = orc_bf16_to_f32(bb);
      scales[(size_t)r * ng + g] = sb;
      biases[(size_t)r * ng + g] = bb;
      for (int i = 0; i < 64; ++i) {
        int q = 0;
        if (sc != 0.0) {
          double t = rint(((double)orc_bf16_to_f32(src[i]) - bi) / sc);
          q = t < 0.0 ? 0 : (t > (double)levels ? levels : (int)t);
        }
        const int e = g * 64 + i;
        if (bits == 8)
          codes[(size_t)r * row_bytes + e] = (uint8_t)q;
        else
          codes[(size_t)r * row_bytes + e / 2] |= (uint8_t)(q << (4 * (e & 1)));
      }
    }
  }
  return ORC_OK;
}

int orc_quantize_kv8(const uint16_t* x, int rows, int cols, uint8_t* codes, uint16_t* scales,
                     uint16_t* biases) {
  return orc_quantize_kv(x, rows, cols, 8, codes, scales, biases);
}

static double kvq_value(const uint8_t* codes, const uint16_t* scales, const uint16_t* biases,
                        int hd, int bits, int t, int d) {
  size_t gi = (size_t)t * (hd / 64) + d / 64;
  return (double)orc_bf16_to_f32(scales[gi]) * kv_code(codes, hd, bits, (size_t)t, d) +
         (double)orc_bf16_to_f32(biases[gi]);
}

void orc_attention_kvq(const float* q, const uint8_t* kq, const uint16_t* ks, const uint16_t* kb,
                       const uint8_t* vq, const uint16_t* vs, const uint16_t* vb, int n_keys,
                       int head_dim, int bits, float* out) {
  size_t n = (size_t)(n_keys > 0 ? n_keys : 1) * head_dim;
  double* kd = (double*)malloc(sizeof(double) * n);
  double* vd = (double*)malloc(sizeof(double) * n);
  for (int t = 0; t < n_keys; ++t)
    for (int d = 0; d < head_dim; ++d) {
      kd[(size_t)t * head_dim + d] = kvq_value(kq, ks, kb, head_dim, bits, t, d);
      vd[(size_t)t * head_dim + d] = kvq_value(vq, vs, vb, head_dim, bits, t, d);
    }
  attention_values(q, kd, vd, n_keys, head_dim, out);
  free(kd);
  free(vd);
}

void orc_attention_kv8(const float* q, const uint8_t* kq, const uint16_t* ks, const uint16_t* kb,
                       const uint8_t* vq, const uint16_t* vs, const uint16_t* vb, int n_keys,
                       int head_dim, float* out) {
  orc_attention_kvq(q, kq, ks, kb, vq, vs, vb, n_keys, head_dim, 8, out);
}

/* the value an exported position of a quantised cache holds: scale * code + bias evaluated
 * in double, rounded to fp32, then to bf16 */
uint16_t orc_kvq_export_value(uint16_t scale, uint16_t bias, int code) {
  double v = (double)orc_bf16_to_f32(scale) * code + (double)orc_bf16_to_f32(bias);
  return orc_f32_to_bf16((float)v);
}

double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* ---- 4-bit affine weights: ŵ = scale * q + bias per group along `in` -------------- */
static double deq_one(const orc_linear* lin, int in_dim, int group, int o, int i) {
  uint32_t word = lin->packed[(size_t)o * (in_dim / 8) + i / 8];
  int q = (int)((word >> (4 * (i % 8))) & 0xFu);
  size_t gi = (size_t)o * (in_dim / group) + i / group;
  return (double)orc_bf16_to_f32(lin->scales[gi]) * q + (double)orc_bf16_to_f32(lin->biases[gi]);
}

/* y[r][o] = sum_i W[o][i] * x[r][i], r < n: each weight row is read once for all n rows
 * (the batched form: one weight read serves the whole wave). */
void orc_linear_apply(const orc_config* cfg, const orc_linear* lin, int out_dim, int in_dim,
                      const float* x, int n, float* y) {
#pragma omp parallel
  {
    double* wrow = (double*)malloc(sizeof(double) * (size_t)in_dim);
#pragma omp for schedule(static)
    for (int o = 0; o < out_dim; ++o) {
      if (cfg->weight_format == 0) {
        const uint16_t* w = lin->w + (size_t)o * in_dim;
        for (int i = 0; i < in_dim; ++i) wrow[i] = (double)orc_bf16_to_f32(w[i]);
      } else {
        for (int i = 0; i < in_dim; ++i) wrow[i] = deq_one(lin, in_dim, cfg->group_size, o, i);
      }
      for (int r = 0; r < n; ++r) {
        const float* xr = x + (size_t)r * in_dim;
        double acc = 0.0;
        for (int i = 0; i < in_dim; ++i) acc += wrow[i] * (double)xr[i];
        y[(size_t)r * out_dim + o] = (float)acc;
      }
    }
    free(wrow);
  }
}

/* greedy sampler: the largest logit, lowest index among equal values */
int orc_argmax(const float* logits, int vocab) {
  int best = 0;
  for (int i = 1; i < vocab; ++i)
    if (logits[i] > logits[best]) best = i;
  return best;
}

/* MLX-style affine quantisation, groups of `group` along each row:
 *   scale = bf16((max - min) / 15), bias = bf16(min),
 *   q = clamp(rint((w - bias) / scale), 0, 15)  (ties to even; q = 0 when scale == 0),
 *   packed word j of a row holds elements 8j..8j+7, element 8j+k in bits 4k..4k+3. */
int orc_quantize_affine4(const uint16_t* w, int rows, int cols, int group, uint32_t* packed,
                         uint16_t* scales, uint16_t* biases) {
  if (group <= 0 || cols % group != 0 || group % 8 != 0) return ORC_EINVAL;
  int ng = cols / group;
  /* rows are independent: the loop over them may run in any order */
#pragma omp parallel for schedule(static)
  for (int r = 0; r < rows; ++r) {
    for (int g = 0; g < ng; ++g) {
      const uint16_t* src = w + (size_t)r * cols + (size_t)g * group;
      double mn = orc_bf16_to_f32(src[0]), mx = mn;
      for (int i = 1; i < group; ++i) {
        double x = orc_bf16_to_f32(src[i]);
        if (x < mn) mn = x;
        if (x > mx) mx = x;
      }
      uint16_t sb = orc_f32_to_bf16((float)((mx - mn) / 15.0));
      uint16_t bb = orc_f32_to_bf16((float)mn);
      double sc = orc_bf16_to_f32(sb), bi = orc_bf16_to_f32(bb);
      scales[(size_t)r * ng + g] = sb;
      biases[(size_t)r * ng + g] = bb;
      for (int j = 0; j < group / 8; ++j) {
        uint32_t word = 0;
        for (int k = 0; k < 8; ++k) {
          double x = orc_bf16_to_f32(src[8 * j + k]);
          int q = 0;
          if (sc != 0.0) {
            double t = rint((x - bi) / sc);
            q = t < 0.0 ? 0 : (t > 15.0 ? 15 : (int)t);
          }
          word |= ((uint32_t)q) << (4 * k);
        }
        packed[(size_t)r * (cols / 8) + (size_t)g * (group / 8) + j] = word;
      }
    }
  }
  return ORC_OK;
}

void orc_dequantize_affine4(const uint32_t* packed, const uint16_t* scales,
                            const uint16_t* biases, int rows, int cols, int group, double* out) {
  orc_linear lin = {0, packed, scales, biases};
  for (int r = 0; r < rows; ++r)
    for (int i = 0; i < cols; ++i) out[(size_t)r * cols + i] = deq_one(&lin, cols, group, r, i);
}

/* ---- the decoder ---------------------------------------------------------------- */
static size_t kv_index(const orc_config* c, int cap, int layer, int kvh, int pos) {
  return ((((size_t)layer * c->n_kv_heads + kvh) * cap) + pos) * (size_t)c->head_dim;
}

/* quantise the K and V rows at (layer, kv head, position) of a quantised cache */
static void kvq_store(const orc_config* c, orc_kv* C, int l, int g, int p) {
  size_t at = kv_index(c, C->capacity, l, g, p), ga = at / 64, ca = at * C->bits / 8;
  orc_quantize_kv(C->k + at, 1, c->head_dim, C->bits, C->kq + ca, C->ks + ga, C->kb + ga);
  orc_quantize_kv(C->v + at, 1, c->head_dim, C->bits, C->vq + ca, C->vs + ga, C->vb + ga);
}

int orc_kv_convert(const orc_config* c, orc_kv* kv) {
  if (!kv->kq || c->head_dim % 64 != 0 || (kv->bits != 8 && kv->bits != 4)) return ORC_EINVAL;
  for (int l = 0; l < c->n_layers; ++l)
    for (int g = 0; g < c->n_kv_heads; ++g)
      for (int p = kv->qlen; p < kv->len; ++p) kvq_store(c, kv, l, g, p);
  kv->qlen = kv->len;
  return ORC_OK;
}

int orc_forward(const orc_model* m, orc_kv* kv, int n_kv, int n, const int* seq, const int* pos,
                const int* tok, const int* want, float* logits) {
  const orc_config* c = &m->cfg;
  const int d = c->d_model, hd = c->head_dim, H = c->n_heads, Hkv = c->n_kv_heads;
  const int qd = H * hd, kvd = Hkv * hd, F = c->d_ff, V = c->vocab;
  if (n < 0 || H % Hkv != 0 || hd % 2 != 0) return ORC_EINVAL;
  for (int s = 0; s < n_kv; ++s)
    if (kv[s].kq && (hd % 64 != 0 || (kv[s].bits != 8 && kv[s].bits != 4))) return ORC_EINVAL;
  /* each sequence's tokens: consecutive positions from its current length, inside capacity */
  int* next = (int*)malloc(sizeof(int) * (size_t)(n_kv > 0 ? n_kv : 1));
  for (int s = 0; s < n_kv; ++s) next[s] = kv[s].len;
  for (int i = 0; i < n; ++i) {
    int s = seq[i];
    if (s < 0 || s >= n_kv || pos[i] != next[s] || pos[i] >= kv[s].capacity || tok[i] < 0 ||
        tok[i] >= V) {
      free(next);
      return ORC_EINVAL;
    }
    next[s]++;
  }
  /* 8-bit caches that already hold codes quantise what this call appends and read codes */
  int* quant = (int*)malloc(sizeof(int) * (size_t)(n_kv > 0 ? n_kv : 1));
  for (int s = 0; s < n_kv; ++s) quant[s] = kv[s].kq != NULL && kv[s].qlen > 0;
  float* x = (float*)malloc(sizeof(float) * (size_t)n * d);
  float* h = (float*)malloc(sizeof(float) * (size_t)n * d);
  float* q = (float*)malloc(sizeof(float) * (size_t)n * qd);
  float* k = (float*)malloc(sizeof(float) * (size_t)n * kvd);
  float* v = (float*)malloc(sizeof(float) * (size_t)n * kvd);
  float* o = (float*)malloc(sizeof(float) * (size_t)n * qd);
  float* a = (float*)malloc(sizeof(float) * (size_t)n * d);
  float* gt = (float*)malloc(sizeof(float) * (size_t)n * F);
  float* up = (float*)malloc(sizeof(float) * (size_t)n * F);

  /* embed */
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < d; ++j) x[(size_t)i * d + j] = orc_bf16_to_f32(m->embed[(size_t)tok[i] * d + j]);

  for (int l = 0; l < c->n_layers; ++l) {
    const orc_layer* L = &m->layers[l];
    /* attention block: batched projections over all n tokens (weights read once) */
    for (int i = 0; i < n; ++i) orc_rmsnorm(x + (size_t)i * d, L->attn_norm, d, c->rms_eps, h + (size_t)i * d);
    orc_linear_apply(c, &L->wq, qd, d, h, n, q);
    orc_linear_apply(c, &L->wk, kvd, d, h, n, k);
    orc_linear_apply(c, &L->wv, kvd, d, h, n, v);
    /* per-token loop: RoPE at the token's own position, save K/V into its own cache at that
     * position, attention over [0, pos] of its own cache */
    for (int i = 0; i < n; ++i) {
      orc_kv* C = &kv[seq[i]];
      int p = pos[i];
      for (int j = 0; j < H; ++j) orc_rope(q + (size_t)i * qd + (size_t)j * hd, hd, p, c->rope_theta);
      for (int g = 0; g < Hkv; ++g) {
        float* kk = k + (size_t)i * kvd + (size_t)g * hd;
        float* vv = v + (size_t)i * kvd + (size_t)g * hd;
        orc_rope(kk, hd, p, c->rope_theta);
        size_t at = kv_index(c, C->capacity, l, g, p);
        for (int e = 0; e < hd; ++e) {
          C->k[at + e] = orc_f32_to_bf16(kk[e]);
          C->v[at + e] = orc_f32_to_bf16(vv[e]);
        }
        if (quant[seq[i]]) kvq_store(c, C, l, g, p);
      }
      const int qm = quant[seq[i]];
#pragma omp parallel for schedule(static)
      for (int j = 0; j < H; ++j) {
        int g = j / (H / Hkv);
        size_t base = kv_index(c, C->capacity, l, g, 0);
        if (qm)
          orc_attention_kvq(q + (size_t)i * qd + (size_t)j * hd, C->kq + base * C->bits / 8,
                            C->ks + base / 64, C->kb + base / 64, C->vq + base * C->bits / 8,
                            C->vs + base / 64, C->vb + base / 64, p + 1, hd, C->bits,
                            o + (size_t)i * qd + (size_t)j * hd);
        else
          orc_attention(q + (size_t)i * qd + (size_t)j * hd, C->k + base, C->v + base, p + 1, hd,
                        o + (size_t)i * qd + (size_t)j * hd);
      }
    }
    orc_linear_apply(c, &L->wo, d, qd, o, n, a);
    for (size_t t = 0; t < (size_t)n * d; ++t) x[t] = x[t] + a[t];
    /* FFN block */
    for (int i = 0; i < n; ++i) orc_rmsnorm(x + (size_t)i * d, L->ffn_norm, d, c->rms_eps, h + (size_t)i * d);
    orc_linear_apply(c, &L->wg, F, d, h, n, gt);
    orc_linear_apply(c, &L->wu, F, d, h, n, up);
    for (size_t t = 0; t < (size_t)n * F; ++t) gt[t] = (float)(orc_silu((double)gt[t]) * (double)up[t]);
    orc_linear_apply(c, &L->wd, d, F, gt, n, a);
    for (size_t t = 0; t < (size_t)n * d; ++t) x[t] = x[t] + a[t];
  }
  for (int s = 0; s < n_kv; ++s) {
    kv[s].len = next[s];
    /* a first call ran on bf16 K/V: its positions are converted now; later calls quantised
     * their positions as they appended them */
    if (kv[s].kq && quant[s]) kv[s].qlen = kv[s].len;
    else if (kv[s].kq && kv[s].len > 0) orc_kv_convert(c, &kv[s]);
  }
  free(quant);

  /* final norm + lm_head for the wanted tokens only (slice before the head) */
  int nw = 0;
  for (int i = 0; i < n; ++i) nw += want[i] ? 1 : 0;
  if (nw > 0) {
    float* hw = (float*)malloc(sizeof(float) * (size_t)nw * d);
    int r = 0;
    for (int i = 0; i < n; ++i)
      if (want[i]) orc_rmsnorm(x + (size_t)i * d, m->final_norm, d, c->rms_eps, hw + (size_t)(r++) * d);
    orc_linear_apply(c, &m->lm_head, V, d, hw, nw, logits);
    free(hw);
  }
  free(x); free(h); free(q); free(k); free(v); free(o); free(a); free(gt); free(up); free(next);
  return ORC_OK;
}

int orc_decode_step_batch(const orc_model* m, orc_kv* kv, int B, const int* last_tokens,
                          float* logits) {
  int* seq = (int*)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
  int* pos = (int*)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
  int* want = (int*)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
  for (int b = 0; b < B; ++b) {
    seq[b] = b;
    pos[b] = kv[b].len;
    want[b] = 1;
  }
  int rc = orc_forward(m, kv, B, B, seq, pos, last_tokens, want, logits);
  free(seq); free(pos); free(want);
  return rc;
}

int orc_prefill_segmented(const orc_model* m, orc_kv* kv, int K, const int* seg_lens,
                          const int* tokens, float* logits) {
  int T = 0;
  for (int s = 0; s < K; ++s) {
    if (seg_lens[s] <= 0 || kv[s].len != 0) return ORC_EINVAL;
    T += seg_lens[s];
  }
  int* seq = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
  int* pos = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
  int* want = (int*)malloc(sizeof(int) * (size_t)(T > 0 ? T : 1));
  int g = 0;
  for (int s = 0; s < K; ++s)
    for (int p = 0; p < seg_lens[s]; ++p, ++g) {
      seq[g] = s;
      pos[g] = p; /* segment-local position, from 0 */
      want[g] = (p == seg_lens[s] - 1);
    }
  int rc = orc_forward(m, kv, K, T, seq, pos, tokens, want, logits);
  free(seq); free(pos); free(want);
  return rc;
}

int orc_prefill_sequence(const orc_model* m, orc_kv* kv, int len, const int* tokens,
                         float* logits_last) {
  if (len <= 0) return ORC_EINVAL;
  int* seq = (int*)calloc((size_t)len, sizeof(int));
  int* pos = (int*)malloc(sizeof(int) * (size_t)len);
  int* want = (int*)calloc((size_t)len, sizeof(int));
  for (int p = 0; p < len; ++p) pos[p] = kv->len + p;
  want[len - 1] = 1;
  int rc = orc_forward(m, kv, 1, len, seq, pos, tokens, want, logits_last);
  free(seq); free(pos); free(want);
  return rc;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
