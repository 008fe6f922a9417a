/*
 * cbt.h -- C ABI of the continuous-batching decode engine (libcbt.so).
 *
 * One GB300, one process.  The library runs a pre-norm decoder transformer
 * (RMSNorm, grouped-query attention with RoPE, SwiGLU FFN) over many live
 * sequences at once:
 *
 *   - cbt_decode_step_batch(seq_ids, last_tokens) -> logits[B]: one token per
 *     live sequence.  Every projection (QKV, O, gate/up, down, lm_head) runs
 *     once over all B rows, so each weight is read from HBM once per step; the
 *     amortisation law on the gnosis page ("The throughput law": sharedCost =
 *     w + L*a against naiveCost = L*(w + a)).  Attention is per sequence: row
 *     s reads its own KV slab over positions [0, t_s], applies RoPE at t_s,
 *     appends its new K/V at t_s and t_s is bumped (gnosis page,
 *     "decode_step_batch -- paint-by-numbers", Delta 1..3).
 *   - cbt_prefill_segmented(seq_ids, seg_lens, tokens): K prompts packed in one
 *     pass; the projections run once over all sum(seg_lens) tokens and
 *     attention is block-diagonal causal, token g of a segment starting at
 *     seg_start attending to [seg_start, g] only (gnosis page, "REVISED: the
 *     hard kernel already exists -- forward_batch_segmented").  Returns the
 *     logits of each segment's last token only (mlx-bun batching design,
 *     section 4.2: slice the last position before the head).
 *   - slabs: one KV slab per live sequence, allocated from a caller-provided
 *     device arena and freed on retire (gnosis page, "1. Native station:
 *     per-sequence KV + a batched decode step": an N-slot KV arena keyed by a
 *     sequence id, prefillSeq / freeSeq).
 *   - greedy sampling: argmax over each row's logits, the lowest vocabulary id
 *     winning ties (mlx-bun batching design, section 4.4 "Vectorized
 *     homogeneous sampling", and its campaign note on tied candidate scores).
 *
 * Conventions for every call:
 *   - Return value: CBT_OK (0) or a negative cbt_status; cbt_status_str()
 *     names it.  Errors the host can see (bad or duplicate slab id, batch
 *     above max_batch, capacity overflow, pool exhausted, null pointers,
 *     sizes out of range) are reported BEFORE any work is queued and leave
 *     the engine unchanged.
 *   - Work is queued asynchronously on the engine's CUDA stream.  Errors only
 *     the device can see (a token id >= vocab) set a device error word that
 *     cbt_last_device_error() reads; the offending row's outputs are then
 *     unspecified, other rows are unaffected, and nothing traps.
 *   - Ownership: the caller owns and frees the weights, the KV arena, token
 *     and logits buffers; the engine borrows them for its lifetime and never
 *     frees them.  The engine owns its scratch memory, which it allocates in
 *     cbt_engine_create and frees in cbt_engine_destroy.
 *   - An engine is not thread safe: one host thread at a time.
 */
#ifndef CBT_H
#define CBT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t cbt_status;
#define CBT_OK 0
#define CBT_ERR_INVALID -1        /* a size or config field out of range */
#define CBT_ERR_NULL -2           /* a required pointer is NULL */
#define CBT_ERR_BAD_SLAB -3       /* slab id unknown or already freed */
#define CBT_ERR_DUP_SLAB -4       /* the same slab id twice in one call */
#define CBT_ERR_BATCH -5          /* B > max_batch or K > max_batch */
#define CBT_ERR_CAPACITY -6       /* a slab would grow past its capacity */
#define CBT_ERR_POOL_EXHAUSTED -7 /* no free extent large enough in the KV arena */
#define CBT_ERR_TOKENS -8         /* sum of seg_lens above max_prefill_tokens */
#define CBT_ERR_CUDA -9           /* a CUDA runtime call failed */
#define CBT_ERR_DEVICE -10        /* the device error word was set (see below) */
#define CBT_ERR_UNSUPPORTED -11   /* shape not supported by the kernels */
#define CBT_ERR_LIMIT -12         /* size above the fixed scratch of cbt_greedy_head_noalloc */

/* device error word codes, as returned by cbt_last_device_error in *code */
#define CBT_DEV_OK 0
#define CBT_DEV_TOKEN_RANGE 1 /* a token id outside [0, vocab) */
#define CBT_DEV_TIMEOUT 2     /* a kernel's bounded wait ran out; it stopped early (info: role) */
#define CBT_DEV_WORK_ITEM 3   /* an attention work item its kernel cannot take (info: item) */

#define CBT_WEIGHTS_BF16 0    /* bf16, row-major [out][in] */
#define CBT_WEIGHTS_AFFINE4 1 /* 4-bit affine, see cbt_linear */

typedef struct {
  int32_t n_layers;
  int32_t d_model;
  int32_t n_heads;    /* query heads */
  int32_t n_kv_heads; /* key/value heads; q head j reads kv head j / (n_heads / n_kv_heads) */
  int32_t head_dim;   /* must be 64 or 128 */
  int32_t d_ff;       /* SwiGLU hidden size */
  int32_t vocab;
  float rms_eps;
  double rope_theta; /* RoPE rotate-half form, pair (i, i + head_dim/2) turned by
                        pos * rope_theta^(-2i/head_dim) */
  int32_t weight_format; /* CBT_WEIGHTS_BF16 or CBT_WEIGHTS_AFFINE4 */
  int32_t group_size;    /* CBT_WEIGHTS_AFFINE4 only: must be 64 */
} cbt_model_config;

/* One projection W [out][in] (y = x W^T), device pointers.
 * BF16:    w = bf16 [out][in] row-major; scales = biases = NULL.
 * AFFINE4: w = uint32 [out][in/8], element 8j+k of a row in bits 4k..4k+3 of word j;
 *          scales, biases = bf16 [out][in/group]; the weight is scale*q + bias of its
 *          group (MLX-style affine quantisation; cbt_quantize_affine4 produces it). */
typedef struct {
  const void* w;
  const void* scales;
  const void* biases;
} cbt_linear;

typedef struct {
  cbt_linear wqkv;       /* [(n_heads + 2 n_kv_heads) * head_dim][d_model]: q rows, k rows, v rows */
  cbt_linear wo;         /* [d_model][n_heads * head_dim] */
  cbt_linear wgu;        /* [2 d_ff][d_model]: gate rows [0, d_ff), up rows [d_ff, 2 d_ff) */
  cbt_linear wd;         /* [d_model][d_ff] */
  const void* attn_norm; /* bf16 [d_model] RMSNorm gain before attention */
  const void* ffn_norm;  /* bf16 [d_model] RMSNorm gain before the FFN */
} cbt_layer_weights;

typedef struct {
  const void* embed;                /* bf16 [vocab][d_model] (never quantised) */
  cbt_linear lm_head;               /* [vocab][d_model] */
  const void* final_norm;           /* bf16 [d_model] */
  const cbt_layer_weights* layers;  /* host array [n_layers]; copied by cbt_engine_create */
} cbt_weights;

typedef struct {
  void* kv_arena;            /* device memory for all KV slabs, 256-byte aligned, borrowed */
  size_t kv_arena_bytes;
  int32_t max_batch;         /* most rows per decode step and most segments per prefill */
  int32_t max_prefill_tokens;/* most tokens (sum of seg_lens) per prefill call */
  void* stream;              /* cudaStream_t all work is queued on; NULL = legacy default */
  int32_t kv_page_tokens;    /* 0: each slab is one extent of the arena, reserved at
                              * cbt_kv_slab_alloc for its whole capacity.  > 0 (a multiple of
                              * 128): paged KV -- a slab takes pages of this many positions
                              * from the arena as its positions are first written (prefill,
                              * decode, import, copy_prefix), so a slab's capacity is only a
                              * limit and no capacity is held unused; a call that needs a page
                              * the arena cannot give fails with CBT_ERR_POOL_EXHAUSTED before
                              * queuing anything (pages it took are returned).  Page p of a
                              * slab holds positions [p * kv_page_tokens, (p + 1) *
                              * kv_page_tokens) in the layout described at cbt_slab_bytes.
                              * Pages may be shared between slabs (cbt_kv_slab_share_prefix);
                              * a call that writes a position in a shared page first queues a
                              * copy of that page into a new page of the writing slab (copy on
                              * write), and that page counts towards the same pool check. */
  int32_t kv_bits;           /* 0 or 16: bf16 KV.  8 or 4: affine KV of that many bits (the
                              * mlx-bun batching design's quantised KV, "--kv-quant 4|8"): per
                              * position and (layer, K|V, kv head), head_dim codes plus a bf16
                              * scale and bias per 64 dims; a value reads back as scale * code +
                              * bias, with L = 2^kv_bits - 1, scale = bf16((max - min) / L),
                              * bias = bf16(min), code = clamp(rint((x - bias) / scale), 0, L)
                              * over its group of 64 (cbt_quantize_kv).  A segment that starts a
                              * sequence (its slab at position 0) is prefilled in bf16 and then
                              * converted (the design's conversion point), so its prefill logits
                              * equal the bf16 engine's; every later call -- a decode step, or a
                              * prefill segment continuing the slab (a chunked prompt) --
                              * quantises each position it appends before attention reads all
                              * positions through their codes.  Slabs (and pages) take
                              * cbt_slab_bytes_kvq bytes; the engine also holds max_batch *
                              * cbt_slab_bytes(cfg, 128) bytes of the arena for the decode rows'
                              * bf16 staging (CBT_ERR_POOL_EXHAUSTED from cbt_engine_create if it
                              * does not fit).  Needs n_heads / n_kv_heads in {1, 2, 4, 8} and
                              * the tensor-core path (cbt_engine_create returns
                              * CBT_ERR_UNSUPPORTED otherwise); works with paged KV.
                              * cbt_kv_slab_import quantises what it imports; cbt_kv_slab_export
                              * gives each value as bf16(fp32(scale * code + bias)), the product
                              * and sum taken in double; cbt_kv_slab_copy_prefix copies codes,
                              * scales and biases; cbt_kv_slab_share_prefix shares pages.  During
                              * a call, intermediate bf16 slabs of the prompts' (or the import's)
                              * size are taken from the arena and returned. */
} cbt_engine_params;

typedef struct {
  int32_t live_slabs;
  int32_t max_batch;
  int64_t slab_bytes_in_use;  /* bytes of the arena held by live slabs */
  int64_t arena_bytes;
  int64_t largest_free_bytes; /* largest single free extent */
  int64_t scratch_bytes;      /* device scratch the engine allocated */
  int64_t decode_steps;       /* decode steps queued so far */
  int64_t prefill_tokens;     /* prefill tokens queued so far */
} cbt_stats;

typedef struct cbt_engine cbt_engine;

/* Bytes of a quantised KV slab (or page) of capacity cap at kv_bits = bits (8 or 4): per
 * (layer, K|V, kv head) block codes [round64(cap)][head_dim * bits / 8] uint8 (at 4 bits element
 * 2i in the low nibble of byte i, 2i + 1 in its high nibble), then bf16 scales and bf16 biases
 * [round64(cap)][head_dim / 64]; the total rounded up to 4 KiB.  0 if head_dim is not a multiple
 * of 64, cap <= 0 or bits is not 8 or 4.  cbt_slab_bytes_kv8(c, cap) = cbt_slab_bytes_kvq(c,
 * cap, 8). */
size_t cbt_slab_bytes_kvq(const cbt_model_config* c, int32_t cap, int32_t bits);
size_t cbt_slab_bytes_kv8(const cbt_model_config* c, int32_t cap);

/* Affine quantisation of bf16 rows, groups of 64 along each row (the kv_bits = bits format).
 *   x       device bf16 [rows][cols], 4-byte aligned; cols a multiple of 64.
 *   bits    8 or 4.
 *   codes   device uint8 [rows][cols * bits / 8] (2-byte aligned at 8 bits); scales, biases
 *           device bf16 [rows][cols / 64].
 *   stream  cudaStream_t (NULL: legacy default stream); queued, not synchronised.
 * CBT_ERR_NULL, CBT_ERR_INVALID (bits, shape or alignment), CBT_ERR_CUDA.
 * cbt_quantize_kv8 is cbt_quantize_kv with bits = 8. */
cbt_status cbt_quantize_kv(const void* x, int32_t rows, int32_t cols, int32_t bits, void* codes,
                           void* scales, void* biases, void* stream);
cbt_status cbt_quantize_kv8(const void* x, int32_t rows, int32_t cols, void* codes, void* scales,
                            void* biases, void* stream);

const char* cbt_status_str(cbt_status s);

/* Create an engine over the caller's weights and KV arena.  Copies the config, the weight
 * pointer tables and the params; allocates device scratch sized for max_batch rows and
 * max_prefill_tokens tokens.  On failure *out is NULL and nothing is allocated. */
cbt_status cbt_engine_create(const cbt_model_config* cfg, const cbt_weights* weights,
                             const cbt_engine_params* params, cbt_engine** out);

/* Synchronise the engine's stream and free everything the engine allocated. */
cbt_status cbt_engine_destroy(cbt_engine* e);

/* Bytes one slab of `capacity_tokens` positions takes in the arena: the capacity rounded up
 * to a multiple of 64 (C), times n_layers * 2 (K, V) * n_kv_heads * head_dim * 2 bytes,
 * rounded up to 4 KiB.  Slab layout (bf16): [layer][K|V][kv head] blocks of C * head_dim
 * elements; a K block is [position][head_dim]; a V block is [position / 64][head_dim][64]
 * (each group of 64 positions transposed), so both attention contractions read K-major
 * tiles.  Import and export use the plain layout described at cbt_kv_slab_import. */
size_t cbt_slab_bytes(const cbt_model_config* cfg, int32_t capacity_tokens);

/* Reserve a slab for one sequence (host-side first-fit allocator over the arena, no
 * device work).  The slab starts empty (position 0).  The slab id is the sequence id
 * every later call uses. */
cbt_status cbt_kv_slab_alloc(cbt_engine* e, int32_t capacity_tokens, int32_t* slab_id);

/* Return a slab to the arena (host-side bookkeeping only).  Work already queued on the
 * engine stream that uses the slab still runs before any later work on that stream can
 * reuse its extent, so a slab may be freed right after the step that last used it. */
cbt_status cbt_kv_slab_free(cbt_engine* e, int32_t slab_id);

/* retire: free the slabs of finished sequences (EOS or length limit), n ids. */
cbt_status cbt_retire(cbt_engine* e, const int32_t* slab_ids, int32_t n);

/* Current position (tokens held) of a slab. */
cbt_status cbt_kv_slab_position(cbt_engine* e, int32_t slab_id, int32_t* pos);

/* Save/restore a sequence's state.  import copies n_tokens positions of K and V into the
 * slab (positions [0, n_tokens)) and sets its position to n_tokens; export copies
 * positions [0, n_tokens) out.  k and v are bf16 [n_layers][n_kv_heads][n_tokens][head_dim],
 * on the host (on_host != 0) or on the device.  Queued on the engine stream. */
cbt_status cbt_kv_slab_import(cbt_engine* e, int32_t slab_id, const void* k, const void* v,
                              int32_t n_tokens, int32_t on_host);
cbt_status cbt_kv_slab_export(cbt_engine* e, int32_t slab_id, void* k, void* v,
                              int32_t n_tokens, int32_t on_host);

/* Prefix reuse: copy positions [0, n_tokens) of slab src_id's K and V into slab dst_id and set
 * dst's position to n_tokens, so a prefill of dst continues after a prefix that was computed
 * once (the mlx-bun batching design, sections 1 and 4.2: sub-agents share long system
 * prompts; a joiner's prefill starts from the longest cached prefix, so N agents sharing a
 * prompt reuse one prefill).  Here the reuse is a device-to-device copy of the prefix's bytes
 * (n_tokens x 2 x n_layers x n_kv_heads x head_dim bf16), queued on the engine stream; the
 * slabs stay independent afterwards.
 *   src_id, dst_id  distinct live slabs; n_tokens <= src's position and <= dst's capacity.
 * Errors (nothing queued, nothing changed): CBT_ERR_BAD_SLAB, CBT_ERR_INVALID (same slab or
 * n_tokens < 0), CBT_ERR_CAPACITY, CBT_ERR_CUDA. */
cbt_status cbt_kv_slab_copy_prefix(cbt_engine* e, int32_t src_id, int32_t dst_id,
                                   int32_t n_tokens);

/* Prefix sharing (the same pages, the mlx-bun batching design, sections 1 and 4.2): slab dst_id
 * takes positions [0, n_tokens) of slab src_id without a copy and its position becomes n_tokens.
 * On a paged engine dst holds src's first ceil(n_tokens / kv_page_tokens) pages by reference
 * (no device work, no arena bytes); the first later write into a shared page by either slab
 * (prefill, decode, import, copy_prefix into it) copies that one page first, so neither slab
 * ever sees the other's later positions, and a page returns to the arena when its last holder
 * frees it.  On a contiguous engine there are no pages to share and the call is
 * cbt_kv_slab_copy_prefix.
 *   src_id, dst_id  distinct live slabs; dst at position 0 (pages it holds are released);
 *                   n_tokens <= src's position and <= dst's capacity.
 * Errors (nothing queued, nothing changed): CBT_ERR_BAD_SLAB, CBT_ERR_INVALID (same slab,
 * n_tokens < 0 or dst's position not 0), CBT_ERR_CAPACITY, and on a contiguous engine those of
 * cbt_kv_slab_copy_prefix. */
cbt_status cbt_kv_slab_share_prefix(cbt_engine* e, int32_t src_id, int32_t dst_id,
                                    int32_t n_tokens);

/* Segmented prefill of K prompts (forward_batch_segmented).
 *   slab_ids  host int32 [K], distinct live slabs.  Segment s's tokens go to positions
 *             [p_s, p_s + seg_lens[s]) of its slab, p_s being the slab's current position
 *             (0 for a fresh slab: positions are segment-local from 0); each token attends
 *             to positions [0, its own] of its own slab only.
 *   seg_lens  host int32 [K], each >= 1, sum <= max_prefill_tokens, p_s + seg_lens[s] <=
 *             capacity.
 *   tokens    device int32 [sum seg_lens], the segments back to back.
 *   logits    device float [K][vocab]: logits of each segment's last token; NULL allowed.
 *   next_tokens device int32 [K]: greedy argmax of those logits; NULL allowed.
 * Afterwards each slab's position is p_s + seg_lens[s]. */
cbt_status cbt_prefill_segmented(cbt_engine* e, const int32_t* slab_ids, const int32_t* seg_lens,
                                 int32_t K, const int32_t* tokens, float* logits,
                                 int32_t* next_tokens);

/* One continuous-batching decode step (decode_step_batch).
 *   slab_ids    host int32 [B], distinct live slabs; row b is the sequence of slab_ids[b].
 *   last_tokens device int32 [B]: the token each row feeds (may be the previous step's
 *               next_tokens buffer, so greedy decode needs no host round trip).
 *   logits      device float [B][vocab] or NULL.
 *   next_tokens device int32 [B] or NULL: greedy argmax of each row, lowest id on ties.
 * Row b's token is placed at position t_b (the slab's current position, which must be
 * below its capacity), attends to [0, t_b] of its own slab, and t_b becomes t_b + 1.
 * B == 0 is a no-op. */
cbt_status cbt_decode_step_batch(cbt_engine* e, const int32_t* slab_ids, int32_t B,
                                 const int32_t* last_tokens, float* logits, int32_t* next_tokens);

/* Synchronise the engine's stream, then read and clear the device error word.
 * *code = CBT_DEV_OK or a CBT_DEV_* code, *info = the offending row or token index.
 * Returns CBT_OK, or CBT_ERR_CUDA if the stream reported an error. */
cbt_status cbt_last_device_error(cbt_engine* e, int32_t* code, int32_t* info);

cbt_status cbt_engine_stats(cbt_engine* e, cbt_stats* out);

/* Number of kernel launches the library queued so far, all engines together (for launch
 * accounting; e may be NULL). */
int64_t cbt_kernel_launches(cbt_engine* e);

/* Measurement.  Kernel classes: */
#define CBT_KCLASS_PROJ 0  /* projections QKV, O, gate/up (+SwiGLU), down, lm_head: weight streaming */
#define CBT_KCLASS_ATTN 1  /* RoPE + KV append and attention over the slabs */
#define CBT_KCLASS_OTHER 2 /* embedding, norms, RoPE tables, argmax, gathers */
#define CBT_NUM_KCLASSES 3

/* Bracket every launch group of the classes in class_mask (bit k = class k) with CUDA
 * events on the engine stream, from now on; 0 turns it off.  Clears earlier records.
 * Events only mark the stream between kernels; they change no result. */
cbt_status cbt_engine_set_timing(cbt_engine* e, int32_t class_mask);

/* Synchronise the stream and sum the records of one class since cbt_engine_set_timing:
 * total device milliseconds, number of bracketed intervals, and the algorithmic bytes those
 * intervals moved (each weight once, activations in and out, each live KV position once). */
cbt_status cbt_engine_timing(cbt_engine* e, int32_t kclass, double* total_ms, int64_t* intervals,
                             double* algorithmic_bytes);

/* Failure-detection test of the bounded device waits.  Every wait in the library's kernels
 * (on an mbarrier, a cluster peer or a flag) gives up after a bounded number of polls, records
 * CBT_DEV_TIMEOUT in the device error word (info: the role that gave up) and lets its kernel
 * end; nothing traps or hangs.  This call arms the next cbt_decode_step_batch of the engine so
 * that its lm_head projection requests none of its weight tiles and every wait of that launch
 * runs out after spin_limit polls.  That step then reports CBT_DEV_TIMEOUT through
 * cbt_last_device_error; its logits and next tokens are unspecified, everything else it does
 * (the K/V it appends, the positions it bumps) is as in a normal step, and later steps are
 * unaffected.  Bf16 weights on the tensor-core path only (else CBT_ERR_UNSUPPORTED);
 * spin_limit > 0 (else CBT_ERR_INVALID). */
cbt_status cbt_engine_test_stall(cbt_engine* e, int32_t spin_limit);

/* In-step stamps (measurement).  With enable != 0, every later decode step -- replayed steps
 * included -- records for each of its projection and attention launches (CBT_KCLASS_PROJ,
 * CBT_KCLASS_ATTN) the earliest time one of the launch's CTAs could start work that depends on
 * the previous kernel and the latest time one of them ended, in globaltimer nanoseconds.  The
 * stamps change no result.  cbt_engine_stamps synchronises the stream and copies the records of
 * the last decode step: *n = their number; for i < min(cap, *n) classes[i] = the launch's class,
 * times[2i] = begin, times[2i + 1] = end.  (A step's launches overlap through programmatic
 * dependent launch; the union of a class's intervals is its share of the step.) */
cbt_status cbt_engine_set_stamps(cbt_engine* e, int32_t enable);
cbt_status cbt_engine_stamps(cbt_engine* e, int32_t cap, int32_t* n, int32_t* classes,
                             uint64_t* times);

/* MLX-style 4-bit affine quantisation of a bf16 matrix on the device, groups of `group`
 * (64) along each row: scale = bf16((max - min) / 15), bias = bf16(min),
 * q = clamp(rint((w - bias) / scale), 0, 15) (ties to even; 0 when scale == 0), packed
 * as in cbt_linear.  w: device bf16 [rows][cols]; packed: device uint32 [rows][cols/8];
 * scales, biases: device bf16 [rows][cols/group].  cols % group == 0.  Queued on `stream`. */
cbt_status cbt_quantize_affine4(const void* w, int32_t rows, int32_t cols, int32_t group,
                                void* packed, void* scales, void* biases, void* stream);

/* ---- Greedy head without any allocation --------------------------------------------------
 * The pages have no counterpart to this call; it exists for callers that cannot allocate
 * device memory: code running where cudaMalloc is forbidden or unsafe (inside another
 * framework's memory pool or allocator hooks, a real-time loop that must not block on the
 * allocator, an embedding runtime that hands over pre-planned buffers only).  It runs the
 * last stage of a decode step on hidden states the caller already has:
 *   logits[r] = RMSNorm(hidden[r], final_norm, cfg->rms_eps) lm_head^T,
 *   next_tokens[r] = argmax(logits[r]) (lowest id on ties),
 * the operations decode_step_batch ends with, computed by the library's CUDA-core kernels
 * (an RMSNorm kernel, a split-K projection whose partial sums are added in a fixed order,
 * the argmax kernel) rather than the tensor-core projection of a decode step, so its logits
 * agree with decode_step_batch's within rounding, not bit for bit.  Its scratch (the
 * normalised rows and the split-K partial sums) lives in one fixed array in the library's
 * device memory, CBT_NOALLOC_SCRATCH_BYTES large.  Every GPU that loads the library holds
 * that array until the process exits.
 *   cfg          model config (d_model, vocab, rms_eps, weight_format, group_size are used)
 *   hidden       device float [n][d_model], the residual stream after the last layer
 *   n            rows, 0 <= n <= CBT_NOALLOC_MAX_ROWS (0 is a no-op)
 *   final_norm   device bf16 [d_model]
 *   lm_head      projection [vocab][d_model] as in cbt_linear (device pointers)
 *   logits       device float [n][vocab], written
 *   next_tokens  device int32 [n], written; may be NULL
 *   stream       cudaStream_t to queue on (NULL = legacy default stream)
 * Returns CBT_ERR_CUDA if one of its own launches fails (an error left by earlier, unrelated
 * work is neither reported nor cleared), and CBT_ERR_LIMIT, before queuing anything, when
 * n > CBT_NOALLOC_MAX_ROWS or when
 * n*d_model + (d_model/slice)*n*vocab floats (slice = 1024, 512 or 256, the largest that
 * divides d_model) exceed the fixed scratch.  It calls no cudaMalloc, cudaFree or any
 * allocating library routine.  The first call on each device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first call before
 * any stream capture.  All calls share the one array and it keeps the last call's
 * contents, so calls that overlap on the GPU (different streams, or threads) race: queue
 * them on one stream, or order them with events. */
#define CBT_NOALLOC_MAX_ROWS 32
#define CBT_NOALLOC_SCRATCH_BYTES (20u << 20)
cbt_status cbt_greedy_head_noalloc(const cbt_model_config* cfg, const float* hidden, int32_t n,
                                   const void* final_norm, const cbt_linear* lm_head,
                                   float* logits, int32_t* next_tokens, void* stream);

#ifdef __cplusplus
}
#endif
#endif
