// kernels.h -- launchers of the engine's CUDA kernels (host side).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

#include <utility>

// kernel launches queued through the launchers below (for launch accounting)
long long kernel_launch_count();
void count_launch(int n = 1);

// Launch with programmatic stream serialization (see pdl_wait / pdl_launch in common.cuh)
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct LinearW {
  const void* w;       // bf16 [M][K] or uint32 [M][K/8]
  const uint16_t* scales;  // affine4 only: bf16 [M][K/64]
  const uint16_t* biases;
  int fmt;             // CBT_WEIGHTS_BF16 / CBT_WEIGHTS_AFFINE4
};

// ---- tensor-core projections (gemm_tc.cu) --------------------------------------------------
struct Kv8Job;

struct TcParams {
  int M, K;          // W is [M][K] bf16; for EPI_SWIGLU M = 2F (gate rows, then up rows)
  int F;             // EPI_SWIGLU: features per output row
  int n_act;         // activation rows (decode rows or prefill tokens)
  int epi;           // Epilogue
  float* out;        // EPI_STORE / EPI_ADD: fp32 [n_act][ldo]
  int ldo;
  uint16_t* act;     // EPI_SWIGLU: bf16 operand of the next projection, [rows][act_ld]
  int act_ld;
  int act_lo;        // row offset of the lo parts (0: plain bf16, no lo part)
  // schedule, filled by the launcher: row tiles, token tiles, 64-column k-blocks
  int RB, NT, KS;
  int* err;          // device error word
  // RMSNorm folded into the projections (decode rows only).  Consumer side: the operand is
  // x * g, and column b of the result is scaled by rsqrt(sum_t ss_in[t][b] / K + eps).
  const float* ss_in;     // [ss_tiles][ss_ld] sums of squares of x over 128-element tiles
  int ss_tiles, ss_ld;
  float eps;
  // Producer side (EPI_ADD): also write the updated rows' sums of squares per 128-row tile
  // ([RB][ss_ld]) and the next projection's operand x * next_gain as bf16 (hi at row t of
  // next_act, lo at row next_lo + t when next_lo > 0; row stride ldo)
  float* ss_out;
  const uint16_t* next_gain;
  uint16_t* next_act;
  int next_lo;
  // EPI_QKV (decode rows): RoPE of q and k at each row's own position, the new K/V appended
  // to the row's slab, q written as the decode attention's operand image (qtile)
  const QueryRow* rows;
  int layer, n_heads, n_kv_heads, head_dim;
  const float* cosv;  // [n_act][head_dim / 2]
  const float* sinv;
  uint16_t* arena;
  uint8_t* qtile;
  // EPI_QKVQ (EPI_QKV on a quantised-KV engine): the new K/V are quantised in the epilogue (groups of 64
  // dims, kvq_bits bits) straight into each row's quantised slab, described by kvq_jobs[row]
  // (dst, dst_cap, dst_p0); arena is then the arena's bytes and nothing is written in bf16
  const Kv8Job* kvq_jobs;
  int kvq_bits;
  // 4-bit affine weights in the native block layout of gemm_q4.cu (launch_q4_rd only)
  const uint8_t* wq;
  unsigned long long* stamp;  // measurement stamp slot (common.cuh), or NULL
  // failure detection test (launch_tc_csk only): the producer requests nothing, so every wait
  // for a tile runs out after spin_limit polls (0: the default limit) and reports a timeout
  int stall_loads;
  uint32_t spin_limit;
};


bool make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows);
// A bf16 [rows][K] matrix seen as 64-column blocks, so one TMA box brings nk consecutive blocks
// of box_rows rows, each landing as a 128-byte-swizzled [box_rows][64] tile: 3-D map
// {64, rows, K/64}.  pair_rows > 0 (SwiGLU's [gate; up], rows = 2 pair_rows): 4-D map
// {64, pair_rows, 2, K/64}, a box brings box_rows gate rows then the same up rows per block.
bool make_tmap_kblocks(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows,
                       uint32_t nk, uint64_t pair_rows);
// N tile for hi/lo (split) activations of n rows, and for plain bf16 activations
int tc_split_bn(int n);
int tc_plain_bn(int n);
// twl (prefill only): the lo parts of weights given as bf16 hi + lo matrices (both maps 64 x 64
// boxes over [M][K]); the product is hi.x_hi + hi.x_lo + lo.x_hi.
bool launch_tc_linear(const CUtensorMap& tw, const CUtensorMap& tx, TcParams p, bool split,
                      int BN, int num_sms, cudaStream_t s, const CUtensorMap* twl = nullptr);

// ---- cluster split-K decode projections (gemm_csk.cu) -----------------------------------------
// Clusters of C CTAs; cluster c takes row tiles c, c + NC, ...; rank r streams k-blocks
// [r*KS/C, (r+1)*KS/C) of each, and the tile's partial sums are reduce-scattered over the
// cluster through distributed shared memory (rank r adds and finishes its chunk of the
// columns).
struct CskPlan {
  int C;       // CTAs per cluster (split of K)
  int NC;      // clusters
  int stages;  // pipeline depth
  int slots;   // inbox slots: most tiles of one cluster (C > 1)
  int nk;      // 64-column blocks per stage (one TMA box of weights, one of operand)
};
constexpr int kCskBlocks = 2;  // nk of the decode projections' tensor maps
bool csk_plan(int RB, int KS, int BN, int num_sms, CskPlan* out);
// y = x W^T over n_act <= BN/2 decode rows (hi/lo operand), any TcParams epilogue.  tw: the
// weights as make_tmap_kblocks(.., 128 rows (SwiGLU: 64 + 64), kCskBlocks, ..); tx: the operand
// as make_tmap_kblocks(.., BN rows, kCskBlocks, 0).
bool launch_tc_csk(const CUtensorMap& tw, const CUtensorMap& tx, TcParams p, int BN, int num_sms,
                   cudaStream_t s);

// ---- 4-bit affine decode projections (gemm_q4.cu: device layout; gemm_q4r.cu: kernel) ------
// Native layout: per (128-row tile, 128-column superblock) one block of kQ4BlockBytes (codes
// as [4][128 rows][16 bytes], then bf16 scale/bias pairs of the block's two 64-column groups).
constexpr int kQ4BlockBytes = 128 * 64 + 128 * 8;
// bytes of the native copy of an [M][K] matrix (F > 0: SwiGLU gate/up pair, M = 2F); 0 when K
// is not a multiple of 128
size_t q4_native_bytes(int M, int K, int F);
// write the native copy from the interchange format (cbt_linear: codes [M][K/8] uint32, bf16
// scales and biases [M][K/64])
bool launch_q4_repack(const uint32_t* packed, const uint16_t* scales, const uint16_t* biases,
                      int M, int K, int F, uint8_t* out, cudaStream_t s);
// expand an interchange-format matrix into bf16 hi and lo parts [M][K] (16-byte aligned):
// w = fp32(s * q + b), hi = bf16(w), lo = bf16(w - hi); for the tensor-core prefill projections
bool launch_q4_expand(const uint32_t* packed, const uint16_t* scales, const uint16_t* biases,
                      int M, int K, uint16_t* hi, uint16_t* lo, int num_sms, cudaStream_t s);
// y = x W^T over n_act <= 32 decode rows with W = p.wq in the native layout, the codes
// dequantised in registers; x is the operand buffer (bf16 rows of K columns: hi parts at rows b,
// lo parts at rows x_lo + b), the rows taken 8 at a time.  Any TcParams epilogue.
bool launch_q4_rd(TcParams p, const uint16_t* x, int x_lo, int num_sms, cudaStream_t s);

// ---- tensor-core decode attention (attn_tc.cu) ------------------------------------------------
struct AttnDecodeArgs {
  const uint8_t* qtile;      // [B][Hkv] Q operand images written by the RoPE kernel
  const QueryRow* rows;      // [B]
  const AttnItem* items;     // work items, grouped by row: row b's items start at item_base[b],
  const int* n_items;        //   kv head g's splits at item_base[b] + g * item_count[b]
                             //   (count on the device, so a captured step stays valid)
  const int* item_base;      // [B]
  const int* item_count;     // [B] splits per (row, kv head)
  int B, layer, n_heads, n_kv_heads, head_dim;
  float* part_o;             // [n_items][G][head_dim] partial outputs
  float2* part_ml;           // [n_items][G] (running max, running sum)
  uint16_t* act;             // attention output as the O projection's bf16 operand
  int act_lo;                // lo rows offset (0: plain bf16)
  int* err;
  float* out_f32;            // if set, the merge writes fp32 [B][n_heads * head_dim] here instead
  unsigned long long* stamp;        // measurement stamp slots (common.cuh) of the attention and
  unsigned long long* stamp_merge;  // of the merge, or NULL
};
// tk: the KV arena as [rows][head_dim] bf16, box {64, 128}; tv: as [rows][64], box {64, head_dim}
bool launch_attn_decode_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnDecodeArgs& a,
                           int num_sms, cudaStream_t s);
// ---- affine KV of 8 or 4 bits (kvq.cu) ---------------------------------------------------------
// A quantised slab (or page) block (layer, K|V, kv head) of capacity cap: codes
// [cap][head_dim * bits / 8] uint8 (4 bits: element 2i in the low nibble of byte i), then bf16
// scales and bf16 biases [cap][head_dim / 64]
CBT_HD long long kvq_block_bytes(int cap, int head_dim, int bits) {
  return (long long)cap * (head_dim * bits / 8 + head_dim / 16);
}
// byte offset of block (layer, K|V, kv head) of the quantised slab or page at byte offset off
CBT_HD long long kvq_block(long long off, int cap, int layer, int kv, int head, int n_kv_heads,
                           int head_dim, int bits) {
  return off + (((long long)layer * 2 + kv) * n_kv_heads + head) *
                   kvq_block_bytes(cap, head_dim, bits);
}
// Positions [t0, t0 + n) of a bf16 slab (or a staging page: a QueryRow base and capacity) to
// be quantised into the quantised slab or page at byte offset dst (layout capacity dst_cap),
// whose first position is dst_p0 (0 for a contiguous slab).
struct Kv8Job {
  long long src_base;
  int src_cap, t0, n, dst_cap;
  long long dst;
  int dst_p0;
};
bool launch_quantize_kv(const uint16_t* x, int rows, int cols, int bits, uint8_t* codes,
                        uint16_t* scales, uint16_t* biases, cudaStream_t s);
// jobs: device [n_jobs]; layers [l0, l0 + nl); max_n = most positions of a job
bool launch_kvq_convert(const Kv8Job* jobs, int n_jobs, int max_n, int l0, int nl, int n_kv_heads,
                        int head_dim, int bits, uint8_t* arena, cudaStream_t s);
struct KvqAttnArgs {
  const uint8_t* qtile;  // [B][Hkv] Q operand images written by the QKV projection's epilogue
  const QueryRow* rows;  // [B]: each row's position (pos)
  const AttnItem* items; // the decode work list (one 128-key sub-chunk per item; kbase = byte
                         // offset of the quantised slab or page holding it, cap, p0)
  const int* n_items;
  const uint8_t* arena;
  int layer, n_heads, n_kv_heads, head_dim;
  float* part_o;         // [n_items][G][head_dim]
  float2* part_ml;       // [n_items][G]
  int* err;
  unsigned long long* stamp;  // measurement stamp slot, or NULL
};
bool launch_attn_decode_q(const KvqAttnArgs& a, int bits, int num_sms, cudaStream_t s);
// attention of prefill tokens over quantised positions [0, pos]: token t's pages (one slab: a
// single entry) are at qpages[tok_first[t] + key / tok_cap[t]]; q from qkv (rotated), o fp32
bool launch_attn_prefill_q(const float* qkv, const QueryRow* rows, const long long* qpages,
                           const int* tok_first, const int* tok_cap, int n, int layer, int n_heads,
                           int n_kv_heads, int head_dim, int max_keys, int bits,
                           const uint8_t* arena, float* o, cudaStream_t s);
// positions [0, n) of one layer of a quantised slab (pages[pos / cap]) as plain bf16
// [n_kv_heads][n][head_dim] K and V
bool launch_kvq_export(const uint8_t* arena, const long long* pages, int cap, int layer,
                       int n_kv_heads, int head_dim, int n, int bits, uint16_t* k, uint16_t* v,
                       cudaStream_t s);
// the split-K merge of the decode attention (attn_tc.cu): partials of each (row, q head)
// combined in item order into the O projection's bf16 hi/lo operand
bool launch_attn_merge(const AttnDecodeArgs& a, cudaStream_t s);

// V of one layer between a plain [kv head][plain_n positions][head_dim] buffer and a slab (or
// page): positions [t0, t0 + n)
void launch_v_convert(uint16_t* plain, uint16_t* arena, const QueryRow& r, int layer,
                      int n_kv_heads, int t0, int n, int plain_n, int head_dim, bool to_slab,
                      cudaStream_t s);

// RMSNorm rows of x into a bf16 operand: hi parts at rows [0, n), lo parts at rows
// [lo_rows, lo_rows + n) when lo_rows > 0
void launch_rmsnorm_act(const float* x, const uint16_t* gain, int n, int d, float eps,
                        uint16_t* act, int lo_rows, cudaStream_t s);
// fp32 rows into a bf16 operand (hi/lo as above)
void launch_f32_to_act(const float* src, int n, int K, uint16_t* act, int lo_rows, cudaStream_t s);

// embed + token range check (and, decode, the first RMSNorm's statistics and operand), with the
// RoPE cos/sin table of the rows' positions (fp32 [n][head_dim / 2], angles in double) built by
// extra blocks of the same launch
void launch_embed_rope(const int32_t* tokens, int n, const uint16_t* table, int d, int vocab,
                       float* x, int* err, float* ss, int ss_ld, const uint16_t* gain,
                       uint16_t* act, int lo_rows, const QueryRow* rows, int head_dim,
                       double theta, float* cosv, float* sinv, cudaStream_t s);
// RMSNorm rows of x into h
cudaError_t launch_rmsnorm(const float* x, const uint16_t* gain, int n, int d, float eps,
                           float* h, cudaStream_t s);
// RoPE q and k in place at each token's position; append k, v (bf16) to its slab; with
// qtile, also write each row's Q operand images for the decode attention ([n][Hkv][16][hd])
void launch_rope_append(float* qkv, const QueryRow* rows, int n, int layer, int n_heads,
                        int n_kv_heads, int head_dim, const float* cosv, const float* sinv,
                        uint16_t* arena, uint8_t* qtile, uint16_t* qb, int q_lo_row,
                        cudaStream_t s);
// qb (prefill): also the rotated q, scaled by 1/sqrt(head_dim), as a bf16 high part at
// qb[t][n_heads*head_dim] and the bf16 rounding of the remainder at qb[q_lo_row + t][...]

// ---- tensor-core segmented prefill attention (attn_prefill.cu) ---------------------------------
// One unit: q head `head` of the 128-query block starting at position q0 of a segment whose
// keys are positions [0, len) of the slab at (base, cap); its queries are packed tokens
// [tok0, tok0 + nq).
struct PrefillUnit {
  long long base;
  int cap, tok0, q0, nq, len, head;
  int pages;  // paged segment: its page bases (QueryRow bases) at pagetab[pages + key / cap]
              // (-1: one slab at base)
};
// tq: the bf16 q buffer as [2][q_lo_row][n_heads*head_dim] rows (high parts, then the
// remainders), box {64, 128}; tk, tv: the KV arena as
// in the decode attention.  o: fp32 [tokens][n_heads*head_dim], softmax(q.K^T) V of each token
// over positions [0, its own] of its segment.
bool launch_attn_prefill_tc(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const PrefillUnit* units, const long long* pagetab, int n_units,
                            int q_lo_row, int layer,
                            int n_heads, int n_kv_heads, int head_dim, float* o, int* err,
                            int num_sms, cudaStream_t s);
// softmax attention of each token over [0, pos] of its own slab; a paged token's keys sit in
// the pages pagetab[tok_pages[t] + key / cap] (tok_pages NULL or -1: one slab)
void launch_attention_naive(const float* qkv, const QueryRow* rows, const long long* pagetab,
                            const int* tok_pages, int n, int layer, int n_heads, int n_kv_heads,
                            int head_dim, int max_keys, const uint16_t* arena, float* o,
                            cudaStream_t s);
// projection y = x W^T with an epilogue; picks the skinny or the tiled kernel
cudaError_t launch_linear(const float* x, int n, int K, const LinearW& W, int M, Epilogue epi,
                          float* out, float* partials, size_t partial_floats, cudaStream_t s);
// greedy argmax per row, lowest index on ties
cudaError_t launch_argmax(const float* logits, int n, int vocab, int32_t* out, cudaStream_t s);
// gather rows idx[i] of src [*, d] into dst [i, d]
void launch_gather_rows(const float* src, const int32_t* idx, int n, int d, float* dst,
                        cudaStream_t s);
// 4-bit affine quantisation of a bf16 matrix
void launch_quantize_affine4(const uint16_t* w, int rows, int cols, int group, uint32_t* packed,
                             uint16_t* scales, uint16_t* biases, cudaStream_t s);
