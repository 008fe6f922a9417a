// engine.cu -- the C ABI: engine state, the slab allocator and the step orchestration.
//
// Host side only.  One engine drives one model on one stream.  Slabs are extents of the
// caller's KV arena handed out by a first-fit allocator with coalescing; each carries its
// capacity and current position (the host mirror of t_s, bumped as steps are queued).  A
// paged engine (kv_page_tokens > 0) gives a slab fixed-size pages from the same allocator as
// its positions are first written, and hands the kernels each page's base; a page may be held
// by several slabs (a shared prompt prefix) and is copied before the first write into it.
// A decode step or a prefill call writes a small per-token row table (slab offset, position,
// capacity) to the device and then queues the whole forward pass on the engine stream.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <new>
#include <unordered_map>
#include <unordered_set>
#include <tuple>
#include <vector>

#include "cbt.h"
#include "kernels.h"

static std::atomic<long long> g_launches{0};
long long kernel_launch_count() { return g_launches.load(); }
void count_launch(int n) { g_launches += n; }

namespace {

constexpr size_t kSlabAlign = 4096;
constexpr int kStampSlots = 1024;  // stamped launches recorded per decode step

struct Slab {
  size_t offset;  // bytes into the arena (contiguous slabs)
  size_t bytes;
  int cap;        // positions the caller asked for (the limit of pos)
  int pos;
  int lcap;       // cap rounded up to 64: the layout's capacity
  std::vector<size_t> pages;  // paged engines: byte offset of each page, in position order
  bool flat = false;  // a call's bf16 intermediate: one extent even on a paged engine
};

template <class T>
cudaError_t dmalloc(T** p, size_t count, size_t* total) {
  size_t bytes = sizeof(T) * (count > 0 ? count : 1);
  bytes = (bytes + 255) & ~size_t(255);
  *total += bytes;
  return cudaMalloc(reinterpret_cast<void**>(p), bytes);
}

}  // namespace

struct cbt_engine {
  cbt_model_config cfg;
  std::vector<cbt_layer_weights> layers;
  cbt_weights w;
  cbt_engine_params p;
  cudaStream_t stream = nullptr;

  // allocator
  std::map<size_t, size_t> free_ext;  // offset -> bytes
  std::unordered_map<int, Slab> slabs;
  int page = 0;            // kv_page_tokens: positions per page (0: contiguous slabs)
  size_t page_bytes = 0;
  std::unordered_map<size_t, int> extra_holders;  // shared pages: holders beyond the first
  // quantised KV (kv_bits = 8 or 4): slabs hold codes; each decode row's new K/V is written in
  // bf16 to its own one-page staging slab (stage_off + b * stage_bytes) and quantised from there;
  // the per-call conversion records (decode rows, prefill segments, an import) on the device
  int kv_bits = 16;
  bool quant() const { return kv_bits != 16; }
  bool q_codes = false;  // this forward pass: prefill tokens attend over codes (continuing slabs)
  int q_jobs = 0, q_jobs_max_n = 0;
  size_t stage_off = 0, stage_bytes = 0;
  Kv8Job* kv8_jobs = nullptr;
  size_t kv8_jobs_cap = 0;
  std::vector<Kv8Job> hjobs;
  // per prefill call: the page bases (QueryRow bases) of every paged segment, and each
  // token's offset into them (read by the prefill attention kernels)
  std::vector<long long> hpagetab;
  std::vector<int> htok_pages;
  long long* pagetab = nullptr;
  int* tok_pages = nullptr;
  size_t pagetab_cap = 0, tok_pages_cap = 0;
  std::vector<const Slab*> hslab;  // the slab of each decode row, for the attention work list
  int next_id = 1;
  size_t in_use = 0;

  // device scratch
  int tmax = 0;
  float *x = nullptr, *h = nullptr, *qkv = nullptr, *o = nullptr, *act = nullptr;
  float *part = nullptr, *xg = nullptr, *logits = nullptr, *cosv = nullptr, *sinv = nullptr;
  int32_t *next_tok = nullptr, *last_idx = nullptr;
  QueryRow* rows = nullptr;
  int* err = nullptr;
  size_t part_floats = 0;
  size_t scratch_bytes = 0;

  std::vector<QueryRow> hrows;
  std::vector<int32_t> hidx;
  int64_t steps = 0, prefill_tokens = 0;

  // tensor-core path (bf16 weights): TMA descriptors of every weight matrix (64x64 boxes)
  // and bf16 operand buffers of the projections
  bool use_tc = false;
  int num_sms = 0;
  struct LayerMaps {
    CUtensorMap qkv, o, gu, d;
  };
  std::vector<LayerMaps> wmaps;     // 64 x 64 boxes (prefill)
  std::vector<LayerMaps> wmaps_kb;  // kCskBlocks 64-column blocks of a 128-row tile per box (decode)
  CUtensorMap lm_map, lm_map_kb;
  // 4-bit affine weights: native block copies for the tensor-core decode projections
  struct Q4Layer {
    uint8_t *qkv = nullptr, *o = nullptr, *gu = nullptr, *d = nullptr;
  };
  std::vector<Q4Layer> q4w;
  uint8_t* q4_lm = nullptr;
  uint8_t* q4_arena = nullptr;
  // 4-bit weights over more than 32 rows (prefill): one matrix at a time expanded into bf16 hi
  // parts (q4x) and lo parts (q4x + q4x_elems), seen through one pair of maps per shape
  enum { kQ4xQkv, kQ4xO, kQ4xGu, kQ4xDown, kQ4xLm, kQ4xShapes };
  uint16_t* q4x = nullptr;
  size_t q4x_elems = 0;
  CUtensorMap q4x_maps[kQ4xShapes][2];
  int act_rows = 0;
  uint16_t *act_h = nullptr, *act_o = nullptr, *act_u = nullptr;
  std::map<std::pair<const void*, int>, CUtensorMap> xmaps;  // (operand buffer, N tile)
  std::map<std::pair<const void*, int>, CUtensorMap> xmaps_kb;
  // tensor-core decode attention: TMA descriptors over the whole KV arena, the per-step work
  // list and the split-K partials (grown on demand)
  CUtensorMap kv_kmap, kv_vmap;
  std::vector<AttnItem> hitems;
  std::vector<int> hitem_base, hitem_count;
  AttnItem* items = nullptr;
  int* item_meta = nullptr;  // [max_batch] bases, [max_batch] counts, then the item total
  size_t items_cap = 0;
  float* att_o = nullptr;
  float2* att_ml = nullptr;
  size_t att_items_cap = 0;
  int item_total = 0;
  uint8_t* qtile = nullptr;  // [max_batch][Hkv] Q operand images of the decode attention
  // tensor-core prefill attention: bf16 q of the call's tokens, its TMA map, the work units
  uint16_t* qb = nullptr;  // [2][qb_rows][qd]: high parts, then remainders
  int qb_rows = 0;
  CUtensorMap q_map;
  std::vector<PrefillUnit> hunits;
  PrefillUnit* pf_units = nullptr;
  size_t pf_cap = 0;
  int pf_n = 0;
  float* ss = nullptr;       // [d/128][ss_ld] per-tile sums of squares of the residual rows
  int ss_ld = 0;
  // staging buffer for host-side import/export of V
  uint16_t* stage = nullptr;
  size_t stage_elems = 0;
  // captured decode steps, keyed by (B, last_tokens, logits, next_tokens)
  struct Captured {
    cudaGraphExec_t exec;
    std::vector<int> stamp_cls;  // kernel class of each stamp slot of the captured step
  };
  std::map<std::tuple<int, const void*, const void*, const void*, bool>, Captured> graphs;
  // measurement stamps (cbt_engine_set_stamps): per stamped launch of a step, [begin, end]
  // failure-detection test (cbt_engine_test_stall): the next decode step's lm_head projection
  // requests nothing and its waits give up after stall_limit polls
  uint32_t stall_limit = 0;
  bool stall_now = false;
  bool stamps_on = false;
  unsigned long long* stamp_buf = nullptr;  // [kStampSlots][2]
  int stamp_n = 0;
  std::vector<int> stamp_cls, last_stamp_cls;

  // measurement: event pairs around launch groups of selected kernel classes
  struct TimeRec {
    int cls;
    cudaEvent_t a, b;
    double bytes;
  };
  int timing_mask = 0;
  std::vector<cudaEvent_t> ev_pool;
  size_t ev_used = 0;
  std::vector<TimeRec> recs;

  int qd() const { return cfg.n_heads * cfg.head_dim; }
  int kvd() const { return cfg.n_kv_heads * cfg.head_dim; }
};

extern "C" const char* cbt_status_str(cbt_status s) {
  switch (s) {
    case CBT_OK: return "ok";
    case CBT_ERR_INVALID: return "invalid argument or configuration";
    case CBT_ERR_NULL: return "required pointer is NULL";
    case CBT_ERR_BAD_SLAB: return "unknown or freed slab id";
    case CBT_ERR_DUP_SLAB: return "slab id repeated in one call";
    case CBT_ERR_BATCH: return "batch larger than max_batch";
    case CBT_ERR_CAPACITY: return "slab capacity exceeded";
    case CBT_ERR_POOL_EXHAUSTED: return "KV arena has no free extent large enough";
    case CBT_ERR_TOKENS: return "prefill tokens above max_prefill_tokens";
    case CBT_ERR_CUDA: return "CUDA runtime error";
    case CBT_ERR_DEVICE: return "device error word set";
    case CBT_ERR_UNSUPPORTED: return "shape not supported";
    case CBT_ERR_LIMIT: return "size above the fixed no-allocation scratch";
    default: return "unknown status";
  }
}

static void free_scratch(cbt_engine* e) {
  void* ptrs[] = {e->x,       e->h,        e->qkv,  e->o,     e->act,    e->part,
                  e->xg,      e->logits,   e->cosv, e->sinv,  e->next_tok, e->last_idx,
                  e->rows,    e->err,      e->act_h, e->act_o, e->act_u,
                  e->items,    e->item_meta, e->att_o, e->att_ml, e->stage,
                  e->qtile,   e->ss,       e->qb,     e->pf_units, e->q4_arena, e->pagetab,
                  e->tok_pages, e->kv8_jobs, e->q4x};
  for (void* q : ptrs)
    if (q) cudaFree(q);
}

static bool linear_ok(const cbt_linear& l, int fmt) {
  if (!l.w) return false;
  if (fmt == CBT_WEIGHTS_AFFINE4 && (!l.scales || !l.biases)) return false;
  return true;
}

// slab capacities are whole 64-key groups (the V layout transposes groups of 64 keys)
static int round_cap(int cap) { return (cap + 63) & ~63; }

extern "C" size_t cbt_slab_bytes(const cbt_model_config* c, int32_t cap) {
  if (!c || cap <= 0) return 0;
  size_t b = (size_t)c->n_layers * 2 * c->n_kv_heads * (size_t)round_cap(cap) * c->head_dim * 2;
  return (b + kSlabAlign - 1) & ~(kSlabAlign - 1);
}

extern "C" size_t cbt_slab_bytes_kvq(const cbt_model_config* c, int32_t cap, int32_t bits) {
  if (!c || cap <= 0 || c->head_dim % 64 || (bits != 8 && bits != 4)) return 0;
  size_t b = (size_t)c->n_layers * 2 * c->n_kv_heads *
             (size_t)kvq_block_bytes(round_cap(cap), c->head_dim, bits);
  return (b + kSlabAlign - 1) & ~(kSlabAlign - 1);
}

extern "C" size_t cbt_slab_bytes_kv8(const cbt_model_config* c, int32_t cap) {
  return cbt_slab_bytes_kvq(c, cap, 8);
}

static bool take_extent(cbt_engine* e, size_t need, size_t* off_out);

// bytes of one of the engine's slabs
static size_t slab_bytes(const cbt_engine* e, int cap) {
  return e->quant() ? cbt_slab_bytes_kvq(&e->cfg, cap, e->kv_bits) : cbt_slab_bytes(&e->cfg, cap);
}

extern "C" cbt_status cbt_engine_create(const cbt_model_config* cfg, const cbt_weights* w,
                                        const cbt_engine_params* p, cbt_engine** out) {
  if (!out) return CBT_ERR_NULL;
  *out = nullptr;
  if (!cfg || !w || !p || !w->layers || !w->embed || !w->final_norm || !p->kv_arena)
    return CBT_ERR_NULL;
  const cbt_model_config& c = *cfg;
  if (c.n_layers <= 0 || c.d_model <= 0 || c.n_heads <= 0 || c.n_kv_heads <= 0 || c.d_ff <= 0 ||
      c.vocab <= 0 || c.n_heads % c.n_kv_heads != 0 || !(c.rms_eps >= 0.f) || !(c.rope_theta > 0))
    return CBT_ERR_INVALID;
  if (c.weight_format != CBT_WEIGHTS_BF16 && c.weight_format != CBT_WEIGHTS_AFFINE4)
    return CBT_ERR_INVALID;
  if (c.weight_format == CBT_WEIGHTS_AFFINE4 && c.group_size != 64) return CBT_ERR_UNSUPPORTED;
  if (c.head_dim != 64 && c.head_dim != 128) return CBT_ERR_UNSUPPORTED;
  const int qd = c.n_heads * c.head_dim;
  if (c.d_model % 256 || qd % 256 || c.d_ff % 256) return CBT_ERR_UNSUPPORTED;
  if (p->max_batch <= 0 || p->max_prefill_tokens <= 0 || p->kv_arena_bytes < kSlabAlign ||
      (reinterpret_cast<uintptr_t>(p->kv_arena) & 255) || p->kv_page_tokens < 0 ||
      p->kv_page_tokens % 128 ||
      (p->kv_bits != 0 && p->kv_bits != 16 && p->kv_bits != 8 && p->kv_bits != 4))
    return CBT_ERR_INVALID;
  const bool qkv = p->kv_bits == 8 || p->kv_bits == 4;
  // the quantised-KV decode attention is built for 1, 2, 4 or 8 q heads per kv head
  if (qkv && c.n_heads / c.n_kv_heads != 1 && c.n_heads / c.n_kv_heads != 2 &&
      c.n_heads / c.n_kv_heads != 4 && c.n_heads / c.n_kv_heads != 8)
    return CBT_ERR_UNSUPPORTED;
  if (!linear_ok(w->lm_head, c.weight_format)) return CBT_ERR_NULL;
  for (int l = 0; l < c.n_layers; ++l) {
    const cbt_layer_weights& L = w->layers[l];
    if (!linear_ok(L.wqkv, c.weight_format) || !linear_ok(L.wo, c.weight_format) ||
        !linear_ok(L.wgu, c.weight_format) || !linear_ok(L.wd, c.weight_format) || !L.attn_norm ||
        !L.ffn_norm)
      return CBT_ERR_NULL;
  }

  cbt_engine* e = new (std::nothrow) cbt_engine();
  if (!e) return CBT_ERR_INVALID;
  e->cfg = c;
  e->layers.assign(w->layers, w->layers + c.n_layers);
  e->w = *w;
  e->w.layers = e->layers.data();
  e->p = *p;
  e->stream = static_cast<cudaStream_t>(p->stream);
  e->free_ext[0] = p->kv_arena_bytes & ~(kSlabAlign - 1);
  e->page = p->kv_page_tokens;
  e->kv_bits = qkv ? p->kv_bits : 16;
  e->page_bytes = e->page ? slab_bytes(e, e->page) : 0;
  if (e->quant()) {  // the decode rows' staging slabs, one 128-position page each
    e->stage_bytes = cbt_slab_bytes(&c, 128);
    size_t off = 0;
    if (!take_extent(e, (size_t)p->max_batch * e->stage_bytes, &off)) {
      delete e;
      return CBT_ERR_POOL_EXHAUSTED;
    }
    e->stage_off = off;
  }

  const int T = std::max(p->max_batch, p->max_prefill_tokens);
  e->tmax = T;
  const int kvd = c.n_kv_heads * c.head_dim;
  const int nqkv = qd + 2 * kvd;
  const int Mmax = std::max({nqkv, c.d_model, 2 * c.d_ff, c.vocab});
  int smax = 1;
  for (int K : {c.d_model, qd, c.d_ff}) {
    int ks = K % 1024 == 0 ? 1024 : (K % 512 == 0 ? 512 : 256);
    smax = std::max(smax, K / ks);
  }
  e->part_floats = (size_t)smax * std::min(T, 32) * Mmax;
  size_t tot = 0;
  cudaError_t rc = cudaSuccess;
  auto chk = [&](cudaError_t r) { if (rc == cudaSuccess) rc = r; };
  chk(dmalloc(&e->x, (size_t)T * c.d_model, &tot));
  chk(dmalloc(&e->h, (size_t)T * std::max(c.d_model, qd), &tot));
  chk(dmalloc(&e->qkv, (size_t)T * nqkv, &tot));
  chk(dmalloc(&e->o, (size_t)T * qd, &tot));
  chk(dmalloc(&e->act, (size_t)T * c.d_ff, &tot));
  chk(dmalloc(&e->part, e->part_floats, &tot));
  chk(dmalloc(&e->xg, (size_t)p->max_batch * c.d_model * 2, &tot));
  chk(dmalloc(&e->logits, (size_t)p->max_batch * c.vocab, &tot));
  chk(dmalloc(&e->cosv, (size_t)T * c.head_dim / 2, &tot));
  chk(dmalloc(&e->sinv, (size_t)T * c.head_dim / 2, &tot));
  chk(dmalloc(&e->next_tok, (size_t)p->max_batch, &tot));
  chk(dmalloc(&e->last_idx, (size_t)p->max_batch, &tot));
  chk(dmalloc(&e->rows, (size_t)T, &tot));
  chk(dmalloc(&e->err, 2, &tot));
  if (e->quant()) {
    e->kv8_jobs_cap = (size_t)std::max(p->max_batch, 64);
    chk(dmalloc(&e->kv8_jobs, e->kv8_jobs_cap, &tot));
  }
  if (rc == cudaSuccess) rc = cudaMemsetAsync(e->err, 0, 2 * sizeof(int), e->stream);
  bool maps_ok = true;
  const bool bf16w = c.weight_format == CBT_WEIGHTS_BF16;
  if (rc == cudaSuccess && (bf16w || (c.d_model % 128 == 0 && qd % 128 == 0 && c.d_ff % 128 == 0))) {
    // tensor-core path: weight descriptors (bf16) or native 4-bit blocks, bf16 operand
    // buffers
    int dev = 0;
    chk(cudaGetDevice(&dev));
    chk(cudaDeviceGetAttribute(&e->num_sms, cudaDevAttrMultiProcessorCount, dev));
    e->act_rows = std::max(64, 2 * T);  // hi rows, then (prefill) the lo rows from row T
    chk(dmalloc(&e->act_h, (size_t)e->act_rows * std::max(c.d_model, qd), &tot));
    chk(dmalloc(&e->act_o, (size_t)e->act_rows * qd, &tot));
    chk(dmalloc(&e->act_u, (size_t)e->act_rows * c.d_ff, &tot));
    if (rc == cudaSuccess) {
      const size_t arows = e->act_rows;
      for (uint16_t* a : {e->act_h, e->act_o, e->act_u}) {
        size_t cols = a == e->act_u ? c.d_ff : (a == e->act_o ? qd : std::max(c.d_model, qd));
        rc = cudaMemsetAsync(a, 0, arows * cols * 2, e->stream);
        if (rc != cudaSuccess) break;
      }
    }
    e->wmaps.resize(c.n_layers);
    e->wmaps_kb.resize(c.n_layers);
    e->q4w.resize(c.n_layers);
    for (int l = 0; l < c.n_layers && maps_ok && bf16w; ++l) {
      const cbt_layer_weights& L = w->layers[l];
      maps_ok = make_tmap_bf16(&e->wmaps[l].qkv, L.wqkv.w, c.d_model, nqkv, 64, 64) &&
                make_tmap_bf16(&e->wmaps[l].o, L.wo.w, qd, c.d_model, 64, 64) &&
                make_tmap_bf16(&e->wmaps[l].gu, L.wgu.w, c.d_model, 2 * c.d_ff, 64, 64) &&
                make_tmap_bf16(&e->wmaps[l].d, L.wd.w, c.d_ff, c.d_model, 64, 64);
    }
    maps_ok = maps_ok && (!bf16w || make_tmap_bf16(&e->lm_map, w->lm_head.w, c.d_model, c.vocab, 64, 64));
    for (int l = 0; l < c.n_layers && maps_ok && bf16w; ++l) {
      const cbt_layer_weights& L = w->layers[l];
      maps_ok = make_tmap_kblocks(&e->wmaps_kb[l].qkv, L.wqkv.w, c.d_model, nqkv, 128, kCskBlocks, 0) &&
                make_tmap_kblocks(&e->wmaps_kb[l].o, L.wo.w, qd, c.d_model, 128, kCskBlocks, 0) &&
                make_tmap_kblocks(&e->wmaps_kb[l].gu, L.wgu.w, c.d_model, 2 * c.d_ff, 64, kCskBlocks,
                                  c.d_ff) &&
                make_tmap_kblocks(&e->wmaps_kb[l].d, L.wd.w, c.d_ff, c.d_model, 128, kCskBlocks, 0);
    }
    maps_ok = maps_ok && (!bf16w || make_tmap_kblocks(&e->lm_map_kb, w->lm_head.w, c.d_model,
                                                      c.vocab, 128, kCskBlocks, 0));
    if (!bf16w && maps_ok && rc == cudaSuccess) {
      // every 4-bit matrix once into the native block layout of the decode projections
      struct Mat {
        const cbt_linear* lin;
        int M, K, F;
        uint8_t** dst;
      };
      std::vector<Mat> mats;
      for (int l = 0; l < c.n_layers; ++l) {
        const cbt_layer_weights& L = w->layers[l];
        mats.push_back({&L.wqkv, nqkv, c.d_model, 0, &e->q4w[l].qkv});
        mats.push_back({&L.wo, c.d_model, qd, 0, &e->q4w[l].o});
        mats.push_back({&L.wgu, 2 * c.d_ff, c.d_model, c.d_ff, &e->q4w[l].gu});
        mats.push_back({&L.wd, c.d_model, c.d_ff, 0, &e->q4w[l].d});
      }
      mats.push_back({&w->lm_head, c.vocab, c.d_model, 0, &e->q4_lm});
      size_t total = 0;
      for (const Mat& m : mats) total += q4_native_bytes(m.M, m.K, m.F);
      chk(dmalloc(&e->q4_arena, total, &tot));
      size_t off = 0;
      for (const Mat& m : mats) {
        if (rc != cudaSuccess || !maps_ok) break;
        *m.dst = e->q4_arena + off;
        maps_ok = launch_q4_repack(static_cast<const uint32_t*>(m.lin->w),
                                   static_cast<const uint16_t*>(m.lin->scales),
                                   static_cast<const uint16_t*>(m.lin->biases), m.M, m.K, m.F,
                                   *m.dst, e->stream);
        off += q4_native_bytes(m.M, m.K, m.F);
      }
      if (T > 32 && maps_ok && rc == cudaSuccess) {
        // projections over more than 32 rows run as dense tensor-core GEMMs over the expanded
        // matrix (the head too when more than 32 rows may ask for logits)
        const int shp[cbt_engine::kQ4xShapes][2] = {
            {nqkv, c.d_model}, {c.d_model, qd}, {2 * c.d_ff, c.d_model}, {c.d_model, c.d_ff},
            {c.vocab, c.d_model}};
        const int nshape = p->max_batch > 32 ? cbt_engine::kQ4xShapes : cbt_engine::kQ4xLm;
        size_t emax = 0;
        for (int i = 0; i < nshape; ++i) emax = std::max(emax, (size_t)shp[i][0] * shp[i][1]);
        chk(dmalloc(&e->q4x, 2 * emax, &tot));
        e->q4x_elems = emax;
        for (int i = 0; i < nshape && rc == cudaSuccess && maps_ok; ++i)
          maps_ok = make_tmap_bf16(&e->q4x_maps[i][0], e->q4x, shp[i][1], shp[i][0], 64, 64) &&
                    make_tmap_bf16(&e->q4x_maps[i][1], e->q4x + emax, shp[i][1], shp[i][0], 64, 64);
      }
    }
    // the whole arena seen as K rows (head_dim wide) and as V^T rows (64 keys wide)
    const uint64_t arena_elems = p->kv_arena_bytes / 2;
    maps_ok = maps_ok && arena_elems / 64 < (1ull << 31) &&
              make_tmap_bf16(&e->kv_kmap, p->kv_arena, c.head_dim, arena_elems / c.head_dim, 64,
                             128) &&
              make_tmap_bf16(&e->kv_vmap, p->kv_arena, 64, arena_elems / 64, 64, c.head_dim);
    if (rc == cudaSuccess) {
      e->hitem_base.resize(p->max_batch);
      e->hitem_count.resize(p->max_batch);
      chk(dmalloc(&e->item_meta, (size_t)2 * p->max_batch + 1, &tot));
      const size_t qbytes = (size_t)p->max_batch * c.n_kv_heads * 16 * c.head_dim * 2;
      chk(dmalloc(&e->qtile, qbytes, &tot));
      e->qb_rows = std::max(T, 128);  // at least one 128-row TMA box
      const size_t qb_elems = (size_t)2 * e->qb_rows * qd;
      chk(dmalloc(&e->qb, qb_elems, &tot));
      if (rc == cudaSuccess) rc = cudaMemsetAsync(e->qb, 0, qb_elems * 2, e->stream);
      maps_ok = maps_ok && rc == cudaSuccess &&
                make_tmap_bf16(&e->q_map, e->qb, qd, 2 * e->qb_rows, 64, 128);
      if (rc == cudaSuccess) rc = cudaMemsetAsync(e->qtile, 0, qbytes, e->stream);
      e->ss_ld = std::max(32, p->max_batch);
      chk(dmalloc(&e->ss, (size_t)((c.d_model + 127) / 128) * e->ss_ld, &tot));
    }
    e->use_tc = maps_ok && c.d_ff % 64 == 0;
  }
  if (rc == cudaSuccess) rc = cudaStreamSynchronize(e->stream);
  if (rc == cudaSuccess && maps_ok && e->quant() && !e->use_tc) maps_ok = false;
  if (rc != cudaSuccess || !maps_ok) {
    free_scratch(e);
    delete e;
    return rc != cudaSuccess ? CBT_ERR_CUDA : CBT_ERR_UNSUPPORTED;
  }
  e->scratch_bytes = tot;
  e->hrows.resize(T);
  e->hidx.resize(p->max_batch);
  *out = e;
  return CBT_OK;
}

extern "C" cbt_status cbt_engine_destroy(cbt_engine* e) {
  if (!e) return CBT_ERR_NULL;
  cudaError_t rc = cudaStreamSynchronize(e->stream);
  free_scratch(e);
  for (cudaEvent_t ev : e->ev_pool) cudaEventDestroy(ev);
  for (auto& kv : e->graphs) cudaGraphExecDestroy(kv.second.exec);
  if (e->stamp_buf) cudaFree(e->stamp_buf);
  delete e;
  return rc == cudaSuccess ? CBT_OK : CBT_ERR_CUDA;
}

// ---- slab allocator ---------------------------------------------------------------------
// first fit: an extent of `need` bytes, or false
static bool take_extent(cbt_engine* e, size_t need, size_t* off_out) {
  for (auto it = e->free_ext.begin(); it != e->free_ext.end(); ++it) {
    if (it->second >= need) {
      size_t off = it->first, rest = it->second - need;
      e->free_ext.erase(it);
      if (rest) e->free_ext[off + need] = rest;
      e->in_use += need;
      *off_out = off;
      return true;
    }
  }
  return false;
}

static void give_extent(cbt_engine* e, size_t off, size_t bytes);

// The QueryRow base and capacity of the slab, or the page, that holds position pos: a page
// holding positions [s, s + page) at element offset o has base o - s * head_dim, so the
// kernels' index helpers take global positions.
static bool paged(const cbt_engine* e, const Slab& sl) { return e->page && !sl.flat; }

static long long row_base(const cbt_engine* e, const Slab& sl, int pos) {
  if (!paged(e, sl)) return (long long)(sl.offset / 2);
  const int pg = pos / e->page;
  return (long long)(sl.pages[pg] / 2) - (long long)pg * e->page * e->cfg.head_dim;
}
static int row_cap(const cbt_engine* e, const Slab& sl) { return paged(e, sl) ? e->page : sl.lcap; }

// Quantised KV: the slab or page holding position pos (byte offset, layout capacity, first
// position)
struct QLoc {
  long long off;
  int cap, p0;
};
static QLoc qloc(const cbt_engine* e, const Slab& sl, int pos) {
  if (!paged(e, sl)) return QLoc{(long long)sl.offset, sl.lcap, 0};
  const int pg = pos / e->page;
  return QLoc{(long long)sl.pages[pg], e->page, pg * e->page};
}

// pages obtainable from the free list (in a paged engine every extent taken is one page, so
// each free extent is a run of page slots, the last one possibly followed by a remainder)
static size_t free_pages(const cbt_engine* e) {
  size_t n = 0;
  for (const auto& kv : e->free_ext) n += kv.second / e->page_bytes;
  return n;
}

// one holder lets go of a page; the last one returns it to the arena
static void release_page(cbt_engine* e, size_t off) {
  auto it = e->extra_holders.find(off);
  if (it == e->extra_holders.end()) {
    give_extent(e, off, e->page_bytes);
  } else if (--it->second == 0) {
    e->extra_holders.erase(it);
  }
}

struct PageWrite {
  int id;
  long long lo, hi;  // the call writes positions [lo, hi) of slab id
};

// Paged engines, before a call queues writes: each listed slab gets pages for positions
// [0, hi), and every page that [lo, hi) touches and another slab also holds is replaced by a
// private copy of it (the copy queued on the stream ahead of the write).  The pages needed are
// counted first, the counting following the same order as the replacement (a page whose
// other holders all copied it away becomes private), so a call the arena cannot serve fails
// with CBT_ERR_POOL_EXHAUSTED before anything changes.
static cbt_status prepare_writes(cbt_engine* e, const std::vector<PageWrite>& writes) {
  if (!e->page) return CBT_OK;
  const long long P = e->page;
  size_t need = 0;
  std::unordered_map<size_t, int> copied;
  for (const PageWrite& w : writes) {
    const Slab& sl = e->slabs[w.id];
    if (sl.flat) continue;
    const long long have = (long long)sl.pages.size(), want = (w.hi + P - 1) / P;
    if (want > have) need += (size_t)(want - have);
    for (long long pg = w.lo / P; w.lo < w.hi && pg < std::min(have, want); ++pg) {
      auto it = e->extra_holders.find(sl.pages[pg]);
      if (it != e->extra_holders.end() && it->second > copied[sl.pages[pg]]) {
        ++need;
        ++copied[sl.pages[pg]];
      }
    }
  }
  if (need > free_pages(e)) return CBT_ERR_POOL_EXHAUSTED;
  char* arena = static_cast<char*>(e->p.kv_arena);
  for (const PageWrite& w : writes) {
    Slab& sl = e->slabs[w.id];
    if (sl.flat) continue;
    const long long have = (long long)sl.pages.size(), want = (w.hi + P - 1) / P;
    for (long long pg = w.lo / P; w.lo < w.hi && pg < std::min(have, want); ++pg) {
      if (!e->extra_holders.count(sl.pages[pg])) continue;
      size_t off = 0;
      take_extent(e, e->page_bytes, &off);  // cannot fail: counted above
      if (cudaMemcpyAsync(arena + off, arena + sl.pages[pg], e->page_bytes,
                          cudaMemcpyDeviceToDevice, e->stream) != cudaSuccess) {
        give_extent(e, off, e->page_bytes);
        return CBT_ERR_CUDA;
      }
      release_page(e, sl.pages[pg]);
      sl.pages[pg] = off;
    }
    while ((long long)sl.pages.size() < want) {
      size_t off = 0;
      take_extent(e, e->page_bytes, &off);
      sl.pages.push_back(off);
    }
  }
  return CBT_OK;
}

extern "C" cbt_status cbt_kv_slab_alloc(cbt_engine* e, int32_t cap, int32_t* id) {
  if (!e || !id) return CBT_ERR_NULL;
  if (cap <= 0) return CBT_ERR_INVALID;
  if (e->page) {  // pages are taken as positions are written
    int sid = e->next_id++;
    e->slabs[sid] = Slab{0, 0, cap, 0, round_cap(cap), {}};
    *id = sid;
    return CBT_OK;
  }
  size_t need = slab_bytes(e, cap), off;
  if (!take_extent(e, need, &off)) return CBT_ERR_POOL_EXHAUSTED;
  int sid = e->next_id++;
  e->slabs[sid] = Slab{off, need, cap, 0, round_cap(cap), {}};
  *id = sid;
  return CBT_OK;
}

extern "C" cbt_status cbt_kv_slab_free(cbt_engine* e, int32_t id) {
  if (!e) return CBT_ERR_NULL;
  auto it = e->slabs.find(id);
  if (it == e->slabs.end()) return CBT_ERR_BAD_SLAB;
  if (e->page) {
    for (size_t off : it->second.pages) release_page(e, off);
    e->slabs.erase(it);
    return CBT_OK;
  }
  size_t off = it->second.offset, bytes = it->second.bytes;
  e->slabs.erase(it);
  give_extent(e, off, bytes);
  return CBT_OK;
}

// return an extent to the free list, merged with its neighbours
static void give_extent(cbt_engine* e, size_t off, size_t bytes) {
  e->in_use -= bytes;
  auto nx = e->free_ext.lower_bound(off);
  if (nx != e->free_ext.end() && off + bytes == nx->first) {  // merge with the next extent
    bytes += nx->second;
    nx = e->free_ext.erase(nx);
  }
  if (nx != e->free_ext.begin()) {  // merge with the previous extent
    auto pv = std::prev(nx);
    if (pv->first + pv->second == off) {
      pv->second += bytes;
      return;
    }
  }
  e->free_ext[off] = bytes;
}

extern "C" cbt_status cbt_retire(cbt_engine* e, const int32_t* ids, int32_t n) {
  if (!e) return CBT_ERR_NULL;
  if (n < 0) return CBT_ERR_INVALID;
  if (n > 0 && !ids) return CBT_ERR_NULL;
  std::unordered_set<int> seen;
  for (int i = 0; i < n; ++i) {
    if (!e->slabs.count(ids[i])) return CBT_ERR_BAD_SLAB;
    if (!seen.insert(ids[i]).second) return CBT_ERR_DUP_SLAB;
  }
  for (int i = 0; i < n; ++i) cbt_kv_slab_free(e, ids[i]);
  return CBT_OK;
}

extern "C" cbt_status cbt_kv_slab_position(cbt_engine* e, int32_t id, int32_t* pos) {
  if (!e || !pos) return CBT_ERR_NULL;
  auto it = e->slabs.find(id);
  if (it == e->slabs.end()) return CBT_ERR_BAD_SLAB;
  *pos = it->second.pos;
  return CBT_OK;
}

// ---- quantised KV: bf16 intermediates and their conversion ------------------------------------
// A bf16 slab of capacity cap for a call's intermediate K/V, one extent of the arena even on a
// paged engine (0 if the arena has no room).
static int temp_bf16_slab(cbt_engine* e, int cap) {
  const size_t need = cbt_slab_bytes(&e->cfg, cap);
  size_t off = 0;
  if (!take_extent(e, need, &off)) return 0;
  const int sid = e->next_id++;
  Slab t{off, need, cap, 0, round_cap(cap), {}};
  t.flat = true;
  e->slabs[sid] = t;
  return sid;
}

// Host bookkeeping only: work queued later on the stream runs after what used the slab.
static void drop_temp(cbt_engine* e, int sid) {
  auto it = e->slabs.find(sid);
  give_extent(e, it->second.offset, it->second.bytes);
  e->slabs.erase(it);
}

// Conversion records for positions [t0, t0 + n) of a bf16 source (QueryRow base and capacity)
// into quantised slab dst: one record per page the positions touch (one for a slab).
static void add_jobs(cbt_engine* e, long long src_base, int src_cap, int t0, int n, const Slab& dst) {
  int p = t0;
  while (p < t0 + n) {
    const QLoc q = qloc(e, dst, p);
    const int end = paged(e, dst) ? std::min(t0 + n, q.p0 + q.cap) : t0 + n;
    e->hjobs.push_back(Kv8Job{src_base, src_cap, p, end - p, q.cap, q.off, q.p0});
    p = end;
  }
}

static void drop_graphs(cbt_engine* e);

// Copy e->hjobs to the device (growing the buffer after the work that may still read it).
static cudaError_t upload_jobs(cbt_engine* e) {
  cudaError_t rc = cudaSuccess;
  if (e->hjobs.size() > e->kv8_jobs_cap) {
    rc = cudaStreamSynchronize(e->stream);
    drop_graphs(e);  // captured steps hold the old buffer address
    cudaFree(e->kv8_jobs);
    e->kv8_jobs = nullptr;
    e->kv8_jobs_cap = 0;
    const size_t cap = std::max(e->hjobs.size(), 2 * e->kv8_jobs_cap);
    if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->kv8_jobs), cap * sizeof(Kv8Job));
    if (rc != cudaSuccess) return rc;
    e->kv8_jobs_cap = cap;
  }
  e->q_jobs = (int)e->hjobs.size();
  e->q_jobs_max_n = 0;
  for (const Kv8Job& j : e->hjobs) e->q_jobs_max_n = std::max(e->q_jobs_max_n, j.n);
  if (e->hjobs.empty()) return cudaSuccess;
  return cudaMemcpyAsync(e->kv8_jobs, e->hjobs.data(), sizeof(Kv8Job) * e->hjobs.size(),
                         cudaMemcpyHostToDevice, e->stream);
}

// Queue the quantisation of e->hjobs (every layer) into their slabs.
static cudaError_t convert_jobs(cbt_engine* e) {
  cudaError_t rc = upload_jobs(e);
  if (rc != cudaSuccess) return rc;
  if (!launch_kvq_convert(e->kv8_jobs, e->q_jobs, e->q_jobs_max_n, 0, e->cfg.n_layers,
                          e->cfg.n_kv_heads, e->cfg.head_dim, e->kv_bits,
                          static_cast<uint8_t*>(e->p.kv_arena), e->stream))
    return cudaErrorLaunchFailure;
  return cudaSuccess;
}

static cbt_status slab_copy_bf16(cbt_engine* e, int32_t id, void* k, void* v, int32_t n,
                                 int32_t on_host, bool to_slab);
static cudaError_t upload_page_tables(cbt_engine* e);

// Export of a quantised slab: every position's K and V as bf16 (scale * code + bias in double,
// rounded to fp32, then to bf16), layer by layer through the device.
static cbt_status export_quant(cbt_engine* e, const Slab& s, void* k, void* v, int32_t n,
                               int32_t on_host) {
  const cbt_model_config& c = e->cfg;
  const size_t layer_elems = (size_t)c.n_kv_heads * n * c.head_dim;
  cudaError_t rc = cudaSuccess;
  if (on_host && e->stage_elems < 2 * layer_elems) {  // device staging of one layer's K and V
    rc = cudaStreamSynchronize(e->stream);
    if (e->stage) cudaFree(e->stage);
    e->stage = nullptr;
    e->stage_elems = 0;
    if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->stage), 4 * layer_elems);
    if (rc != cudaSuccess) return CBT_ERR_CUDA;
    e->stage_elems = 2 * layer_elems;
  }
  e->hpagetab.clear();
  if (paged(e, s))
    for (size_t off : s.pages) e->hpagetab.push_back((long long)off);
  else
    e->hpagetab.push_back((long long)s.offset);
  e->htok_pages.clear();
  rc = upload_page_tables(e);
  const int cap = paged(e, s) ? e->page : s.lcap;
  for (int l = 0; l < c.n_layers && rc == cudaSuccess; ++l) {
    uint16_t* ku = static_cast<uint16_t*>(k) + (size_t)l * layer_elems;
    uint16_t* vu = static_cast<uint16_t*>(v) + (size_t)l * layer_elems;
    uint16_t* kd = on_host ? e->stage : ku;
    uint16_t* vd = on_host ? e->stage + layer_elems : vu;
    if (!launch_kvq_export(static_cast<const uint8_t*>(e->p.kv_arena), e->pagetab, cap, l,
                           c.n_kv_heads, c.head_dim, n, e->kv_bits, kd, vd, e->stream)) {
      rc = cudaErrorLaunchFailure;
      break;
    }
    if (on_host) {
      rc = cudaMemcpyAsync(ku, kd, layer_elems * 2, cudaMemcpyDeviceToHost, e->stream);
      if (rc == cudaSuccess)
        rc = cudaMemcpyAsync(vu, vd, layer_elems * 2, cudaMemcpyDeviceToHost, e->stream);
      if (rc == cudaSuccess) rc = cudaStreamSynchronize(e->stream);  // the staging is reused
    }
  }
  return rc == cudaSuccess ? CBT_OK : CBT_ERR_CUDA;
}

// Import into a quantised slab: the plain K/V go to a bf16 intermediate slab, which is
// quantised; export dequantises (export_quant).
static cbt_status slab_copy(cbt_engine* e, int32_t id, void* k, void* v, int32_t n, int32_t on_host,
                            bool to_slab) {
  if (!e || !k || !v) return CBT_ERR_NULL;
  if (!e->quant()) return slab_copy_bf16(e, id, k, v, n, on_host, to_slab);
  auto it = e->slabs.find(id);
  if (it == e->slabs.end()) return CBT_ERR_BAD_SLAB;
  if (n < 0) return CBT_ERR_INVALID;
  if (!to_slab) {
    if (n > it->second.pos) return CBT_ERR_CAPACITY;
    if (n == 0) return CBT_OK;
    return export_quant(e, it->second, k, v, n, on_host);
  }
  if (n > it->second.cap) return CBT_ERR_CAPACITY;
  if (n == 0) {
    it->second.pos = 0;
    return CBT_OK;
  }
  const int tmp = temp_bf16_slab(e, n);
  if (!tmp) return CBT_ERR_POOL_EXHAUSTED;
  cbt_status st = prepare_writes(e, {{id, 0, (long long)n}});
  if (st == CBT_OK) st = slab_copy_bf16(e, tmp, k, v, n, on_host, true);
  if (st == CBT_OK) {
    const Slab& t = e->slabs[tmp];
    e->hjobs.clear();
    add_jobs(e, (long long)(t.offset / 2), t.lcap, 0, n, e->slabs[id]);
    if (convert_jobs(e) != cudaSuccess) st = CBT_ERR_CUDA;
  }
  drop_temp(e, tmp);
  if (st == CBT_OK) e->slabs[id].pos = n;
  return st;
}

static cbt_status slab_copy_bf16(cbt_engine* e, int32_t id, void* k, void* v, int32_t n,
                                 int32_t on_host, bool to_slab) {
  auto it = e->slabs.find(id);
  if (it == e->slabs.end()) return CBT_ERR_BAD_SLAB;
  Slab& s = it->second;
  if (n < 0) return CBT_ERR_INVALID;
  if (n > s.cap || (!to_slab && n > s.pos)) return CBT_ERR_CAPACITY;
  if (to_slab) {
    const cbt_status st = prepare_writes(e, {{id, 0, (long long)n}});
    if (st != CBT_OK) return st;
  }
  const cbt_model_config& c = e->cfg;
  const size_t row = (size_t)c.head_dim * 2;
  cudaMemcpyKind kind = on_host ? (to_slab ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToHost)
                                : cudaMemcpyDeviceToDevice;
  cudaError_t rc = cudaSuccess;
  const size_t layer_elems = (size_t)c.n_kv_heads * n * c.head_dim;
  if (on_host && n > 0 && e->stage_elems < layer_elems) {  // staging for the V transposition
    rc = cudaStreamSynchronize(e->stream);
    if (e->stage) cudaFree(e->stage);
    e->stage = nullptr;
    e->stage_elems = 0;
    if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->stage), layer_elems * 2);
    if (rc != cudaSuccess) return CBT_ERR_CUDA;
    e->stage_elems = layer_elems;
  }
  // runs of positions: the whole slab, or page by page
  const int P = row_cap(e, s);
  const bool pg = paged(e, s);
  const int runs = pg ? (n + P - 1) / P : (n > 0 ? 1 : 0);
  for (int l = 0; l < c.n_layers && rc == cudaSuccess && n > 0; ++l) {
    uint16_t* vu = static_cast<uint16_t*>(v) + (size_t)l * layer_elems;
    uint16_t* plain = on_host ? e->stage : vu;
    if (on_host && to_slab)
      rc = cudaMemcpyAsync(plain, vu, layer_elems * 2, cudaMemcpyHostToDevice, e->stream);
    for (int r = 0; r < runs && rc == cudaSuccess; ++r) {
      const int a = pg ? r * P : 0, cnt = pg ? std::min(n, a + P) - a : n;
      char* blk = static_cast<char*>(e->p.kv_arena) + (pg ? s.pages[r] : s.offset);
      // K: rows [a, a + cnt) of each kv head's [position][head_dim] block
      char* user = static_cast<char*>(k) + ((size_t)l * c.n_kv_heads * n + a) * row;
      char* slab = blk + ((size_t)l * 2) * c.n_kv_heads * (size_t)P * row;
      size_t upitch = (size_t)n * row, spitch = (size_t)P * row, width = (size_t)cnt * row;
      if (to_slab)
        rc = cudaMemcpy2DAsync(slab, spitch, user, upitch, width, c.n_kv_heads, kind, e->stream);
      else
        rc = cudaMemcpy2DAsync(user, upitch, slab, spitch, width, c.n_kv_heads, kind, e->stream);
      if (rc != cudaSuccess) break;
      // V: transposed 64-key groups in the slab, converted on the device
      const QueryRow qr{row_base(e, s, a), 0, P};
      launch_v_convert(plain, static_cast<uint16_t*>(e->p.kv_arena), qr, l, c.n_kv_heads, a, cnt,
                       n, c.head_dim, to_slab, e->stream);
      rc = cudaGetLastError();
    }
    if (rc == cudaSuccess && on_host && !to_slab)
      rc = cudaMemcpyAsync(vu, plain, layer_elems * 2, cudaMemcpyDeviceToHost, e->stream);
  }
  if (rc == cudaSuccess && on_host && !to_slab) rc = cudaStreamSynchronize(e->stream);
  if (rc != cudaSuccess) return CBT_ERR_CUDA;
  if (to_slab) s.pos = n;
  return CBT_OK;
}

extern "C" cbt_status cbt_kv_slab_import(cbt_engine* e, int32_t id, const void* k, const void* v,
                                         int32_t n, int32_t on_host) {
  return slab_copy(e, id, const_cast<void*>(k), const_cast<void*>(v), n, on_host, true);
}

extern "C" cbt_status cbt_kv_slab_export(cbt_engine* e, int32_t id, void* k, void* v, int32_t n,
                                         int32_t on_host) {
  return slab_copy(e, id, k, v, n, on_host, false);
}

// Quantised slabs: each (layer, K|V, kv head) block holds codes, scales and biases position by
// position, so the prefix is three strided copies per run of positions (the slab, or a page).
static cbt_status copy_prefix_quant(cbt_engine* e, const Slab& src, const Slab& dst, int n) {
  const cbt_model_config& c = e->cfg;
  const int hd = c.head_dim, bits = e->kv_bits, row = hd * bits / 8, ng = hd / 64;
  const size_t blocks = (size_t)c.n_layers * 2 * c.n_kv_heads;
  char* arena = static_cast<char*>(e->p.kv_arena);
  for (int p = 0; p < n;) {
    const QLoc a = qloc(e, src, p), b = qloc(e, dst, p);
    const int end = std::min(n, std::min(a.p0 + a.cap, b.p0 + b.cap));
    const size_t m = (size_t)(end - p);
    const size_t la = (size_t)(p - a.p0), lb = (size_t)(p - b.p0);
    const size_t pa = (size_t)kvq_block_bytes(a.cap, hd, bits), pb = (size_t)kvq_block_bytes(b.cap, hd, bits);
    // codes, then scales, then biases of positions [p, end)
    const size_t sa[3] = {la * row, (size_t)a.cap * row + la * ng * 2,
                          (size_t)a.cap * row + (size_t)a.cap * ng * 2 + la * ng * 2};
    const size_t sb[3] = {lb * row, (size_t)b.cap * row + lb * ng * 2,
                          (size_t)b.cap * row + (size_t)b.cap * ng * 2 + lb * ng * 2};
    const size_t w[3] = {m * row, m * ng * 2, m * ng * 2};
    for (int r = 0; r < 3; ++r)
      if (cudaMemcpy2DAsync(arena + b.off + sb[r], pb, arena + a.off + sa[r], pa, w[r], blocks,
                            cudaMemcpyDeviceToDevice, e->stream) != cudaSuccess)
        return CBT_ERR_CUDA;
    p = end;
  }
  return CBT_OK;
}

extern "C" cbt_status cbt_kv_slab_copy_prefix(cbt_engine* e, int32_t src_id, int32_t dst_id,
                                              int32_t n) {
  if (!e) return CBT_ERR_NULL;
  auto si = e->slabs.find(src_id), di = e->slabs.find(dst_id);
  if (si == e->slabs.end() || di == e->slabs.end()) return CBT_ERR_BAD_SLAB;
  if (src_id == dst_id || n < 0) return CBT_ERR_INVALID;
  const Slab& src = si->second;
  Slab& dst = di->second;
  if (n > src.pos || n > dst.cap) return CBT_ERR_CAPACITY;
  const cbt_status st = prepare_writes(e, {{dst_id, 0, (long long)n}});
  if (st != CBT_OK) return st;
  if (e->quant()) {
    const cbt_status qs = copy_prefix_quant(e, src, dst, n);
    if (qs == CBT_OK) dst.pos = n;
    return qs;
  }
  // every (layer, K|V, kv head) block is a run of positions at the same place in both slabs (or
  // pages): one strided copy per run, of whole 64-position groups (a V block keeps each group
  // of 64 positions transposed; capacities and page sizes are multiples of 64, so the groups
  // line up)
  const cbt_model_config& c = e->cfg;
  const size_t row = (size_t)c.head_dim * 2;
  const size_t blocks = (size_t)c.n_layers * 2 * c.n_kv_heads;
  const int runs = e->page ? (n + e->page - 1) / e->page : (n > 0 ? 1 : 0);
  for (int r = 0; r < runs; ++r) {
    const int m = e->page ? std::min(e->page, n - r * e->page) : n;
    const size_t width = (size_t)((m + 63) / 64 * 64) * row;
    const char* from = static_cast<const char*>(e->p.kv_arena) + (e->page ? src.pages[r] : src.offset);
    char* to = static_cast<char*>(e->p.kv_arena) + (e->page ? dst.pages[r] : dst.offset);
    const size_t sp = (size_t)row_cap(e, src) * row, dp = (size_t)row_cap(e, dst) * row;
    if (cudaMemcpy2DAsync(to, dp, from, sp, width, blocks, cudaMemcpyDeviceToDevice, e->stream) !=
        cudaSuccess)
      return CBT_ERR_CUDA;
  }
  dst.pos = n;
  return CBT_OK;
}

extern "C" cbt_status cbt_kv_slab_share_prefix(cbt_engine* e, int32_t src_id, int32_t dst_id,
                                               int32_t n) {
  if (!e) return CBT_ERR_NULL;
  auto si = e->slabs.find(src_id), di = e->slabs.find(dst_id);
  if (si == e->slabs.end() || di == e->slabs.end()) return CBT_ERR_BAD_SLAB;
  if (src_id == dst_id || n < 0 || di->second.pos != 0) return CBT_ERR_INVALID;
  if (!e->page) return cbt_kv_slab_copy_prefix(e, src_id, dst_id, n);
  const Slab& src = si->second;
  Slab& dst = di->second;
  if (n > src.pos || n > dst.cap) return CBT_ERR_CAPACITY;
  for (size_t off : dst.pages) release_page(e, off);
  dst.pages.clear();
  for (int pg = 0; pg < (n + e->page - 1) / e->page; ++pg) {
    dst.pages.push_back(src.pages[pg]);
    ++e->extra_holders[src.pages[pg]];
  }
  dst.pos = n;
  return CBT_OK;
}

// ---- measurement ------------------------------------------------------------------------
static cudaEvent_t next_event(cbt_engine* e) {
  if (e->ev_used == e->ev_pool.size()) {
    cudaEvent_t ev;
    if (cudaEventCreate(&ev) != cudaSuccess) return nullptr;
    e->ev_pool.push_back(ev);
  }
  return e->ev_pool[e->ev_used++];
}

// open an interval for class cls if it is being timed; returns the record index or -1
static int tbegin(cbt_engine* e, int cls) {
  if (!(e->timing_mask & (1 << cls))) return -1;
  cudaEvent_t a = next_event(e), b = next_event(e);
  if (!a || !b) return -1;
  cudaEventRecord(a, e->stream);
  e->recs.push_back({cls, a, b, 0.0});
  return (int)e->recs.size() - 1;
}

static void tend(cbt_engine* e, int rec, double bytes) {
  if (rec < 0) return;
  cudaEventRecord(e->recs[rec].b, e->stream);
  e->recs[rec].bytes = bytes;
}

extern "C" cbt_status cbt_engine_set_timing(cbt_engine* e, int32_t mask) {
  if (!e) return CBT_ERR_NULL;
  if (cudaStreamSynchronize(e->stream) != cudaSuccess) return CBT_ERR_CUDA;
  e->timing_mask = mask;
  e->recs.clear();
  e->ev_used = 0;
  return CBT_OK;
}

extern "C" cbt_status cbt_engine_timing(cbt_engine* e, int32_t cls, double* ms, int64_t* n,
                                        double* bytes) {
  if (!e || !ms || !n || !bytes) return CBT_ERR_NULL;
  if (cls < 0 || cls >= CBT_NUM_KCLASSES) return CBT_ERR_INVALID;
  if (cudaStreamSynchronize(e->stream) != cudaSuccess) return CBT_ERR_CUDA;
  double t = 0.0, by = 0.0;
  int64_t cnt = 0;
  for (const auto& r : e->recs) {
    if (r.cls != cls) continue;
    float f = 0.f;
    if (cudaEventElapsedTime(&f, r.a, r.b) != cudaSuccess) return CBT_ERR_CUDA;
    t += f;
    by += r.bytes;
    ++cnt;
  }
  *ms = t;
  *n = cnt;
  *bytes = by;
  return CBT_OK;
}

extern "C" cbt_status cbt_engine_test_stall(cbt_engine* e, int32_t spin_limit) {
  if (!e) return CBT_ERR_NULL;
  if (spin_limit <= 0) return CBT_ERR_INVALID;
  if (!e->use_tc || e->cfg.weight_format != CBT_WEIGHTS_BF16) return CBT_ERR_UNSUPPORTED;
  e->stall_limit = (uint32_t)spin_limit;
  return CBT_OK;
}

extern "C" cbt_status cbt_engine_set_stamps(cbt_engine* e, int32_t enable) {
  if (!e) return CBT_ERR_NULL;
  if (cudaStreamSynchronize(e->stream) != cudaSuccess) return CBT_ERR_CUDA;
  if (enable && !e->stamp_buf &&
      cudaMalloc(reinterpret_cast<void**>(&e->stamp_buf), 2 * kStampSlots * sizeof(unsigned long long)) !=
          cudaSuccess) {
    e->stamp_buf = nullptr;
    return CBT_ERR_CUDA;
  }
  e->stamps_on = enable != 0;
  e->last_stamp_cls.clear();
  return CBT_OK;
}

extern "C" cbt_status cbt_engine_stamps(cbt_engine* e, int32_t cap, int32_t* n, int32_t* classes,
                                        uint64_t* times) {
  if (!e || !n) return CBT_ERR_NULL;
  if (cap < 0) return CBT_ERR_INVALID;
  if (cudaStreamSynchronize(e->stream) != cudaSuccess) return CBT_ERR_CUDA;
  const int m = (int)e->last_stamp_cls.size();
  *n = m;
  if (!e->stamp_buf || m == 0 || cap == 0) return CBT_OK;
  if (!classes || !times) return CBT_ERR_NULL;
  const int k = std::min(cap, m);
  for (int i = 0; i < k; ++i) classes[i] = e->last_stamp_cls[i];
  if (cudaMemcpy(times, e->stamp_buf, 2 * (size_t)k * sizeof(uint64_t), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return CBT_ERR_CUDA;
  return CBT_OK;
}

static double weight_bytes(const cbt_model_config& c, long long M, long long K) {
  if (c.weight_format == CBT_WEIGHTS_BF16) return 2.0 * M * K;
  return 0.5 * M * K + 4.0 * M * (K / c.group_size);  // codes + bf16 scale and bias
}

// ---- the forward pass over n tokens whose rows are already on the device ----------------
static LinearW lw(const cbt_linear& l, int fmt) {
  return LinearW{l.w, static_cast<const uint16_t*>(l.scales),
                 static_cast<const uint16_t*>(l.biases), fmt};
}

// n tokens (decode rows or packed prefill tokens); n_out rows get logits: all n when
// gather == false, else the n_out rows listed in e->last_idx
// One projection y = x W^T over n rows, timed as class PROJ; algorithmic bytes: the weights
// once, x in, y out (read and written again for a residual add).
static void projection(cbt_engine* e, const float* x, int n, int K, const cbt_linear& W, int M,
                       Epilogue epi, float* out) {
  const cbt_model_config& c = e->cfg;
  const int Mo = epi == EPI_SWIGLU ? M / 2 : M;
  int t = tbegin(e, CBT_KCLASS_PROJ);
  launch_linear(x, n, K, lw(W, c.weight_format), M, epi, out, e->part, e->part_floats, e->stream);
  tend(e, t, weight_bytes(c, M, K) + 4.0 * n * K + 4.0 * n * Mo * (epi == EPI_ADD ? 2 : 1));
}

// Tensor-core path: operands are bf16 hi/lo pairs (x = hi + lo).  Up to 32 rows keep their lo
// parts at row BN/2 of the operand buffer (the MMA's padded N side), more rows at row tmax.
static int tc_lo_rows(const cbt_engine* e, int n) {
  return n <= 32 ? tc_split_bn(n) / 2 : e->tmax;
}

static const CUtensorMap* xmap(cbt_engine* e, const uint16_t* buf, int K, int BN) {
  auto key = std::make_pair(static_cast<const void*>(buf), BN);
  auto it = e->xmaps.find(key);
  if (it != e->xmaps.end()) return &it->second;
  CUtensorMap m;
  if (!make_tmap_bf16(&m, buf, K, e->act_rows, 64, BN)) return nullptr;
  return &(e->xmaps[key] = m);
}

// the operand buffer seen in blocks of kCskBlocks 64-column tiles (decode projections)
static const CUtensorMap* xmap_kb(cbt_engine* e, const uint16_t* buf, int K, int BN) {
  auto key = std::make_pair(static_cast<const void*>(buf), BN);
  auto it = e->xmaps_kb.find(key);
  if (it != e->xmaps_kb.end()) return &it->second;
  CUtensorMap m;
  if (!make_tmap_kblocks(&m, buf, K, e->act_rows, BN, kCskBlocks, 0)) return nullptr;
  return &(e->xmaps_kb[key] = m);
}

// The next stamp slot of this step for a launch of class cls (NULL when stamps are off).
static unsigned long long* next_stamp(cbt_engine* e, int cls) {
  if (!e->stamps_on || e->stamp_n >= kStampSlots) return nullptr;
  e->stamp_cls.push_back(cls);
  return e->stamp_buf + 2 * (size_t)e->stamp_n++;
}

// y = x W^T over n rows on the tensor cores, operand x in the bf16 buffer xbuf [rows][K].
// norm_in: the operand is x * g and each column is scaled by its RMSNorm factor, from the
// sums of squares in e->ss.  next_gain (EPI_ADD): also write the updated rows' sums of squares
// to e->ss and x * next_gain into e->act_h, the operand of the projection that follows.
// 4-bit weights: q4w is the native copy (decode rows); q4lin the interchange-format matrix and
// q4shape its entry in q4x_maps, for more than 32 rows (expanded, then a dense GEMM).
static bool tc_projection(cbt_engine* e, const CUtensorMap& wmap, const CUtensorMap& wmap_kb,
                          const uint8_t* q4w, const cbt_linear* q4lin, int q4shape,
                          const uint16_t* xbuf, int n, int K, int M, Epilogue epi, float* out,
                          int ldo, uint16_t* act_out, int act_ld, bool norm_in = false,
                          const uint16_t* next_gain = nullptr, int layer = 0) {
  const bool split = n <= 32;
  const int BN = split ? tc_split_bn(n) : tc_plain_bn(n);
  const CUtensorMap* xm = split ? xmap_kb(e, xbuf, K, BN) : xmap(e, xbuf, K, BN);
  if (!xm) return false;
  TcParams p{};
  p.ss_ld = e->ss_ld;
  if (norm_in) {
    p.ss_in = e->ss;
    p.ss_tiles = (e->cfg.d_model + 127) / 128;
    p.eps = e->cfg.rms_eps;
  }
  if (epi == EPI_QKV || epi == EPI_QKVQ) {  // RoPE + KV append + the attention's Q operand
    p.rows = e->rows;
    p.layer = layer;
    p.n_heads = e->cfg.n_heads;
    p.n_kv_heads = e->cfg.n_kv_heads;
    p.head_dim = e->cfg.head_dim;
    p.cosv = e->cosv;
    p.sinv = e->sinv;
    p.arena = static_cast<uint16_t*>(e->p.kv_arena);
    p.qtile = e->qtile;
    if (epi == EPI_QKVQ) {  // the new K/V quantised in the epilogue, into each row's slab
      p.kvq_jobs = e->kv8_jobs;
      p.kvq_bits = e->kv_bits;
    }
  }
  if (next_gain) {
    p.ss_out = e->ss;
    p.next_gain = next_gain;
    p.next_act = e->act_h;
    p.next_lo = tc_lo_rows(e, n);
  }
  p.M = M;
  p.K = K;
  p.F = epi == EPI_SWIGLU ? M / 2 : 0;
  p.n_act = n;
  p.epi = epi;
  p.out = out;
  p.ldo = ldo;
  p.act = act_out;
  p.act_ld = act_ld;
  p.act_lo = tc_lo_rows(e, n);
  p.err = e->err;
  if (n <= 32) p.stamp = next_stamp(e, CBT_KCLASS_PROJ);  // the decode projections
  if (e->stall_now) {
    p.stall_loads = 1;
    p.spin_limit = e->stall_limit;
    e->stall_now = false;
  }
  const int Mo = epi == EPI_SWIGLU ? M / 2 : M;
  int t = tbegin(e, CBT_KCLASS_PROJ);
  // decode rows: cluster split-K (partial sums meet in distributed shared memory); prefill
  // tokens: whole tiles per CTA
  bool ok;
  if (e->cfg.weight_format != CBT_WEIGHTS_BF16 && split) {
    p.wq = q4w;
    ok = launch_q4_rd(p, xbuf, tc_lo_rows(e, n), e->num_sms, e->stream);
  } else if (e->cfg.weight_format != CBT_WEIGHTS_BF16) {
    uint16_t* hi = e->q4x;
    ok = hi != nullptr && q4lin != nullptr && (size_t)M * K <= e->q4x_elems &&
         launch_q4_expand(static_cast<const uint32_t*>(q4lin->w),
                          static_cast<const uint16_t*>(q4lin->scales),
                          static_cast<const uint16_t*>(q4lin->biases), M, K, hi, hi + e->q4x_elems,
                          e->num_sms, e->stream) &&
         launch_tc_linear(e->q4x_maps[q4shape][0], *xm, p, false, BN, e->num_sms, e->stream,
                          &e->q4x_maps[q4shape][1]);
  } else {
    ok = split ? launch_tc_csk(wmap_kb, *xm, p, BN, e->num_sms, e->stream)
               : launch_tc_linear(wmap, *xm, p, split, BN, e->num_sms, e->stream);
  }
  tend(e, t, weight_bytes(e->cfg, M, K) + 4.0 * n * K + 4.0 * n * Mo * (epi == EPI_ADD ? 2 : 1));
  return ok;
}

// n tokens (decode rows or packed prefill tokens); n_out rows get logits: all n when
// gather == false, else the n_out rows listed in e->last_idx.  total_keys = sum over the
// tokens of (pos + 1), the KV positions attention reads per layer and kv head.
static cudaError_t forward(cbt_engine* e, int n, const int32_t* tokens, int max_keys,
                           long long total_keys, bool gather, int n_out, float* logits,
                           int32_t* next) {
  const cbt_model_config& c = e->cfg;
  cudaStream_t s = e->stream;
  const int d = c.d_model, qd = e->qd(), kvd = e->kvd(), F = c.d_ff;
  uint16_t* arena = static_cast<uint16_t*>(e->p.kv_arena);
  const bool quant = e->quant();
  // K and V read per element: bf16, or bits / 8 bytes of codes plus a bf16 scale and bias per 64
  const double kv_el = quant ? e->kv_bits / 8.0 + 1.0 / 16.0 : 2.0;
  const double attn_bytes = 2.0 * kv_el * kvd * (double)total_keys
                            + 4.0 * n * (qd + 2 * kvd)              // q, k, v in
                            + 2.0 * 2.0 * n * kvd + 4.0 * n * qd;   // K/V appended, o out
  // 4-bit weights go through the tensor cores for up to 32 rows (the decode projections), and
  // for more rows when the engine holds the expansion scratch (dense GEMMs over bf16 hi + lo)
  // (whose maps cover lm_head whenever more than 32 rows may ask for logits)
  const bool tcp = e->use_tc && (e->cfg.weight_format == CBT_WEIGHTS_BF16 || n <= 32 ||
                                 e->q4x != nullptr);
  // decode on the tensor cores folds every RMSNorm into the projection that consumes it:
  // the residual-add epilogues and the embedding leave per-tile sums of squares in e->ss
  const bool fused = tcp && !gather && n <= 32;
  const int lo = tc_lo_rows(e, n), lo_out = tc_lo_rows(e, n_out);
  bool ok = true;
  e->stamp_n = 0;
  e->stamp_cls.clear();
  int t = tbegin(e, CBT_KCLASS_OTHER);
  launch_embed_rope(tokens, n, static_cast<const uint16_t*>(e->w.embed), d, c.vocab, e->x, e->err,
                    fused ? e->ss : nullptr, e->ss_ld,
                    static_cast<const uint16_t*>(e->layers[0].attn_norm), fused ? e->act_h : nullptr,
                    lo, e->rows, c.head_dim, c.rope_theta, e->cosv, e->sinv, s);
  tend(e, t, 2.0 * n * d + 4.0 * n * d);
  for (int l = 0; l < c.n_layers && ok; ++l) {
    const cbt_layer_weights& L = e->layers[l];
    const uint16_t* an = static_cast<const uint16_t*>(L.attn_norm);
    const uint16_t* fn = static_cast<const uint16_t*>(L.ffn_norm);
    if (!fused) {
      t = tbegin(e, CBT_KCLASS_OTHER);
      if (tcp) launch_rmsnorm_act(e->x, an, n, d, c.rms_eps, e->act_h, lo, s);
      else launch_rmsnorm(e->x, an, n, d, c.rms_eps, e->h, s);
      tend(e, t, 8.0 * n * d);
    }
    // decode on the tensor cores rotates q and k, appends K/V and lays out the attention's Q
    // operand in the QKV projection's epilogue; otherwise a separate kernel does it
    if (tcp)
      ok &= tc_projection(e, e->wmaps[l].qkv, e->wmaps_kb[l].qkv, e->q4w[l].qkv, &L.wqkv,
                          cbt_engine::kQ4xQkv, e->act_h, n, d, qd + 2 * kvd,
                          fused ? (quant ? EPI_QKVQ : EPI_QKV) : EPI_STORE, e->qkv, qd + 2 * kvd, nullptr, 0, fused,
                          nullptr, l);
    else
      projection(e, e->h, n, d, L.wqkv, qd + 2 * kvd, EPI_STORE, e->qkv);
    t = tbegin(e, CBT_KCLASS_ATTN);
    const bool tc_prefill = tcp && gather && e->pf_n > 0;
    if (!fused)
      launch_rope_append(e->qkv, e->rows, n, l, c.n_heads, c.n_kv_heads, c.head_dim, e->cosv,
                         e->sinv, arena, (!gather && (tcp || quant)) ? e->qtile : nullptr,
                         tc_prefill ? e->qb : nullptr, e->qb_rows, s);
    uint8_t* arena8 = static_cast<uint8_t*>(e->p.kv_arena);
    if (quant && !gather) {
      // quantised KV decode: the fused QKV epilogue quantised each row's new K/V into its slab;
      // otherwise they went to the row's staging page (the RoPE kernel above) and are
      // quantised here.  Then split attention over the codes on the tensor cores and the merge
      // into the O projection's operand
      if (!fused)
        ok &= launch_kvq_convert(e->kv8_jobs, n, 1, l, 1, c.n_kv_heads, c.head_dim, e->kv_bits,
                                 arena8, s);
      KvqAttnArgs qa{};
      qa.qtile = e->qtile;
      qa.rows = e->rows;
      qa.items = e->items;
      qa.n_items = e->item_meta + 2 * e->p.max_batch;
      qa.arena = arena8;
      qa.layer = l;
      qa.n_heads = c.n_heads;
      qa.n_kv_heads = c.n_kv_heads;
      qa.head_dim = c.head_dim;
      qa.part_o = e->att_o;
      qa.part_ml = e->att_ml;
      qa.err = e->err;
      qa.stamp = next_stamp(e, CBT_KCLASS_ATTN);
      ok &= launch_attn_decode_q(qa, e->kv_bits, e->num_sms, s);
      AttnDecodeArgs ma{};
      ma.item_base = e->item_meta;
      ma.item_count = e->item_meta + e->p.max_batch;
      ma.B = n;
      ma.n_heads = c.n_heads;
      ma.n_kv_heads = c.n_kv_heads;
      ma.head_dim = c.head_dim;
      ma.part_o = e->att_o;
      ma.part_ml = e->att_ml;
      ma.act = e->act_o;
      ma.act_lo = lo;
      ma.out_f32 = tcp ? nullptr : e->o;  // the CUDA-core O projection reads fp32
      ma.stamp_merge = next_stamp(e, CBT_KCLASS_ATTN);
      ok &= launch_attn_merge(ma, s);
    } else if (quant && e->q_codes) {
      // prefill tokens continuing quantised slabs: their K/V (in a bf16 intermediate) are
      // quantised first, then each token attends over the codes of [0, its position]
      ok &= launch_kvq_convert(e->kv8_jobs, e->q_jobs, e->q_jobs_max_n, l, 1, c.n_kv_heads,
                               c.head_dim, e->kv_bits, arena8, s);
      ok &= launch_attn_prefill_q(e->qkv, e->rows, e->pagetab, e->tok_pages, e->tok_pages + n, n, l,
                                  c.n_heads, c.n_kv_heads, c.head_dim, max_keys, e->kv_bits,
                                  arena8, e->o, s);
      if (tcp) launch_f32_to_act(e->o, n, qd, e->act_o, lo, s);
    } else if (tcp && !gather) {  // decode: split-K flash decoding on the tensor cores
      AttnDecodeArgs a{};
      a.qtile = e->qtile;
      a.rows = e->rows;
      a.items = e->items;
      a.n_items = e->item_meta + 2 * e->p.max_batch;
      a.item_base = e->item_meta;
      a.item_count = e->item_meta + e->p.max_batch;
      a.B = n;
      a.layer = l;
      a.n_heads = c.n_heads;
      a.n_kv_heads = c.n_kv_heads;
      a.head_dim = c.head_dim;
      a.part_o = e->att_o;
      a.part_ml = e->att_ml;
      a.act = e->act_o;
      a.act_lo = lo;
      a.err = e->err;
      a.stamp = next_stamp(e, CBT_KCLASS_ATTN);
      a.stamp_merge = next_stamp(e, CBT_KCLASS_ATTN);
      ok &= launch_attn_decode_tc(e->kv_kmap, e->kv_vmap, a, e->num_sms, s);
    } else {
      if (tc_prefill)  // flash attention per segment on the tensor cores
        ok &= launch_attn_prefill_tc(e->q_map, e->kv_kmap, e->kv_vmap, e->pf_units, e->pagetab,
                                     e->pf_n,
                                     e->qb_rows, l, c.n_heads, c.n_kv_heads, c.head_dim, e->o,
                                     e->err, e->num_sms, s);
      else
        launch_attention_naive(e->qkv, e->rows, e->page ? e->pagetab : nullptr,
                               e->page ? e->tok_pages : nullptr, n, l, c.n_heads, c.n_kv_heads,
                               c.head_dim,
                               max_keys, arena, e->o, s);
      if (tcp) launch_f32_to_act(e->o, n, qd, e->act_o, lo, s);
    }
    tend(e, t, attn_bytes);
    if (tcp)
      ok &= tc_projection(e, e->wmaps[l].o, e->wmaps_kb[l].o, e->q4w[l].o, &L.wo, cbt_engine::kQ4xO,
                          e->act_o, n, qd, d, EPI_ADD, e->x, d, nullptr, 0,
                          false, fused ? fn : nullptr);
    else
      projection(e, e->o, n, qd, L.wo, d, EPI_ADD, e->x);
    if (!fused) {
      t = tbegin(e, CBT_KCLASS_OTHER);
      if (tcp) launch_rmsnorm_act(e->x, fn, n, d, c.rms_eps, e->act_h, lo, s);
      else launch_rmsnorm(e->x, fn, n, d, c.rms_eps, e->h, s);
      tend(e, t, 8.0 * n * d);
    }
    if (tcp) {
      ok &= tc_projection(e, e->wmaps[l].gu, e->wmaps_kb[l].gu, e->q4w[l].gu, &L.wgu,
                          cbt_engine::kQ4xGu, e->act_h, n, d, 2 * F, EPI_SWIGLU, nullptr, 0,
                          e->act_u, F, fused);
      // the down projection's epilogue prepares the next layer's (or the final) RMSNorm
      const uint16_t* next_g = l + 1 < c.n_layers
                                   ? static_cast<const uint16_t*>(e->layers[l + 1].attn_norm)
                                   : static_cast<const uint16_t*>(e->w.final_norm);
      ok &= tc_projection(e, e->wmaps[l].d, e->wmaps_kb[l].d, e->q4w[l].d, &L.wd,
                          cbt_engine::kQ4xDown, e->act_u, n, F, d, EPI_ADD, e->x, d, nullptr, 0,
                          false, fused ? next_g : nullptr);
    } else {
      projection(e, e->h, n, d, L.wgu, 2 * F, EPI_SWIGLU, e->act);
      projection(e, e->act, n, F, L.wd, d, EPI_ADD, e->x);
    }
  }
  if (!ok) return cudaErrorNotSupported;
  const float* xf = e->x;
  float* hf = e->xg + (size_t)e->p.max_batch * d;
  const uint16_t* gn = static_cast<const uint16_t*>(e->w.final_norm);
  if (!fused) {
    t = tbegin(e, CBT_KCLASS_OTHER);
    if (gather) {
      launch_gather_rows(e->x, e->last_idx, n_out, d, e->xg, s);
      xf = e->xg;
    }
    if (tcp) launch_rmsnorm_act(xf, gn, n_out, d, c.rms_eps, e->act_h, lo_out, s);
    else launch_rmsnorm(xf, gn, n_out, d, c.rms_eps, hf, s);
    tend(e, t, 8.0 * n_out * d);
  }
  float* lg = logits ? logits : e->logits;
  e->stall_now = e->stall_limit != 0 && fused && c.weight_format == CBT_WEIGHTS_BF16;
  if (tcp) {
    if (!tc_projection(e, e->lm_map, e->lm_map_kb, e->q4_lm, &e->w.lm_head, cbt_engine::kQ4xLm,
                       e->act_h, n_out, d, c.vocab, EPI_STORE, lg, c.vocab, nullptr,
                       0, fused))
      return cudaErrorNotSupported;
  } else {
    projection(e, hf, n_out, d, e->w.lm_head, c.vocab, EPI_STORE, lg);
  }
  t = tbegin(e, CBT_KCLASS_OTHER);
  launch_argmax(lg, n_out, c.vocab, next ? next : e->next_tok, s);
  tend(e, t, 4.0 * n_out * c.vocab);
  return cudaGetLastError();
}

static void drop_graphs(cbt_engine* e);
static cudaError_t upload_page_tables(cbt_engine* e);

// Work list of the tensor-core decode attention for the rows in e->hrows[0..B): per row and kv
// head, runs of 128-key sub-chunks over positions [0, pos].  Grows the item and partial
// buffers when needed and copies the list to the device on the engine stream.
//
// Sub-chunks per item: one, or two for a row whose own context reaches kLongSubs sub-chunks
// (half the partial outputs and merge work of a long row, with items still plentiful enough
// to balance the grid).  The choice depends on the row's own length, so a row's result does
// not depend on the other rows of the step.  Paged slabs keep one (an item lies in one page,
// and pages may be 128 positions); so does quantised KV (its kernel takes one per item).
static constexpr int kLongSubs = 64;
static int subs_per_item(const cbt_engine* e, const Slab& sl, int nsub) {
  return (nsub >= kLongSubs && !e->quant() && !paged(e, sl)) ? 2 : 1;
}

static cudaError_t plan_decode_attention(cbt_engine* e, int B) {
  const int Hkv = e->cfg.n_kv_heads, G = e->cfg.n_heads / Hkv, hd = e->cfg.head_dim;
  e->hitems.clear();
  for (int b = 0; b < B; ++b) {
    const int nsub = (e->hrows[b].pos + 1 + 127) / 128;
    const int per = subs_per_item(e, *e->hslab[b], nsub);
    const int splits = (nsub + per - 1) / per;
    e->hitem_base[b] = (int)e->hitems.size();
    e->hitem_count[b] = splits;
    for (int g = 0; g < Hkv; ++g)
      for (int sp = 0; sp < splits; ++sp) {
        AttnItem it{b, g, sp * per, std::min(nsub, (sp + 1) * per),
                    row_base(e, *e->hslab[b], sp * per * 128), 0, 0, e->hrows[b].pos + 1};
        if (e->quant()) {  // the quantised slab or page: byte offset, capacity, first position
          const QLoc q = qloc(e, *e->hslab[b], sp * per * 128);
          it.kbase = q.off;
          it.cap = q.cap;
          it.p0 = q.p0;
        }
        e->hitems.push_back(it);
      }
  }
  const size_t n = e->hitems.size();
  cudaError_t rc = cudaSuccess;
  if (n > e->att_items_cap) {
    size_t cap = std::max(n, e->att_items_cap * 2);
    rc = cudaStreamSynchronize(e->stream);
    drop_graphs(e);  // captured steps hold the old buffer addresses
    cudaFree(e->items);
    cudaFree(e->att_o);
    cudaFree(e->att_ml);
    e->items = nullptr;
    e->att_o = nullptr;
    e->att_ml = nullptr;
    e->att_items_cap = 0;
    if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->items), cap * sizeof(AttnItem));
    if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->att_o), cap * G * hd * sizeof(float));
    if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->att_ml), cap * G * sizeof(float2));
    if (rc != cudaSuccess) return rc;
    e->att_items_cap = cap;
  }
  rc = cudaMemcpyAsync(e->items, e->hitems.data(), n * sizeof(AttnItem), cudaMemcpyHostToDevice,
                       e->stream);
  e->item_total = (int)n;
  if (rc == cudaSuccess)
    rc = cudaMemcpyAsync(e->item_meta, e->hitem_base.data(), B * sizeof(int),
                         cudaMemcpyHostToDevice, e->stream);
  if (rc == cudaSuccess)
    rc = cudaMemcpyAsync(e->item_meta + e->p.max_batch, e->hitem_count.data(), B * sizeof(int),
                         cudaMemcpyHostToDevice, e->stream);
  if (rc == cudaSuccess)
    rc = cudaMemcpyAsync(e->item_meta + 2 * e->p.max_batch, &e->item_total, sizeof(int),
                         cudaMemcpyHostToDevice, e->stream);
  return rc;
}

// The decode step as a CUDA graph, captured once per (B, token/logits/next buffers) and
// replayed: ~300 kernel launches become one graph launch, and the kernels' programmatic
// dependencies let each one's prologue overlap its predecessor's tail.  Every per-step input
// (row table, attention work list and its length) lives in device buffers written before the
// launch, so a captured graph stays valid while those buffers keep their addresses.
static void drop_graphs(cbt_engine* e) {
  for (auto& kv : e->graphs) cudaGraphExecDestroy(kv.second.exec);
  e->graphs.clear();
}

static cudaError_t run_decode_graph(cbt_engine* e, int B, const int32_t* tokens, int max_keys,
                                    long long total_keys, float* logits, int32_t* next) {
  auto key = std::make_tuple(B, static_cast<const void*>(tokens), static_cast<const void*>(logits),
                             static_cast<const void*>(next), e->stamps_on);
  auto it = e->graphs.find(key);
  if (it == e->graphs.end()) {
    if (e->graphs.size() >= 16) drop_graphs(e);
    cudaGraph_t g = nullptr;
    cudaError_t rc = cudaStreamBeginCapture(e->stream, cudaStreamCaptureModeThreadLocal);
    if (rc != cudaSuccess) return rc;
    cudaError_t frc = forward(e, B, tokens, max_keys, total_keys, false, B, logits, next);
    rc = cudaStreamEndCapture(e->stream, &g);
    if (frc != cudaSuccess || rc != cudaSuccess) {
      if (g) cudaGraphDestroy(g);
      return frc != cudaSuccess ? frc : rc;
    }
    cudaGraphExec_t ex = nullptr;
    rc = cudaGraphInstantiate(&ex, g, 0);
    cudaGraphDestroy(g);
    if (rc != cudaSuccess) return rc;
    it = e->graphs.emplace(key, cbt_engine::Captured{ex, e->stamp_cls}).first;
  }
  e->last_stamp_cls = it->second.stamp_cls;
  return cudaGraphLaunch(it->second.exec, e->stream);
}

extern "C" cbt_status cbt_decode_step_batch(cbt_engine* e, const int32_t* ids, int32_t B,
                                            const int32_t* last_tokens, float* logits,
                                            int32_t* next_tokens) {
  if (!e) return CBT_ERR_NULL;
  if (B < 0) return CBT_ERR_INVALID;
  if (B == 0) return CBT_OK;
  if (!ids || !last_tokens) return CBT_ERR_NULL;
  if (B > e->p.max_batch) return CBT_ERR_BATCH;
  std::unordered_set<int> seen;
  int max_keys = 0;
  long long total_keys = 0;
  std::vector<PageWrite> writes;
  for (int b = 0; b < B; ++b) {
    auto it = e->slabs.find(ids[b]);
    if (it == e->slabs.end()) return CBT_ERR_BAD_SLAB;
    if (!seen.insert(ids[b]).second) return CBT_ERR_DUP_SLAB;
    const Slab& sl = it->second;
    if (sl.pos + 1 > sl.cap) return CBT_ERR_CAPACITY;
    writes.push_back({ids[b], sl.pos, sl.pos + 1});
  }
  const cbt_status st = prepare_writes(e, writes);
  if (st != CBT_OK) return st;
  e->hslab.resize(B);
  e->hjobs.clear();
  for (int b = 0; b < B; ++b) {
    const Slab& sl = e->slabs[ids[b]];
    if (e->quant()) {
      // the new K/V go to row b's staging page (positions [s, s + 128) around pos), and from
      // there into the quantised slab (or the page holding pos)
      const long long sb = (long long)((e->stage_off + (size_t)b * e->stage_bytes) / 2) -
                           (long long)(sl.pos / 128) * 128 * e->cfg.head_dim;
      e->hrows[b] = QueryRow{sb, sl.pos, 128};
      const QLoc q = qloc(e, sl, sl.pos);
      e->hjobs.push_back(Kv8Job{sb, 128, sl.pos, 1, q.cap, q.off, q.p0});
    } else {
      e->hrows[b] = QueryRow{row_base(e, sl, sl.pos), sl.pos, row_cap(e, sl)};
    }
    e->hslab[b] = &sl;
    max_keys = std::max(max_keys, sl.pos + 1);
    total_keys += sl.pos + 1;
  }
  cudaError_t rc = cudaMemcpyAsync(e->rows, e->hrows.data(), sizeof(QueryRow) * B,
                                   cudaMemcpyHostToDevice, e->stream);
  if (rc == cudaSuccess && e->quant())
    rc = cudaMemcpyAsync(e->kv8_jobs, e->hjobs.data(), sizeof(Kv8Job) * B, cudaMemcpyHostToDevice,
                         e->stream);
  if (rc == cudaSuccess && e->page) {  // for the CUDA-core attention (rows above its limits)
    e->hpagetab.clear();
    e->htok_pages.assign(B, -1);
    for (int b = 0; b < B; ++b) {
      e->htok_pages[b] = (int)e->hpagetab.size();
      for (size_t pg = 0; pg < e->hslab[b]->pages.size(); ++pg)
        e->hpagetab.push_back(row_base(e, *e->hslab[b], (int)pg * e->page));
    }
    rc = upload_page_tables(e);
  }
  if (rc == cudaSuccess && e->use_tc) rc = plan_decode_attention(e, B);
  if (rc == cudaSuccess && e->stamps_on) {  // begin slots to the maximum, end slots to 0
    rc = cudaMemset2DAsync(e->stamp_buf, 16, 0xFF, 8, kStampSlots, e->stream);
    if (rc == cudaSuccess)
      rc = cudaMemset2DAsync(e->stamp_buf + 1, 16, 0, 8, kStampSlots, e->stream);
  }
  if (rc == cudaSuccess) {
    if (e->use_tc && e->timing_mask == 0 && e->stream != nullptr && e->stall_limit == 0) {
      rc = run_decode_graph(e, B, last_tokens, max_keys, total_keys, logits, next_tokens);
    } else {
      rc = forward(e, B, last_tokens, max_keys, total_keys, false, B, logits, next_tokens);
      e->last_stamp_cls = e->stamp_cls;
    }
  }
  e->stall_limit = 0;  // the stall is armed for one step
  e->stall_now = false;
  if (rc != cudaSuccess) return rc == cudaErrorNotSupported ? CBT_ERR_UNSUPPORTED : CBT_ERR_CUDA;
  for (int b = 0; b < B; ++b) e->slabs[ids[b]].pos += 1;
  e->steps += 1;
  return CBT_OK;
}

// Work units of the tensor-core prefill attention: per segment, 128-query block and q head,
// the longest blocks (most key blocks) first so the persistent grid ends evenly.  Copies the
// list to the device (growing the buffer) on the engine stream; pf_n = 0 leaves the call on
// the plain attention kernel.
// Paged engines: the call's page bases and each token's (or decode row's) offset into them, to
// the device (buffers grow as needed, after the work that may still read them)
static cudaError_t upload_page_tables(cbt_engine* e) {
  cudaError_t rc = cudaSuccess;
  const size_t np = std::max<size_t>(1, e->hpagetab.size()), nt = std::max<size_t>(1, e->htok_pages.size());
  if (np > e->pagetab_cap || nt > e->tok_pages_cap) {
    rc = cudaStreamSynchronize(e->stream);
    if (np > e->pagetab_cap) {
      if (e->pagetab) cudaFree(e->pagetab);
      e->pagetab = nullptr;
      e->pagetab_cap = 0;
      if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->pagetab), 2 * np * sizeof(long long));
      if (rc == cudaSuccess) e->pagetab_cap = 2 * np;
    }
    if (nt > e->tok_pages_cap) {
      if (e->tok_pages) cudaFree(e->tok_pages);
      e->tok_pages = nullptr;
      e->tok_pages_cap = 0;
      if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->tok_pages), 2 * nt * sizeof(int));
      if (rc == cudaSuccess) e->tok_pages_cap = 2 * nt;
    }
    if (rc != cudaSuccess) return rc;
  }
  if (!e->hpagetab.empty())
    rc = cudaMemcpyAsync(e->pagetab, e->hpagetab.data(), e->hpagetab.size() * sizeof(long long),
                         cudaMemcpyHostToDevice, e->stream);
  if (rc == cudaSuccess && !e->htok_pages.empty())
    rc = cudaMemcpyAsync(e->tok_pages, e->htok_pages.data(), e->htok_pages.size() * sizeof(int),
                         cudaMemcpyHostToDevice, e->stream);
  return rc;
}

static cudaError_t plan_prefill_attention(cbt_engine* e, const int32_t* ids, const int32_t* lens,
                                          int K) {
  e->pf_n = 0;
  const int hd = e->cfg.head_dim;
  if (!e->use_tc || (hd != 64 && hd != 128)) return cudaSuccess;
  e->hunits.clear();
  struct Blk {
    int work;
    PrefillUnit u;
  };
  std::vector<Blk> blks;
  int tok = 0;
  for (int s = 0; s < K; ++s) {
    const Slab& sl = e->slabs[ids[s]];
    const int L = lens[s];
    for (int q = 0; q < L; q += 128) {
      PrefillUnit u{};
      u.base = row_base(e, sl, 0);
      u.cap = row_cap(e, sl);
      u.pages = e->page ? e->htok_pages[tok] : -1;
      u.tok0 = tok + q;
      u.q0 = sl.pos + q;
      u.nq = std::min(128, L - q);
      u.len = sl.pos + L;
      const int work = (u.q0 + u.nq - 1) / 128 + 1;
      for (int h = 0; h < e->cfg.n_heads; ++h) {
        u.head = h;
        blks.push_back(Blk{work, u});
      }
    }
    tok += L;
  }
  std::stable_sort(blks.begin(), blks.end(), [](const Blk& a, const Blk& b) { return a.work > b.work; });
  for (const Blk& b : blks) e->hunits.push_back(b.u);
  const size_t n = e->hunits.size();
  cudaError_t rc = cudaSuccess;
  if (n > e->pf_cap) {
    rc = cudaStreamSynchronize(e->stream);
    if (e->pf_units) cudaFree(e->pf_units);
    e->pf_units = nullptr;
    e->pf_cap = 0;
    if (rc == cudaSuccess) rc = cudaMalloc(reinterpret_cast<void**>(&e->pf_units), n * sizeof(PrefillUnit));
    if (rc != cudaSuccess) return rc;
    e->pf_cap = n;
  }
  rc = cudaMemcpyAsync(e->pf_units, e->hunits.data(), n * sizeof(PrefillUnit),
                       cudaMemcpyHostToDevice, e->stream);
  if (rc == cudaSuccess) e->pf_n = (int)n;
  return rc;
}

static cbt_status prefill_impl(cbt_engine* e, const int32_t* ids, const int32_t* lens, int32_t K,
                               const int32_t* tokens, float* logits, int32_t* next_tokens);

// Quantised engines.  A segment that starts a sequence (its slab at position 0) follows the
// mlx-bun batching design's conversion point: it is prefilled in bf16 (a bf16 intermediate slab)
// and its K/V are then quantised into its own slab.  A segment that continues a sequence (a
// later chunk of its prompt) attends over codes, as every step after the first does: its K/V go
// to a bf16 intermediate, are quantised into the slab layer by layer, and each token attends
// over the codes of positions [0, its own].  Runs of consecutive segments of one kind are
// separate passes (segments never see each other, so this changes no result).
static cbt_status prefill_quant(cbt_engine* e, const int32_t* ids, const int32_t* lens, int32_t K,
                                const int32_t* tokens, float* logits, int32_t* next_tokens) {
  if (K < 0) return CBT_ERR_INVALID;
  if (K == 0) return CBT_OK;
  if (!ids || !lens || !tokens) return CBT_ERR_NULL;
  if (K > e->p.max_batch) return CBT_ERR_BATCH;
  std::unordered_set<int> seen;
  long long T = 0;
  for (int s = 0; s < K; ++s) {
    auto it = e->slabs.find(ids[s]);
    if (it == e->slabs.end()) return CBT_ERR_BAD_SLAB;
    if (!seen.insert(ids[s]).second) return CBT_ERR_DUP_SLAB;
    if (lens[s] <= 0) return CBT_ERR_INVALID;
    if ((long long)it->second.pos + lens[s] > it->second.cap) return CBT_ERR_CAPACITY;
    T += lens[s];
  }
  if (T > e->p.max_prefill_tokens) return CBT_ERR_TOKENS;
  // every intermediate first, then the destination pages, so a call the arena cannot serve
  // changes nothing
  std::vector<int32_t> tmp(K, 0);
  cbt_status st = CBT_OK;
  std::vector<PageWrite> writes;
  for (int s = 0; s < K && st == CBT_OK; ++s) {
    const Slab& d = e->slabs[ids[s]];
    const int f64 = d.pos & ~63;  // the intermediate holds positions [f64, pos + len)
    tmp[s] = temp_bf16_slab(e, d.pos + lens[s] - f64);
    if (!tmp[s]) st = CBT_ERR_POOL_EXHAUSTED;
    writes.push_back({ids[s], d.pos, (long long)d.pos + lens[s]});
  }
  if (st == CBT_OK) st = prepare_writes(e, writes);
  if (st != CBT_OK) {
    for (int s = 0; s < K; ++s)
      if (tmp[s]) drop_temp(e, tmp[s]);
    return st;
  }
  const int V = e->cfg.vocab, hd = e->cfg.head_dim;
  long long tok0 = 0;
  for (int r0 = 0; r0 < K && st == CBT_OK;) {
    const bool fresh = e->slabs[ids[r0]].pos == 0;
    int r1 = r0;
    long long n_run = 0;
    while (r1 < K && (e->slabs[ids[r1]].pos == 0) == fresh) n_run += lens[r1++];
    const int32_t* run_tokens = tokens + tok0;
    float* run_logits = logits ? logits + (size_t)r0 * V : nullptr;
    int32_t* run_next = next_tokens ? next_tokens + r0 : nullptr;
    if (fresh) {
      st = prefill_impl(e, tmp.data() + r0, lens + r0, r1 - r0, run_tokens, run_logits, run_next);
      if (st == CBT_OK) {
        e->hjobs.clear();
        for (int s = r0; s < r1; ++s) {
          const Slab& t = e->slabs[tmp[s]];
          add_jobs(e, (long long)(t.offset / 2), t.lcap, 0, lens[s], e->slabs[ids[s]]);
        }
        if (convert_jobs(e) != cudaSuccess) st = CBT_ERR_CUDA;
      }
    } else {
      // rows: each token's bf16 intermediate (its QueryRow base maps positions from f64);
      // conversion records per layer; page tables of the codes each token attends over
      e->hjobs.clear();
      e->hpagetab.clear();
      e->htok_pages.assign(2 * n_run, 0);
      long long total_keys = 0;
      int max_keys = 0, g = 0;
      for (int s = r0; s < r1; ++s) {
        const Slab& d = e->slabs[ids[s]];
        const Slab& t = e->slabs[tmp[s]];
        const int f64 = d.pos & ~63;
        const long long base = (long long)(t.offset / 2) - (long long)f64 * hd;
        add_jobs(e, base, t.lcap, d.pos, lens[s], d);
        const int first = (int)e->hpagetab.size();
        if (paged(e, d))
          for (size_t off : d.pages) e->hpagetab.push_back((long long)off);
        else
          e->hpagetab.push_back((long long)d.offset);
        for (int j = 0; j < lens[s]; ++j, ++g) {
          e->hrows[g] = QueryRow{base, d.pos + j, t.lcap};
          e->htok_pages[g] = first;
          e->htok_pages[n_run + g] = paged(e, d) ? e->page : d.lcap;
        }
        e->hidx[s - r0] = g - 1;
        max_keys = std::max(max_keys, d.pos + lens[s]);
        total_keys += (long long)lens[s] * d.pos + (long long)lens[s] * (lens[s] + 1) / 2;
      }
      cudaError_t rc = upload_jobs(e);
      if (rc == cudaSuccess)
        rc = cudaMemcpyAsync(e->rows, e->hrows.data(), sizeof(QueryRow) * n_run,
                             cudaMemcpyHostToDevice, e->stream);
      if (rc == cudaSuccess)
        rc = cudaMemcpyAsync(e->last_idx, e->hidx.data(), sizeof(int32_t) * (r1 - r0),
                             cudaMemcpyHostToDevice, e->stream);
      if (rc == cudaSuccess) rc = upload_page_tables(e);
      e->pf_n = 0;  // the codes are read by their own attention kernel
      if (rc == cudaSuccess) {
        e->q_codes = true;
        rc = forward(e, (int)n_run, run_tokens, max_keys, total_keys, true, r1 - r0, run_logits,
                     run_next);
        e->q_codes = false;
      }
      if (rc != cudaSuccess) st = rc == cudaErrorNotSupported ? CBT_ERR_UNSUPPORTED : CBT_ERR_CUDA;
      if (st == CBT_OK) {
        e->prefill_tokens += n_run;
        for (int s = r0; s < r1; ++s) e->slabs[ids[s]].pos += lens[s];
      }
    }
    if (st == CBT_OK && fresh)
      for (int s = r0; s < r1; ++s) e->slabs[ids[s]].pos = lens[s];
    tok0 += n_run;
    r0 = r1;
  }
  for (int s = 0; s < K; ++s)
    if (tmp[s]) drop_temp(e, tmp[s]);
  return st;
}

extern "C" cbt_status cbt_prefill_segmented(cbt_engine* e, const int32_t* ids,
                                            const int32_t* lens, int32_t K, const int32_t* tokens,
                                            float* logits, int32_t* next_tokens) {
  if (!e) return CBT_ERR_NULL;
  if (e->quant()) return prefill_quant(e, ids, lens, K, tokens, logits, next_tokens);
  return prefill_impl(e, ids, lens, K, tokens, logits, next_tokens);
}

static cbt_status prefill_impl(cbt_engine* e, const int32_t* ids, const int32_t* lens, int32_t K,
                               const int32_t* tokens, float* logits, int32_t* next_tokens) {
  if (K < 0) return CBT_ERR_INVALID;
  if (K == 0) return CBT_OK;
  if (!ids || !lens || !tokens) return CBT_ERR_NULL;
  if (K > e->p.max_batch) return CBT_ERR_BATCH;
  std::unordered_set<int> seen;
  long long T = 0, total_keys = 0;
  int max_keys = 0;
  for (int s = 0; s < K; ++s) {
    auto it = e->slabs.find(ids[s]);
    if (it == e->slabs.end()) return CBT_ERR_BAD_SLAB;
    if (!seen.insert(ids[s]).second) return CBT_ERR_DUP_SLAB;
    if (lens[s] <= 0) return CBT_ERR_INVALID;
    const Slab& sl = it->second;
    if ((long long)sl.pos + lens[s] > sl.cap) return CBT_ERR_CAPACITY;
    T += lens[s];
    max_keys = std::max(max_keys, sl.pos + lens[s]);
    total_keys += (long long)lens[s] * sl.pos + (long long)lens[s] * (lens[s] + 1) / 2;
  }
  if (T > e->p.max_prefill_tokens) return CBT_ERR_TOKENS;
  std::vector<PageWrite> writes;
  for (int s = 0; s < K; ++s) {
    const long long p0 = e->slabs[ids[s]].pos;
    writes.push_back({ids[s], p0, p0 + lens[s]});
  }
  const cbt_status pst = prepare_writes(e, writes);
  if (pst != CBT_OK) return pst;
  // paged segments: every page base of the segment once, each token pointing at its segment's
  e->hpagetab.clear();
  e->htok_pages.assign(T, -1);
  int g = 0;
  for (int s = 0; s < K; ++s) {
    const Slab& sl = e->slabs[ids[s]];
    const int first = (int)e->hpagetab.size();
    if (paged(e, sl))
      for (size_t pg = 0; pg < sl.pages.size(); ++pg)
        e->hpagetab.push_back(row_base(e, sl, (int)pg * e->page));
    for (int j = 0; j < lens[s]; ++j, ++g) {
      e->hrows[g] = QueryRow{row_base(e, sl, sl.pos + j), sl.pos + j, row_cap(e, sl)};
      if (paged(e, sl)) e->htok_pages[g] = first;
    }
    e->hidx[s] = g - 1;
  }
  cudaError_t rc = cudaMemcpyAsync(e->rows, e->hrows.data(), sizeof(QueryRow) * T,
                                   cudaMemcpyHostToDevice, e->stream);
  if (rc == cudaSuccess)
    rc = cudaMemcpyAsync(e->last_idx, e->hidx.data(), sizeof(int32_t) * K, cudaMemcpyHostToDevice,
                         e->stream);
  if (rc == cudaSuccess && e->page) rc = upload_page_tables(e);
  if (rc == cudaSuccess) rc = plan_prefill_attention(e, ids, lens, K);
  if (rc == cudaSuccess)
    rc = forward(e, (int)T, tokens, max_keys, total_keys, true, K, logits, next_tokens);
  if (rc != cudaSuccess) return rc == cudaErrorNotSupported ? CBT_ERR_UNSUPPORTED : CBT_ERR_CUDA;
  for (int s = 0; s < K; ++s) e->slabs[ids[s]].pos += lens[s];
  e->prefill_tokens += T;
  return CBT_OK;
}

extern "C" cbt_status cbt_last_device_error(cbt_engine* e, int32_t* code, int32_t* info) {
  if (!e || !code || !info) return CBT_ERR_NULL;
  int h[2] = {0, 0};
  cudaError_t rc = cudaStreamSynchronize(e->stream);
  if (rc == cudaSuccess) rc = cudaMemcpy(h, e->err, sizeof(h), cudaMemcpyDeviceToHost);
  if (rc == cudaSuccess) rc = cudaMemset(e->err, 0, sizeof(h));
  if (rc != cudaSuccess) return CBT_ERR_CUDA;
  *code = h[0];
  *info = h[1];
  return CBT_OK;
}

extern "C" cbt_status cbt_engine_stats(cbt_engine* e, cbt_stats* out) {
  if (!e || !out) return CBT_ERR_NULL;
  out->live_slabs = (int32_t)e->slabs.size();
  out->max_batch = e->p.max_batch;
  out->slab_bytes_in_use = (int64_t)e->in_use;
  out->arena_bytes = (int64_t)(e->p.kv_arena_bytes & ~(kSlabAlign - 1));
  size_t big = 0;
  for (auto& kv : e->free_ext) big = std::max(big, kv.second);
  out->largest_free_bytes = (int64_t)big;
  out->scratch_bytes = (int64_t)e->scratch_bytes;
  out->decode_steps = e->steps;
  out->prefill_tokens = e->prefill_tokens;
  return CBT_OK;
}

extern "C" int64_t cbt_kernel_launches(cbt_engine* e) {
  (void)e;
  return kernel_launch_count();
}

extern "C" cbt_status cbt_quantize_kv(const void* x, int32_t rows, int32_t cols, int32_t bits,
                                      void* codes, void* scales, void* biases, void* stream) {
  if (!x || !codes || !scales || !biases) return CBT_ERR_NULL;
  if (bits != 8 && bits != 4) return CBT_ERR_INVALID;
  if (rows < 0 || cols <= 0 || cols % 64 || (reinterpret_cast<uintptr_t>(x) & 3) ||
      (bits == 8 && (reinterpret_cast<uintptr_t>(codes) & 1)) ||
      (reinterpret_cast<uintptr_t>(scales) & 1) || (reinterpret_cast<uintptr_t>(biases) & 1))
    return CBT_ERR_INVALID;
  return launch_quantize_kv(static_cast<const uint16_t*>(x), rows, cols, bits,
                            static_cast<uint8_t*>(codes), static_cast<uint16_t*>(scales),
                            static_cast<uint16_t*>(biases), static_cast<cudaStream_t>(stream))
             ? CBT_OK
             : CBT_ERR_CUDA;
}

extern "C" cbt_status cbt_quantize_kv8(const void* x, int32_t rows, int32_t cols, void* codes,
                                       void* scales, void* biases, void* stream) {
  return cbt_quantize_kv(x, rows, cols, 8, codes, scales, biases, stream);
}

extern "C" cbt_status cbt_quantize_affine4(const void* w, int32_t rows, int32_t cols, int32_t group,
                                           void* packed, void* scales, void* biases, void* stream) {
  if (!w || !packed || !scales || !biases) return CBT_ERR_NULL;
  if (rows <= 0 || cols <= 0 || group <= 0 || group % 8 || cols % group) return CBT_ERR_INVALID;
  launch_quantize_affine4(static_cast<const uint16_t*>(w), rows, cols, group,
                          static_cast<uint32_t*>(packed), static_cast<uint16_t*>(scales),
                          static_cast<uint16_t*>(biases), static_cast<cudaStream_t>(stream));
  return cudaGetLastError() == cudaSuccess ? CBT_OK : CBT_ERR_CUDA;
}
