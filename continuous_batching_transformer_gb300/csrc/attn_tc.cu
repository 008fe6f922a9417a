// attn_tc.cu -- decode attention on the 5th-generation tensor cores (sm_103a).
//
// Split-K flash decoding over each row's own slab: a work item is (row b, kv head g, a run of
// 128-key sub-chunks).  All q heads of the kv head's group are processed together, so the
// group's K/V is read from HBM once.  For each sub-chunk:
//   S^T[key][j] = K[key] . Q[j]   tcgen05.mma, M = 128 keys, N = 16 (q rows: 8 hi + 8 lo parts)
//   softmax on S^T: one thread per key (TMEM lane = key), running max/sum per head
//   O^T[d][j]  = V^T[d] . P[j]    tcgen05.mma, M = 128 dims, N = 16 (p rows: 8 hi + 8 lo)
// and O is accumulated in registers (one thread per dim) with the running-max rescale.
// A producer warp loads K and V^T tiles through two arena-wide TMA tensor maps (K rows of
// head_dim, V rows of 64 keys) and the group's Q operand, which the RoPE kernel already laid
// out as the swizzled hi/lo image the MMA reads, with a 1-D bulk copy.  K and V have their own
// buffers and barriers, so the next K tile streams in while this sub-chunk's softmax and P.V
// run.  Three CTAs share an SM so their latency chains overlap; items run on a persistent
// grid.  Each item leaves unnormalised partial outputs with their (max, sum); attn_merge
// combines them.
#include "kernels.h"
#include "tc_common.cuh"

namespace {

constexpr int kSub = 128;      // keys per sub-chunk (MMA M)
constexpr int kBox = 16384;    // one 128 x 128-byte tile
constexpr int kCompute = 128;  // threads of warps 0..3; warp 4 is the producer
constexpr int kCtasPerSm = 3;
// Two threads issue each contraction's MMAs (threads 0 and 32, half of the k-steps each, into
// accumulators of their own, added when read): one thread issues a tcgen05.mma only about
// every 60 ns, which made the eight MMAs of S and of P.V a long step of every sub-chunk.
constexpr int kIssuers = 2;
constexpr uint32_t kTmemCols = 64;  // issuer i: S^T in columns 32 i .. +15, O^T in 32 i + 16 .. +15

__device__ __forceinline__ void st_bf16(uint8_t* base, uint32_t off, uint16_t v) {
  *reinterpret_cast<uint16_t*>(base + off) = v;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// barrier over `n` threads that also returns whether `pred` held in any of them, so that a
// failed (timed-out) wait makes every participant leave together
__device__ __forceinline__ bool bar_any(int id, int n, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void flag_timeout(int* err, volatile int* abort_flag, int where) {
  *abort_flag = 1;
  if (atomicCAS(err, 0, CBT_DEV_TIMEOUT) == 0) err[1] = where;
}

// the maxima (MAX) or sums of N values of every lane, across the warp: the N reductions
// interleaved level by level, so their shuffle latencies overlap
template <int N, bool MAX>
__device__ __forceinline__ void warp_reduce_n(float (&v)[N]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float t[N];
#pragma unroll
    for (int h = 0; h < N; ++h) t[h] = __shfl_xor_sync(0xffffffffu, v[h], o);
#pragma unroll
    for (int h = 0; h < N; ++h) v[h] = MAX ? fmaxf(v[h], t[h]) : v[h] + t[h];
  }
}

// G q heads per kv head, GT = G rounded up to 1, 2, 4 or 8: the softmax and the output
// accumulation run over GT heads (the MMAs' unused head rows are zero), masked to G
template <int HD, int GT>
__global__ void __launch_bounds__(160, kCtasPerSm)
    k_attn_decode(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                  const uint8_t* __restrict__ qtile, const QueryRow* __restrict__ rows,
                  const AttnItem* __restrict__ items, const int* __restrict__ n_items_dev,
                  int layer, int n_kv_heads, int G, float* __restrict__ part_o,
                  float2* __restrict__ part_ml, int* err, unsigned long long* stamp) {
  constexpr int nKh = HD / 64;                          // K boxes (64 dims each)
  constexpr uint32_t kQBytes = 16 * HD * 2;             // Q operand image
  constexpr uint32_t kKBytes = kSub * HD * 2;           // K tile
  constexpr uint32_t kVBytes = 2 * HD * 128;            // V^T tile: two boxes of HD rows x 64 keys
  constexpr uint32_t kIdesc = tc::idesc_bf16(128, 16);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;                       // nKh boxes
  uint8_t* sV = sK + nKh * kBox;            // 2 boxes (HD rows used of each 128)
  uint8_t* sQ = sV + 2 * kBox;              // [16 rows][HD]: nKh groups of 2 KB
  uint8_t* sP = sQ + nKh * 2048;            // [16 rows][128 keys]: 2 groups of 2 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * 2048);
  uint64_t *kfull = bars, *vfull = bars + 1, *qfull = bars + 2;
  uint64_t *kempty = bars + 3, *vempty = bars + 4, *qempty = bars + 5;
  uint64_t *bar_s = bars + 6, *bar_o = bars + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(tmem_slot + 4);  // [4 warps][8 heads]
  float* red2 = red + 32;                                // [4 warps][8 heads]
  float* l_run = red2 + 32;                              // [8]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    // full barriers: the producer's arrival; empty and MMA barriers: both issuers' commits
    for (int i = 0; i < 8; ++i) tc::mbar_init(&bars[i], i < 3 ? 1 : kIssuers);
    *abort_flag = 0;
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&tk);
    tc::tma_prefetch_desc(&tv);
  }
  if (warp == 0) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch();
  // the work list and the row table are step inputs copied before the step's first kernel, so
  // they may be read before waiting for the previous kernel
  const int n_items = *n_items_dev;

  if (warp == 4) {
    // ---- producer: per item the Q image, per sub-chunk a K tile and a V^T tile
    if (lane == 0) {
      const uint64_t pol = tc::policy_evict_first();
      uint32_t qn = 0, kn = 0, vn = 0;
      bool ok = true;
      auto load_kv = [&](const QueryRow& row, const AttnItem& w, int sub) -> bool {
        const QueryRow r{w.kbase, row.pos, row.cap};  // the slab or page holding the item
        const long long krow = kv_block(r, layer, 0, w.g, n_kv_heads, HD) / HD;
        const long long vrow = kv_block(r, layer, 1, w.g, n_kv_heads, HD) / 64;
        if (!tc::mbar_wait(kempty, (kn & 1) ^ 1)) {
          flag_timeout(err, abort_flag, 22);
          return false;
        }
        tc::mbar_expect_tx(kfull, kKBytes);
#pragma unroll
        for (int h = 0; h < nKh; ++h)
          tc::tma_load_2d(sK + h * kBox, &tk, kfull, h * 64, (int)(krow + sub * kSub), pol);
        ++kn;
        if (!tc::mbar_wait(vempty, (vn & 1) ^ 1)) {
          flag_timeout(err, abort_flag, 23);
          return false;
        }
        tc::mbar_expect_tx(vfull, kVBytes);
#pragma unroll
        for (int j = 0; j < 2; ++j)
          tc::tma_load_2d(sV + j * kBox, &tv, vfull, 0, (int)(vrow + (long long)(2 * sub + j) * HD),
                          pol);
        ++vn;
        return true;
      };
      // Keys and values before the new position were written by earlier steps: the first
      // sub-chunk's tiles are requested before waiting for the previous kernel (which appends
      // the new position and writes Q), unless the sub-chunk holds the new position.
      int pre_sub = -1;
      if ((int)blockIdx.x < n_items) {
        const AttnItem w = items[blockIdx.x];
        const QueryRow r = rows[w.b];
        if (w.s0 < r.pos / kSub) {
          ok = load_kv(r, w, w.s0);
          pre_sub = w.s0;
        }
      }
      pdl_wait();
      for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
        const AttnItem w = items[it];
        const QueryRow r = rows[w.b];
        if (!tc::mbar_wait(qempty, (qn & 1) ^ 1)) {
          flag_timeout(err, abort_flag, 21);
          break;
        }
        tc::mbar_expect_tx(qfull, kQBytes);
        tc::bulk_load(sQ, qtile + ((size_t)w.b * n_kv_heads + w.g) * kQBytes, kQBytes, qfull);
        ++qn;
        for (int sub = w.s0; sub < w.s1 && ok; ++sub) {
          if (it == (int)blockIdx.x && sub == pre_sub) continue;  // already requested
          ok = load_kv(r, w, sub);
        }
      }
      // no copies in flight at exit: the last Q, K and V loads have landed
      if (qn) tc::mbar_wait(qfull, (qn - 1) & 1);
      if (kn) tc::mbar_wait(kfull, (kn - 1) & 1);
      if (vn) tc::mbar_wait(vfull, (vn - 1) & 1);
    }
  } else {
    // ---- compute warps: MMA issue (thread 0), softmax (thread = key), accumulate (thread = dim)
    // P rows of the heads past GT (and their lo rows) are never written: zero once
    for (int i = tid; i < 2 * 2048 / 4; i += kCompute) reinterpret_cast<uint32_t*>(sP)[i] = 0u;
    pdl_wait();  // Q, the new K/V and the partial buffers are shared with earlier kernels
    if (tid == 0) stamp_begin(stamp);
    uint32_t qn = 0, kn = 0, vn = 0, sn = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
      const AttnItem w = items[it];
      const int n = rows[w.b].pos + 1;
      if (tid < 8) l_run[tid] = 0.f;
      // the running max of every head, kept by every thread: each computes it from the same
      // inputs in the same order, so no exchange is needed between the max and the weights
      float m_run[GT];
#pragma unroll
      for (int h = 0; h < GT; ++h) m_run[h] = -INFINITY;
      float oacc[GT];
#pragma unroll
      for (int h = 0; h < GT; ++h) oacc[h] = 0.f;
      tc::named_bar_sync(1, kCompute);

      for (int sub = w.s0; sub < w.s1; ++sub, ++sn) {
        if (tid == 0 || tid == 32) {  // issuer i: k-steps [i HD/32, (i + 1) HD/32)
          const int iss = tid >> 5;
          bool good = true;
          if (sub == w.s0) good = tc::mbar_wait(qfull, qn & 1);
          good = good && tc::mbar_wait(kfull, kn & 1);
          if (!good) {
            flag_timeout(err, abort_flag, 24);
          } else {
            tc::tc_fence_after();
            constexpr int kSteps = HD / 16 / kIssuers;
#pragma unroll
            for (int k = 0; k < kSteps; ++k) {
              const int kk = iss * kSteps + k;
              const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sK + (kk >> 2) * kBox)) + 2 * (kk & 3);
              const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sQ + (kk >> 2) * 2048)) + 2 * (kk & 3);
              tc::mma_bf16(tmem + 32 * iss, ad, bd, kIdesc, k > 0 ? 1u : 0u);
            }
            tc::mma_commit(bar_s);
            tc::mma_commit(kempty);                 // K buffer free once the MMA has read it
            if (sub == w.s1 - 1) tc::mma_commit(qempty);  // and the Q image after the last one
          }
        }
        ++kn;
        const bool bad_s = *abort_flag || !tc::mbar_wait(bar_s, sn & 1);
        if (bar_any(2, kCompute, bad_s)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        // scores of this thread's key: S^T lane = key, columns j (hi) + 8 + j (lo)
        uint32_t raw[16], raw2[16];
        tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16), raw);
        tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 32, raw2);
        tc::tmem_ld_wait();
        const int key = sub * kSub + tid;
        const bool valid = key < n;
        float s[GT], mx[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          s[h] = valid ? (__uint_as_float(raw[h]) + __uint_as_float(raw[8 + h])) +
                             (__uint_as_float(raw2[h]) + __uint_as_float(raw2[8 + h]))
                       : -INFINITY;
          mx[h] = s[h];
        }
        warp_reduce_n<GT, true>(mx);
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < GT; ++h) red[warp * 8 + h] = mx[h];
        }
        tc::named_bar_sync(1, kCompute);
        float scl[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) {
          const float mloc = fmaxf(fmaxf(red[h], red[8 + h]), fmaxf(red[16 + h], red[24 + h]));
          const float mo = m_run[h];
          const float mn = fmaxf(mo, mloc);
          scl[h] = mo == -INFINITY ? 0.f : __expf(mo - mn);
          m_run[h] = mn;
        }
        float ps[GT];
#pragma unroll
        for (int h = 0; h < GT; ++h) {  // P rows of heads >= GT stay zero (set at the start)
          const float p = (valid && h < G) ? __expf(s[h] - m_run[h]) : 0.f;
          const uint16_t hi = f32_to_bf16(p);
          st_bf16(sP, sw128_offset(h, tid, 2048), hi);
          st_bf16(sP, sw128_offset(8 + h, tid, 2048), f32_to_bf16(p - bf16_to_f32(hi)));
          ps[h] = p;
        }
        warp_reduce_n<GT, false>(ps);
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < GT; ++h) red2[warp * 8 + h] = ps[h];
        }
        if (sub * kSub + kSub > n) {
          // keys past t_s: their V^T columns may hold stale values, so once V has landed
          // those columns are set to zero (P is zero there too)
          const bool bad_v = !tc::mbar_wait(vfull, vn & 1);
          if (bar_any(2, kCompute, bad_v)) {
            flag_timeout(err, abort_flag, 25);
            ok = false;
            break;
          }
          if (!valid) {
            uint8_t* vt = sV + (tid >> 6) * kBox;
            for (int d = 0; d < HD; ++d) st_bf16(vt, sw128_offset(d, tid & 63, 0), 0);
          }
        }
        fence_proxy_async();
        tc::tc_fence_before();
        tc::named_bar_sync(1, kCompute);
        if (tid < GT) {
          float sc = scl[0];
#pragma unroll
          for (int h = 1; h < GT; ++h)
            if (h == tid) sc = scl[h];
          l_run[tid] = l_run[tid] * sc + red2[tid] + red2[8 + tid] + red2[16 + tid] + red2[24 + tid];
        }
        if (tid == 0 || tid == 32) {  // issuer i: keys [64 i, 64 i + 64)
          const int iss = tid >> 5;
          if (!tc::mbar_wait(vfull, vn & 1)) {
            flag_timeout(err, abort_flag, 26);
          } else {
            tc::tc_fence_after();
            constexpr int kSteps = kSub / 16 / kIssuers;
#pragma unroll
            for (int k = 0; k < kSteps; ++k) {
              const int kk = iss * kSteps + k;
              const uint64_t ad = tc::sdesc_sw128(tc::smem_u32(sV + (kk >> 2) * kBox)) + 2 * (kk & 3);
              const uint64_t bd = tc::sdesc_sw128(tc::smem_u32(sP + (kk >> 2) * 2048)) + 2 * (kk & 3);
              tc::mma_bf16(tmem + 32 * iss + 16, ad, bd, kIdesc, k > 0 ? 1u : 0u);
            }
            tc::mma_commit(bar_o);
            tc::mma_commit(vempty);
          }
        }
        ++vn;
        const bool bad_o = *abort_flag || !tc::mbar_wait(bar_o, sn & 1);
        if (bar_any(2, kCompute, bad_o)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 16, raw);
        tc::tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + 48, raw2);
        tc::tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < GT; ++h)
          oacc[h] = oacc[h] * scl[h] + ((__uint_as_float(raw[h]) + __uint_as_float(raw[8 + h])) +
                                        (__uint_as_float(raw2[h]) + __uint_as_float(raw2[8 + h])));
        tc::tc_fence_before();
      }
      ++qn;
      if (!ok) break;
      // partial output of this item, relative to m_run
      if (tid < HD) {
        for (int h = 0; h < G; ++h) part_o[((size_t)it * G + h) * HD + tid] = oacc[h];
      }
      if (tid < G) {
        float mm = m_run[0];
#pragma unroll
        for (int h = 1; h < GT; ++h)
          if (h == tid) mm = m_run[h];
        part_ml[(size_t)it * G + tid] = make_float2(mm, l_run[tid]);
      }
      tc::named_bar_sync(1, kCompute);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (tid == 0) stamp_end(stamp);
}

// Combine the partials of each (row, q head): o = sum_i o_i e^(m_i - M) / sum_i l_i e^(m_i - M)
// and write it as the bf16 (hi/lo) operand of the output projection.  One 128-thread block per
// (row, q head), one pass over the partials: warp w takes splits w, w + 4, ... in order with
// a running maximum (lane = head_dim / 32 output dimensions; the loads of several splits are
// in flight together), then the four warps' (max, sum, output) are combined in a fixed order.
// The order depends only on the row's own splits.
__global__ void __launch_bounds__(128)
    k_attn_merge(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                 const int* __restrict__ item_base, const int* __restrict__ item_count, int B,
                 int n_heads, int n_kv_heads, int head_dim, uint16_t* act, int lo_rows,
                 float* out_f32, unsigned long long* stamp) {
  pdl_wait();
  pdl_launch();
  if (threadIdx.x == 0) stamp_begin(stamp);
  __shared__ float wm[4], wl[4];
  __shared__ float wsum[4][128];
  const int hq = blockIdx.x, b = blockIdx.y;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int G = n_heads / n_kv_heads, g = hq / G, h = hq % G;
  const int cnt = item_count[b];
  const int first = item_base[b] + g * cnt;
  const float2* ml = part_ml + (size_t)first * G + h;  // split i at ml[i * G]
  const int per = head_dim / 32;  // 4 (head_dim 128) or 2 (64)
  float m = -INFINITY, l = 0.f;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int i = warp; i < cnt; i += 4) {
    const float2 v = __ldcg(ml + (size_t)i * G);
    const float* po = part_o + ((size_t)(first + i) * G + h) * head_dim + lane * per;
    float o[4];
    if (per == 4) {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(po));
      o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w;
    } else {
      const float2 f = __ldcg(reinterpret_cast<const float2*>(po));
      o[0] = f.x; o[1] = f.y; o[2] = 0.f; o[3] = 0.f;
    }
    const float mn = fmaxf(m, v.x);
    const float sc = m == -INFINITY ? 0.f : __expf(m - mn);
    const float wgt = __expf(v.x - mn);
    l = fmaf(l, sc, v.y * wgt);
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[j] = fmaf(acc[j], sc, o[j] * wgt);
    m = mn;
  }
  if (lane == 0) {
    wm[warp] = m;
    wl[warp] = l;
  }
  for (int j = 0; j < per; ++j) wsum[warp][lane * per + j] = acc[j];
  __syncthreads();
  if (t < head_dim) {
    const float M = fmaxf(fmaxf(wm[0], wm[1]), fmaxf(wm[2], wm[3]));
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {  // a warp without splits has m = -inf and contributes 0
      const float sc = wm[w] == -INFINITY ? 0.f : __expf(wm[w] - M);
      L = fmaf(wl[w], sc, L);
      o = fmaf(wsum[w][t], sc, o);
    }
    o = o / L;
    const int K = n_heads * head_dim;
    const int col = hq * head_dim + t;
    if (t == 0) stamp_end(stamp);
    if (out_f32) {
      out_f32[(size_t)b * K + col] = o;
      return;
    }
    const uint16_t hi = f32_to_bf16(o);
    act[(size_t)b * K + col] = hi;
    if (lo_rows > 0) act[(size_t)(lo_rows + b) * K + col] = f32_to_bf16(o - bf16_to_f32(hi));
  }
}

template <int HD, int GT>
cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const AttnDecodeArgs& a,
                          int grid, cudaStream_t s) {
  constexpr int nKh = HD / 64;
  constexpr size_t smem = 1024 + (nKh + 2) * kBox + nKh * 2048 + 2 * 2048 + 512;
  static_assert(smem * kCtasPerSm <= 228 * 1024, "shared memory budget");
  cudaError_t rc = cudaFuncSetAttribute(k_attn_decode<HD, GT>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (rc != cudaSuccess) return rc;
  return launch_pdl(k_attn_decode<HD, GT>, dim3(grid), dim3(160), smem, s, tk, tv, a.qtile, a.rows,
                    a.items, a.n_items, a.layer, a.n_kv_heads, a.n_heads / a.n_kv_heads, a.part_o,
                    a.part_ml, a.err, a.stamp);
}

}  // namespace

bool launch_attn_decode_tc(const CUtensorMap& tk, const CUtensorMap& tv, const AttnDecodeArgs& a,
                           int num_sms, cudaStream_t s) {
  if (a.n_heads % a.n_kv_heads || a.n_heads / a.n_kv_heads > 8) return false;
  const int grid = kCtasPerSm * num_sms;  // persistent; the item count is read on the device
  cudaError_t rc;
  const int G = a.n_heads / a.n_kv_heads;
  const int gt = G <= 1 ? 1 : G <= 2 ? 2 : G <= 4 ? 4 : 8;
  if (a.head_dim == 128)
    rc = gt == 1 ? launch_decode<128, 1>(tk, tv, a, grid, s)
         : gt == 2 ? launch_decode<128, 2>(tk, tv, a, grid, s)
         : gt == 4 ? launch_decode<128, 4>(tk, tv, a, grid, s)
                   : launch_decode<128, 8>(tk, tv, a, grid, s);
  else if (a.head_dim == 64)
    rc = gt == 1 ? launch_decode<64, 1>(tk, tv, a, grid, s)
         : gt == 2 ? launch_decode<64, 2>(tk, tv, a, grid, s)
         : gt == 4 ? launch_decode<64, 4>(tk, tv, a, grid, s)
                   : launch_decode<64, 8>(tk, tv, a, grid, s);
  else return false;
  if (rc != cudaSuccess) return false;
  return launch_attn_merge(a, s);
}

bool launch_attn_merge(const AttnDecodeArgs& a, cudaStream_t s) {
  return launch_pdl(k_attn_merge, dim3(a.n_heads, a.B), dim3(128), 0, s, a.part_o, a.part_ml,
                    a.item_base, a.item_count, a.B, a.n_heads, a.n_kv_heads, a.head_dim, a.act,
                    a.act_lo, a.out_f32, a.stamp_merge) == cudaSuccess;
}
